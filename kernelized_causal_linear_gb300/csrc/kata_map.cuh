// Packed features of the lift maps (the rank-one PSD lift, KATA-M_g, KATA-Sigma_g
// and the orthant map; [KATA] Sec. 3.1 and Sec. 4.1), feature by feature, for the
// kernels that form psi entries one at a time: the CUDA-core path (kata_simt.cu)
// and the feature lift of the explicit-feature tensor path (kata_feat.cu).
#pragma once
#include "kata_internal.cuh"

namespace kata {
namespace {

// Packed feature f of a map as entries of its matrix: psi_f = cf * (add + scl *
// sum_{a < terms} x[i0 + a step] x[j0 + a step]) (one term except for Sigma_g,
// whose matrix sums the g block outer products; add is eps on its diagonal).
struct Feat {
    int i0, j0, terms, step;
    float cf, add, scl;
    bool orthant = false;   // psi_f = max(x[i0], 0) + add instead
    // x: coordinate c at x[c * xs]
    template <typename X>
    __device__ __forceinline__ float operator()(const X *x, int xs) const {
        if (orthant) return fmaxf(to_f(x[i0 * xs]), 0.f) + add;
        float e = 0.f;
        for (int a = 0; a < terms; ++a)
            e = fmaf(to_f(x[(i0 + a * step) * xs]), to_f(x[(j0 + a * step) * xs]), e);
        return cf * fmaf(scl, e, add);
    }
};

__device__ __forceinline__ Feat map_feature(int f, int d, const MapSpec &mp) {
    Feat ft;
    int i, j;
    if (mp.kind == 3) {
        ft = Feat{f, f, 0, 0, 1.f, mp.eps, 1.f};
        ft.orthant = true;
        return ft;
    }
    if (mp.kind == 0) {
        vech_pair(f, d, i, j);
        ft = Feat{i, j, 1, 0, 1.f, 0.f, 1.f};
    } else {
        const int m = d / mp.g, nb = m * (m + 1) / 2;
        if (mp.kind == 1) {
            const int a = f / nb;
            vech_pair(f - a * nb, m, i, j);
            ft = Feat{a * m + i, a * m + j, 1, 0, 1.f, 0.f, 1.f};
        } else {
            vech_pair(f, m, i, j);
            ft = Feat{i, j, mp.g, m, 1.f, i == j ? mp.eps : 0.f, mp.scale};
        }
    }
    ft.cf = ft.i0 == ft.j0 ? 1.f : kSqrt2;
    return ft;
}

}  // namespace
}  // namespace kata
