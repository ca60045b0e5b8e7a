// CUDA-core (fp32 FFMA) implementation of the KATA chunked forward.
//
// This is the path for fp32 inputs, where the 1e-4 accuracy target rules out
// the tensor cores' reduced-precision operands.  It follows the three-stage
// pipeline of the KATA paper (App. E.1 "Three-kernel pipeline"; Sec. 4.1
// Eq. 17-20):
//
//   1. chunk state   S_loc[c] = Psi(K_c)^T [V_c | 1]            (Eq. 17 term)
//   2. prefix scan   S_pre[c] = sum_{c' < c} S_loc[c']           (Sec. 4.2)
//   3. chunk output  N = Psi(Q_c) S_pre[c] + P [V_c | 1],
//                    P = (Q_c K_c^T)^2 .* M, O = N[:, :dv] / N[:, dv] (Eq. 18-20)
//
// The feature lift (Sec. 3.1) is fused: psi entries are formed in registers
// from the q/k rows staged in shared memory and never written to memory.  The
// intra-chunk weights use the closed form of psi(q).psi(k): (q.k)^2 for the full
// map, sum_a (q_a.k_a)^2 for M_g, eps^2 m + eps s (|q|^2 + |k|^2) +
// s^2 sum_{a,b} (q_a.k_b)^2 for Sigma_g (Sec. 4.1, reduced PSD families), and
// sum_i (q_i^+ + eps)(k_i^+ + eps) for the orthant map (one feature per
// coordinate, the pages' linear-state family).
//
// Workspace: per-chunk states [B*H][N_C][n][dv+1] fp32, scanned in place.
#include <cstdlib>
#include <cstring>

#include "kata_simt_common.cuh"

namespace kata {
namespace {

using namespace simt;

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

// <psi(q), psi(k)> of a map from the raw vectors; q at q[c * qs], k at k[c].
__device__ __forceinline__ float map_weight(const float *q, int qs, const float *k, int d,
                                            const MapSpec &mp) {
    if (mp.kind == 0) {
        float dot = 0.f;
        for (int i = 0; i < d; ++i) dot = fmaf(q[i * qs], k[i], dot);
        return dot * dot;
    }
    if (mp.kind == 3) {
        float w = 0.f;
        for (int i = 0; i < d; ++i)
            w = fmaf(fmaxf(q[i * qs], 0.f) + mp.eps, fmaxf(k[i], 0.f) + mp.eps, w);
        return w;
    }
    const int m = d / mp.g;
    float w = 0.f;
    if (mp.kind == 1) {
        for (int a = 0; a < mp.g; ++a) {
            float dot = 0.f;
            for (int i = 0; i < m; ++i) dot = fmaf(q[(a * m + i) * qs], k[a * m + i], dot);
            w = fmaf(dot, dot, w);
        }
        return w;
    }
    float qn = 0.f, kn = 0.f;
    for (int i = 0; i < d; ++i) {
        qn = fmaf(q[i * qs], q[i * qs], qn);
        kn = fmaf(k[i], k[i], kn);
    }
    for (int a = 0; a < mp.g; ++a)
        for (int b = 0; b < mp.g; ++b) {
            float dot = 0.f;
            for (int i = 0; i < m; ++i) dot = fmaf(q[(a * m + i) * qs], k[b * m + i], dot);
            w = fmaf(dot, dot, w);
        }
    return mp.eps * mp.eps * m + mp.eps * mp.scale * (qn + kn) + mp.scale * mp.scale * w;
}

// ---------------------------------------------------------------- stage 1
template <typename T>
__global__ void __launch_bounds__(kFeatTile)
chunk_state_kernel(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ st,
                   int T_, int d, int dv, int C, int n, int NC, int nft, MapSpec mp) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x;
    const int bh = blockIdx.y;
    const int ft = blockIdx.z % nft;
    const int cg = blockIdx.z / nft;
    const int t0 = c * C;
    const int tc = min(C, T_ - t0);
    const int cols = min(kColGroup, dv - cg * kColGroup);
    const int W = dv + 1;

    float *ks = sm;                 // [C][d]
    float *vs = ks + C * d;         // [C][32]
    const T *kc = k + ((size_t)bh * T_ + t0) * d;
    const T *vc = v + ((size_t)bh * T_ + t0) * dv + cg * kColGroup;
    for (int e = threadIdx.x; e < tc * d; e += blockDim.x) ks[e] = to_f(kc[e]);
    for (int e = threadIdx.x; e < tc * kColGroup; e += blockDim.x) {
        const int t = e / kColGroup, jj = e % kColGroup;
        vs[t * kColGroup + jj] = jj < cols ? to_f(vc[(size_t)t * dv + jj]) : 0.f;
    }
    __syncthreads();

    float acc[kStride];
#pragma unroll
    for (int jj = 0; jj < kStride; ++jj) acc[jj] = 0.f;
    const int f = ft * kFeatTile + threadIdx.x;
    if (f < n) {
        const Feat ft = map_feature(f, d, mp);
        for (int t = 0; t < tc; ++t) {
            const float a = ft(ks + t * d, 1);   // psi(k_t)_f
            fma_row32(a, vs + t * kColGroup, acc);
            acc[kColGroup] += a;
        }
    }
    // through shared memory so that each warp writes contiguous row segments
    store_state_rows(acc, sm, st + ((size_t)bh * NC + c) * (size_t)n * W, ft, cg, cols, n, dv);
}

// ---------------------------------------------------------------- stage 2
// Exclusive prefix over chunks, independently per (b, h, element), in place.
// Each thread walks the chunk axis for four consecutive elements (one float4);
// consecutive threads touch consecutive elements, so every step is a coalesced
// sweep, and each thread keeps up to eight loads in flight.
// With state_out set, the inclusive total of element e = f * W + c is written to
// state_out[bh][f][c] (c < W - 1) or z_out[bh][f] (c = W - 1); with totals set,
// to totals[bh][e].
__global__ void __launch_bounds__(256)
scan_kernel(float *__restrict__ st, int NC, int64_t E, float *__restrict__ state_out,
            float *__restrict__ z_out, int W, float *__restrict__ totals) {
    // four consecutive elements per thread (the launcher uses this kernel only
    // when E is a multiple of 4); up to 8 records are loaded before any is written
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t E4 = E >> 2;
    if (e4 >= E4) return;
    float4 *p = reinterpret_cast<float4 *>(st + (size_t)blockIdx.y * NC * E) + e4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < NC; c += 8) {
        const int m = NC - c < 8 ? NC - c : 8;
        float4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) x[j] = p[(size_t)j * E4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < m) {
                p[(size_t)j * E4] = run;
                run.x += x[j].x;
                run.y += x[j].y;
                run.z += x[j].z;
                run.w += x[j].w;
            }
        }
        p += (size_t)8 * E4;
    }
    if (totals) reinterpret_cast<float4 *>(totals + (size_t)blockIdx.y * E)[e4] = run;
    if (state_out) {
        const int64_t nf = E / W;
        const float rv[4] = {run.x, run.y, run.z, run.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t e = 4 * e4 + u, f = e / W, col = e % W;
            if (col < W - 1)
                state_out[((size_t)blockIdx.y * nf + f) * (W - 1) + col] = rv[u];
            else
                z_out[(size_t)blockIdx.y * nf + f] = rv[u];
        }
    }
}

// The same scan one element per thread, for records whose length is not a
// multiple of 4 (reduced maps with few features, e.g. Sigma_4 at d = 16).
__global__ void __launch_bounds__(256)
scan_kernel_scalar(float *__restrict__ st, int NC, int64_t E, float *__restrict__ state_out,
                   float *__restrict__ z_out, int W, float *__restrict__ totals) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float *p = st + (size_t)blockIdx.y * NC * E + e;
    float run = 0.f;
    for (int c = 0; c < NC; ++c) {
        const float x = p[(size_t)c * E];
        p[(size_t)c * E] = run;
        run += x;
    }
    if (totals) totals[(size_t)blockIdx.y * E + e] = run;
    if (state_out) {
        const int64_t nf = E / W, f = e / W, col = e % W;
        if (col < W - 1)
            state_out[((size_t)blockIdx.y * nf + f) * (W - 1) + col] = run;
        else
            z_out[(size_t)blockIdx.y * nf + f] = run;
    }
}

// Two-level form of the same exclusive scan, for records that leave the GPU idle
// with one thread per four elements (few heads, small states, many chunks): the
// chunk axis is cut into P parts of L chunks; (1) each part's total, (2) an
// exclusive scan of the totals over the parts (its last value is the inclusive
// total), (3) each part rescans from its offset.  Like the pages' tree scan it
// exposes parallelism along the chunk axis; it reads the records twice.
__global__ void __launch_bounds__(256)
scan_part_totals(const float *__restrict__ st, float *__restrict__ tot, int NC, int64_t E, int L,
                 int P) {
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, E4 = E >> 2;
    if (e4 >= E4) return;
    const int p = blockIdx.z, c0 = p * L, c1 = min(NC, c0 + L);
    const float4 *src = reinterpret_cast<const float4 *>(st + (size_t)blockIdx.y * NC * E) + e4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = c0; c < c1; c += 8) {   // up to 8 loads in flight
        const int m = c1 - c < 8 ? c1 - c : 8;
        float4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) x[j] = src[(size_t)(c + j) * E4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) {
                run.x += x[j].x;
                run.y += x[j].y;
                run.z += x[j].z;
                run.w += x[j].w;
            }
    }
    reinterpret_cast<float4 *>(tot)[((size_t)blockIdx.y * P + p) * E4 + e4] = run;
}

__global__ void __launch_bounds__(256)
scan_part_offsets(float *__restrict__ tot, int P, int64_t E, float *__restrict__ state_out,
                  float *__restrict__ z_out, int W, float *__restrict__ totals) {
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, E4 = E >> 2;
    if (e4 >= E4) return;
    float4 *t = reinterpret_cast<float4 *>(tot) + (size_t)blockIdx.y * P * E4 + e4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < P; ++p) {
        const float4 x = t[(size_t)p * E4];
        t[(size_t)p * E4] = run;
        run.x += x.x;
        run.y += x.y;
        run.z += x.z;
        run.w += x.w;
    }
    if (totals) reinterpret_cast<float4 *>(totals + (size_t)blockIdx.y * E)[e4] = run;
    if (state_out) {
        const int64_t nf = E / W;
        const float rv[4] = {run.x, run.y, run.z, run.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t e = 4 * e4 + u, f = e / W, col = e % W;
            if (col < W - 1)
                state_out[((size_t)blockIdx.y * nf + f) * (W - 1) + col] = rv[u];
            else
                z_out[(size_t)blockIdx.y * nf + f] = rv[u];
        }
    }
}

__global__ void __launch_bounds__(256)
scan_part_apply(float *__restrict__ st, const float *__restrict__ tot, int NC, int64_t E, int L,
                int P) {
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, E4 = E >> 2;
    if (e4 >= E4) return;
    const int p = blockIdx.z, c0 = p * L, c1 = min(NC, c0 + L);
    float4 *dst = reinterpret_cast<float4 *>(st + (size_t)blockIdx.y * NC * E) + e4;
    float4 run = reinterpret_cast<const float4 *>(tot)[((size_t)blockIdx.y * P + p) * E4 + e4];
    for (int c = c0; c < c1; c += 8) {   // up to 8 loads in flight
        const int m = c1 - c < 8 ? c1 - c : 8;
        float4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) x[j] = dst[(size_t)(c + j) * E4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < m) {
                dst[(size_t)(c + j) * E4] = run;
                run.x += x[j].x;
                run.y += x[j].y;
                run.z += x[j].z;
                run.w += x[j].w;
            }
    }
}

// ---------------------------------------------------------------- stage 3
// One block per (chunk, head, column group); thread r owns output row r.
template <typename T>
__global__ void __launch_bounds__(128)
output_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const float *__restrict__ st, T *__restrict__ out, int T_, int d, int dv,
              int C, int n, int NC, MapSpec mp) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x;
    const int bh = blockIdx.y;
    const int cg = blockIdx.z;
    const int r = threadIdx.x;
    const int t0 = c * C;
    const int tc = min(C, T_ - t0);
    const int cols = min(kColGroup, dv - cg * kColGroup);
    const int W = dv + 1;

    float *qsT = sm;                // [d][C]  (transposed: conflict-free per-row reads)
    float *ks = qsT + d * C;        // [C][d]
    float *vs = ks + C * d;         // [C][32]
    float *stg = vs + C * kColGroup;  // [kStageRows][kRow]
    const T *qc = q + ((size_t)bh * T_ + t0) * d;
    const T *kc = k + ((size_t)bh * T_ + t0) * d;
    const T *vc = v + ((size_t)bh * T_ + t0) * dv + cg * kColGroup;
    for (int e = threadIdx.x; e < C * d; e += blockDim.x) {
        const int t = e / d, i = e % d;
        const bool ok = t < tc;
        qsT[i * C + t] = ok ? to_f(qc[e]) : 0.f;
        ks[e] = ok ? to_f(kc[e]) : 0.f;
    }
    for (int e = threadIdx.x; e < C * kColGroup; e += blockDim.x) {
        const int t = e / kColGroup, jj = e % kColGroup;
        vs[t * kColGroup + jj] = (t < tc && jj < cols) ? to_f(vc[(size_t)t * dv + jj]) : 0.f;
    }

    float acc[kStride];
#pragma unroll
    for (int jj = 0; jj < kStride; ++jj) acc[jj] = 0.f;

    // inter-chunk term: psi(q_r) . [S_pre | Z_pre]; features are walked in order:
    // (fi, fj) within matrix blk of width w (M_g: blocks one after another)
    const float *sp = st + ((size_t)bh * NC + c) * (size_t)n * W;
    const int w = mp.kind == 0 ? d : d / mp.g;
    const int terms = mp.kind == 2 ? mp.g : 1;
    const float scl = mp.kind == 2 ? mp.scale : 1.f;
    int blk = 0, fi = 0, fj = 0;
    for (int f0 = 0; f0 < n; f0 += kStageRows) {
        const int nf = min(kStageRows, n - f0);
        __syncthreads();
        stage_state_rows(sp, stg, f0, nf, cg, cols, dv);
        __syncthreads();
        for (int fr = 0; fr < nf; ++fr) {
            if (mp.kind == 3) {   // orthant: feature f0 + fr is coordinate f0 + fr
                const float a = fmaxf(qsT[(f0 + fr) * C + r], 0.f) + mp.eps;
                const float *sr = stg + fr * kRow;
                fma_row32(a, sr, acc);
                acc[kColGroup] = fmaf(a, sr[kColGroup], acc[kColGroup]);
                continue;
            }
            float e = 0.f;
            const int i0 = blk * w + fi, j0 = blk * w + fj;
            for (int a = 0; a < terms; ++a)
                e = fmaf(qsT[(i0 + a * w) * C + r], qsT[(j0 + a * w) * C + r], e);
            const float add = (mp.kind == 2 && fi == fj) ? mp.eps : 0.f;
            const float a = fmaf(scl, e, add) * (fi == fj ? 1.f : kSqrt2);
            const float *sr = stg + fr * kRow;
            fma_row32(a, sr, acc);
            acc[kColGroup] = fmaf(a, sr[kColGroup], acc[kColGroup]);
            if (++fj == w) {
                if (++fi == w) {
                    fi = 0;
                    ++blk;
                }
                fj = fi;
            }
        }
    }

    // intra-chunk term: weights (q_r . k_s)^2 for s <= r (causal, diagonal kept)
    if (r < tc) {
        for (int s = 0; s <= r; ++s) {
            const float w = map_weight(qsT + r, C, ks + s * d, d, mp);
            fma_row32(w, vs + s * kColGroup, acc);
            acc[kColGroup] += w;
        }
        // Eq. 20 normalisation; a zero denominator gives a zero row
        const float den = acc[kColGroup];
        const float inv = den > 0.f ? 1.f / den : 0.f;
        T *orow = out + ((size_t)bh * T_ + t0 + r) * dv + cg * kColGroup;
#pragma unroll
        for (int jj = 0; jj < kColGroup; ++jj)
            if (jj < cols) orow[jj] = from_f<T>(den > 0.f ? acc[jj] * inv : 0.f);
    }
}

// ---------------------------------------------------------------- lift
template <typename T>
__global__ void __launch_bounds__(256)
lift_kernel(const T *__restrict__ x, float *__restrict__ phi, int64_t rows, int d, int n,
            MapSpec mp) {
    const int64_t total = rows * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / n;
        const int f = (int)(e % n);
        phi[e] = map_feature(f, d, mp)(x + r * d, 1);
    }
}

template <typename T>
cudaError_t simt_forward_t(const FwdShape &s, const T *q, const T *k, const T *v, T *out,
                           float *st, cudaStream_t stream, const StateOut &so,
                           const MapSpec &mp) {
    const int n = mp.n(s.d), NC = s.NC(), BH = s.BH();
    const int nft = (n + kFeatTile - 1) / kFeatTile;
    const int ncg = (s.dv + kColGroup - 1) / kColGroup;

    size_t sm1 = sizeof(float) * (size_t)(s.C * s.d + s.C * kColGroup);
    sm1 = sm1 > sizeof(float) * kFeatTile * kStride ? sm1 : sizeof(float) * kFeatTile * kStride;
    cudaFuncSetAttribute(chunk_state_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm1);
    {
        TraceScope tr("simt_chunk_state", stream);
        chunk_state_kernel<T><<<dim3(NC, BH, nft * ncg), kFeatTile, sm1, stream>>>(
            k, v, st, s.T, s.d, s.dv, s.C, n, NC, nft, mp);
    }
    const int64_t E = (int64_t)n * (s.dv + 1);
    float *part_ws = st + (size_t)BH * NC * E;   // part totals of the two-level scan
    cudaError_t e = scan_exclusive_launch(st, BH, NC, E, "simt_scan", stream, so, s.dv + 1,
                                          nullptr, part_ws);
    if (e != cudaSuccess) return e;

    const size_t sm3 = sizeof(float) *
                       (size_t)(2 * s.d * s.C + s.C * kColGroup + kStageRows * kRow);
    cudaFuncSetAttribute(output_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm3);
    {
        TraceScope tr("simt_output", stream);
        output_kernel<T><<<dim3(NC, BH, ncg), s.C, sm3, stream>>>(q, k, v, st, out, s.T, s.d,
                                                                    s.dv, s.C, n, NC, mp);
    }
    return cudaGetLastError();
}

}  // namespace

// Parts of the two-level scan for a record set (1: the one-pass scan).  The
// one-pass scan is used while one thread per four elements fills the GPU; the
// environment variable KATA_CHUNK_SCAN=sequential or =blocked forces either
// form (both give the same exclusive prefix; for measuring them).
int scan_parts(int BH, int NC, int64_t E, bool have_ws) {
    if (!have_ws || E % 4 != 0 || NC < 32) return 1;
    const char *env0 = getenv("KATA_CHUNK_SCAN");
    if (NC < 128 && !(env0 && strcmp(env0, "blocked") == 0)) return 1;   // too few parts to pay
    const int cap = NC / 16;   // the workspace holds NC / 16 + 1 parts per head
    const char *env = getenv("KATA_CHUNK_SCAN");
    const bool force_seq = env && strcmp(env, "sequential") == 0;
    const bool force_blk = env && strcmp(env, "blocked") == 0;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            sms = v;
        else
            sms = 148;
        cudaGetLastError();
    }
    const int64_t threads = (E / 4) * BH, want = (int64_t)sms * 2048;
    if (force_seq || (!force_blk && threads >= want / 2)) return 1;
    int64_t P = (want + threads - 1) / threads;
    P = P < 2 ? 2 : P > cap ? cap : P;
    const int L = (int)((NC + P - 1) / P);
    return (NC + L - 1) / L;
}

cudaError_t scan_exclusive_launch(float *data, int BH, int n, int64_t E, const char *stage,
                                  cudaStream_t stream, const StateOut &so, int W, float *totals,
                                  float *part_ws) {
    if (so.state && (W < 2 || E % W != 0)) return cudaErrorInvalidValue;
    const int P = scan_parts(BH, n, E, part_ws != nullptr);
    if (P > 1) {
        const int L = (n + P - 1) / P;
        const unsigned gx = (unsigned)((E / 4 + 255) / 256);
        TraceScope tr("simt_scan_blocked", stream);
        scan_part_totals<<<dim3(gx, BH, P), 256, 0, stream>>>(data, part_ws, n, E, L, P);
        scan_part_offsets<<<dim3(gx, BH), 256, 0, stream>>>(part_ws, P, E, so.state, so.z, W,
                                                             totals);
        scan_part_apply<<<dim3(gx, BH, P), 256, 0, stream>>>(data, part_ws, n, E, L, P);
        return cudaGetLastError();
    }
    TraceScope tr(stage, stream);
    if (E % 4 != 0)
        scan_kernel_scalar<<<dim3((unsigned)((E + 255) / 256), BH), 256, 0, stream>>>(
            data, n, E, so.state, so.z, W, totals);
    else
        scan_kernel<<<dim3((unsigned)((E / 4 + 255) / 256), BH), 256, 0, stream>>>(
            data, n, E, so.state, so.z, W, totals);
    return cudaGetLastError();
}

size_t simt_workspace_bytes(const FwdShape &s, const MapSpec &map) {
    // per-chunk states, then the part totals of the two-level scan (NC / 16 + 1 parts)
    return sizeof(float) * (size_t)s.BH() * ((size_t)s.NC() + (size_t)(s.NC() / 16 + 1)) *
           (size_t)map.n(s.d) * (size_t)(s.dv + 1);
}

cudaError_t simt_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                         void *out, void *workspace, cudaStream_t stream, const StateOut &so,
                         const MapSpec &map) {
    float *st = static_cast<float *>(workspace);
    if (s.dtype == 0)
        return simt_forward_t<float>(s, (const float *)q, (const float *)k, (const float *)v,
                                     (float *)out, st, stream, so, map);
    return simt_forward_t<__nv_bfloat16>(s, (const __nv_bfloat16 *)q,
                                         (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
                                         (__nv_bfloat16 *)out, st, stream, so, map);
}

cudaError_t lift_launch(const void *x, float *phi, int64_t rows, int d, int dtype,
                        cudaStream_t stream, const MapSpec &map) {
    const int n = map.n(d);
    const int64_t total = rows * n;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    TraceScope tr("lift", stream);
    if (dtype == 0)
        lift_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>((const float *)x, phi, rows, d, n,
                                                                 map);
    else
        lift_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
            (const __nv_bfloat16 *)x, phi, rows, d, n, map);
    return cudaGetLastError();
}

}  // namespace kata
