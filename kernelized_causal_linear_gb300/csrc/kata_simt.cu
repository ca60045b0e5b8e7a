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
// Stages 1 and 3 are register-tiled products (8 rows x 4 columns per thread)
// over 32-deep shared-memory slabs.  The feature lift (Sec. 3.1) is fused: psi
// entries are formed in the slabs from the q/k rows staged in shared memory and
// never written to global memory.  The intra-chunk weights use the closed form of
// psi(q).psi(k): (q.k)^2 for the full map, sum_a (q_a.k_a)^2 for M_g,
// eps^2 m + eps s (|q|^2 + |k|^2) + s^2 sum_{a,b} (q_a.k_b)^2 for Sigma_g
// (Sec. 4.1, reduced PSD families), and sum_i (q_i^+ + eps)(k_i^+ + eps) for the
// orthant map (one feature per coordinate, the pages' linear-state family).
//
// Workspace: per-chunk states [B*H][N_C][n][dv+1] fp32, scanned in place.
#include <cstdlib>
#include <cstring>

#include "kata_map.cuh"
#include "kata_simt_common.cuh"

namespace kata {
namespace {


// ---------------------------------------------------------------- tiles
constexpr int kTM = 8;            // rows per thread tile
constexpr int kTN = 4;            // value columns per thread tile
constexpr int kKS = 32;           // depth of one shared-memory slab
constexpr int kSlabCols = 64;     // value columns per block (dv = 128: two blocks)
constexpr int kMaxThreads = 288;  // 16 row groups x 16 column groups + the normaliser warp
// Both tiled kernels are compiled for at most 112 registers a thread, so that two
// blocks of kMaxThreads fit on an SM.

// Thread roles of a block of ng row groups x ncg column groups: thread tid < ng * ncg
// owns row group tid / ncg and column group tid % ncg; the warp after the value
// threads (rounded up to whole warps) owns the normaliser, lane l row group l.
struct Roles {
    int rg, cg, nl;
    bool val, nrm;
    __device__ Roles(int ng, int ncg) {
        const int tid = threadIdx.x, nval = ng * ncg, nvp = (nval + 31) & ~31;
        val = tid < nval;
        rg = val ? tid / ncg : 0;
        cg = val ? tid % ncg : 0;
        nl = tid - nvp;
        nrm = nl >= 0 && nl < ng;
    }
};
__host__ __device__ inline int block_threads(int ng, int ncg) {
    return ((ng * ncg + 31) & ~31) + 32;
}

// acc[i][j] += A[kk][TM rg + i] * B[kk][4 cg + j] over one slab (A: kKS rows of
// lda, B: kKS rows of kSlabCols); TM = 8, 4 or 2 rows per thread.
template <int TM>
__device__ __forceinline__ void load_rows(const float *p, float (&x)[TM]) {
    if constexpr (TM == 8) {
        const float4 a0 = *reinterpret_cast<const float4 *>(p);
        const float4 a1 = *reinterpret_cast<const float4 *>(p + 4);
        x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w;
        x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
    } else if constexpr (TM == 4) {
        const float4 a0 = *reinterpret_cast<const float4 *>(p);
        x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w;
    } else {
        const float2 a0 = *reinterpret_cast<const float2 *>(p);
        x[0] = a0.x; x[1] = a0.y;
    }
}
template <int TM>
__device__ __forceinline__ void slab_fma(const float *A, int lda, const float *B, int rg, int cg,
                                         float (&acc)[TM][kTN]) {
    const float *a = A + rg * TM;
    const float *b = B + cg * kTN;
#pragma unroll 8
    for (int kk = 0; kk < kKS; ++kk) {
        float av[TM];
        load_rows<TM>(a + kk * lda, av);
        const float4 b0 = *reinterpret_cast<const float4 *>(b + kk * kSlabCols);
        const float bv[kTN] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < kTN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

// den[i] += A[kk][TM rg + i] * z[kk] over one slab (the normaliser column).
template <int TM>
__device__ __forceinline__ void slab_den(const float *A, int lda, const float *z, int rg,
                                         float (&den)[TM]) {
    const float *a = A + rg * TM;
#pragma unroll 8
    for (int kk = 0; kk < kKS; ++kk) {
        float av[TM];
        load_rows<TM>(a + kk * lda, av);
        const float zz = z[kk];
#pragma unroll
        for (int i = 0; i < TM; ++i) den[i] = fmaf(av[i], zz, den[i]);
    }
}

// Feature table of features f0 .. f0 + cnt - 1 (psi_f = A_f * sum_a x_i x_j + B_f,
// coordinates packed as i0 | j0 << 16; orthant: psi_f = the transformed x_i0).
__device__ __forceinline__ void feature_table(int f0, int cnt, int n, int d, const MapSpec &mp,
                                              int *fij, float *fA, float *fB) {
    for (int fl = threadIdx.x; fl < cnt; fl += blockDim.x) {
        const int f = f0 + fl;
        int ij = 0;
        float a = 0.f, b = 0.f;
        if (f < n) {
            const Feat ft = map_feature(f, d, mp);
            ij = ft.i0 | (ft.j0 << 16);
            a = ft.cf * ft.scl;
            b = ft.cf * ft.add;
        }
        fij[fl] = ij;
        fA[fl] = a;
        fB[fl] = b;
    }
}

// psi_f of the vector x (coordinate c at x[c * xs]) from its table entry.
// KIND: the map fixed at compile time (0 full, 3 orthant) or -1 (read at run time).
template <int KIND>
__device__ __forceinline__ float psi_at(const float *x, int xs, int ij, float A, float B,
                                        int terms, int step, bool orth) {
    const int i0 = ij & 0xffff, j0 = ij >> 16;
    if constexpr (KIND == 0) return fmaf(A, x[i0 * xs] * x[j0 * xs], B);   // one term, no eps
    if constexpr (KIND == 3) return x[i0 * xs];
    if (orth) return x[i0 * xs];
    float e = 0.f;
    for (int a = 0; a < terms; ++a)
        e = fmaf(x[(i0 + a * step) * xs], x[(j0 + a * step) * xs], e);
    return fmaf(A, e, B);
}

// The orthant map's coordinate transform max(x, 0) + eps; other maps use x.
__device__ __forceinline__ float map_coord(float x, const MapSpec &mp) {
    return mp.kind == 3 ? fmaxf(x, 0.f) + mp.eps : x;
}

// Gate products of a chunk (one thread, tc <= C steps): gam[t] = gamma_t,
// pre[t] = prod_{r<=t} gamma_r from the chunk start, suf[t] = prod_{r>t} gamma_r
// to the chunk end; positions past tc get gam 1 and pre, suf 0.  Running
// products of the gates themselves, so gamma = 0 and gamma = 1 are exact.
__device__ __forceinline__ void chunk_gates(const float *__restrict__ g, int tc, int C,
                                            float *gam, float *pre, float *suf) {
    if (threadIdx.x == 0) {
        float p = 1.f;
        for (int t = 0; t < C; ++t) {
            const float x = t < tc ? g[t] : 1.f;
            gam[t] = x;
            p *= x;
            pre[t] = t < tc ? p : 0.f;
        }
        float s = 1.f;
        for (int t = C - 1; t >= 0; --t) {
            suf[t] = t < tc ? s : 0.f;
            if (t < tc) s *= gam[t];
        }
    }
}

template <typename T>
__device__ __forceinline__ void store4(T *p, const float (&x)[kTN]);
template <>
__device__ __forceinline__ void store4<float>(float *p, const float (&x)[kTN]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, const float (&x)[kTN]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

// 4-byte asynchronous global -> shared copy (zero fill when !ok; src must then
// still be a valid address) and its group commit / wait.
__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool ok) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src),
                 "r"(ok ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// The chunk's value rows (the slab's columns, zero past tc rows or ncol columns)
// into shared memory as they are stored: vr[t][0 .. kSlabCols).
template <typename T>
__device__ __forceinline__ void stage_values(const T *vc, int dv, int tc, int C, int ncol, T *vr) {
    for (int e = threadIdx.x; e < C * kSlabCols; e += blockDim.x) {
        const int t = e / kSlabCols, cc = e % kSlabCols;
        vr[e] = (t < tc && cc < ncol) ? vc[(size_t)t * dv + cc] : from_f<T>(0.f);
    }
}

// ---------------------------------------------------------------- stage 1
// One block per (chunk, head, column slab), walking the n features in ntile
// tiles of ng row groups (8 features each): per tile, features x the slab's
// value columns over the chunk's tokens in 32-token slabs.  The key rows, the
// value rows and the feature table are staged once for all tiles.  Gated: v_s
// and the ones column scaled by suf_s.
template <typename T, bool kGated, int KIND>
__global__ void __maxnreg__(112)
tiled_state_kernel(const T *__restrict__ k, const T *__restrict__ v,
                   const float *__restrict__ gamma, float *__restrict__ st,
                   float *__restrict__ cgate, int T_, int d, int dv, int C, int n, int NC,
                   int ntile, int ng, MapSpec mp) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, bh = blockIdx.y, cs = blockIdx.z;
    const int t0 = c * C, tc = min(C, T_ - t0);
    const int W = dv + 1, FT = ng * kTM;
    const int ncol = min(kSlabCols, dv - cs * kSlabCols), ncg = ncol / kTN;
    const Roles ro(ng, ncg);

    float *ks = sm;                          // [C][d] key rows (map coordinates)
    float *As = ks + C * d;                  // [2][kKS][FT]   psi_f(k_s)
    float *Bs = As + 2 * kKS * FT;           // [2][kKS][kSlabCols]  v_s (decayed)
    float *zs = Bs + 2 * kKS * kSlabCols;    // [2][kKS]       1 (decayed)
    float *gam = zs + 2 * kKS;               // [C] gates, prefix and suffix products
    float *pre = gam + C;
    float *suf = pre + C;
    float *fA = suf + C;                     // [n] feature table
    float *fB = fA + n;
    int *fij = reinterpret_cast<int *>(fB + n);
    T *vr = reinterpret_cast<T *>(fij + n);  // [C][kSlabCols] value rows as stored

    const T *kc = k + ((size_t)bh * T_ + t0) * d;
    const T *vc = v + ((size_t)bh * T_ + t0) * dv + cs * kSlabCols;
    for (int e = threadIdx.x; e < C * d; e += blockDim.x)
        ks[e] = e < tc * d ? map_coord(to_f(kc[e]), mp) : 0.f;
    stage_values(vc, dv, tc, C, ncol, vr);
    if (kGated) chunk_gates(gamma + (size_t)bh * T_ + t0, tc, C, gam, pre, suf);
    feature_table(0, n, n, d, mp, fij, fA, fB);
    __syncthreads();
    if (kGated && cs == 0 && threadIdx.x == 0) cgate[(size_t)bh * NC + c] = pre[tc - 1];

    const bool orth = mp.kind == 3;
    const int terms = mp.kind == 2 ? mp.g : 1, step = mp.kind == 2 ? d / mp.g : 0;
    const int nks = (tc + kKS - 1) / kKS;
    // fill units: feature fl with tokens k0, k0 + nsplit, ... of a slab
    const int nsplit = blockDim.x >= FT ? blockDim.x / FT : 1;
    float *rec = st + ((size_t)bh * NC + c) * (size_t)n * W;
    int slab = 0;   // slabs over all tiles: buffer parity
    for (int ft = 0; ft < ntile; ++ft) {
        const int f0 = ft * FT;
        float acc[kTM][kTN] = {};
        float den[kTM] = {};
        for (int j = 0; j < nks; ++j, ++slab) {
            const int s0 = j * kKS;
            float *A = As + (slab & 1) * kKS * FT;
            float *B = Bs + (slab & 1) * kKS * kSlabCols;
            float *z = zs + (slab & 1) * kKS;
            for (int u = threadIdx.x; u < FT * nsplit; u += blockDim.x) {
                const int fl = u % FT, f = f0 + fl;
                const int ij = f < n ? fij[f] : 0;
                const float fa = f < n ? fA[f] : 0.f, fb = f < n ? fB[f] : 0.f;
                for (int kk = u / FT; kk < kKS; kk += nsplit) {
                    const int t = s0 + kk;
                    A[kk * FT + fl] = (t < tc && f < n)
                                          ? psi_at<KIND>(ks + t * d, 1, ij, fa, fb, terms, step, orth)
                                          : 0.f;
                }
            }
            for (int e = threadIdx.x; e < kKS * kSlabCols; e += blockDim.x) {
                float x = to_f(vr[s0 * kSlabCols + e]);
                if (kGated) x *= suf[s0 + e / kSlabCols];
                B[e] = x;
            }
            if (threadIdx.x < kKS) {
                const int t = s0 + threadIdx.x;
                z[threadIdx.x] = t < tc ? (kGated ? suf[t] : 1.f) : 0.f;
            }
            __syncthreads();
            if (ro.val) slab_fma<kTM>(A, FT, B, ro.rg, ro.cg, acc);
            else if (ro.nrm) slab_den<kTM>(A, FT, z, ro.nl, den);
        }
        if (ro.val) {
#pragma unroll
            for (int i = 0; i < kTM; ++i) {
                const int f = f0 + ro.rg * kTM + i;
                if (f < n) {
                    float *row = rec + (size_t)f * W + cs * kSlabCols + ro.cg * kTN;
#pragma unroll
                    for (int jj = 0; jj < kTN; ++jj) row[jj] = acc[i][jj];
                }
            }
        } else if (ro.nrm && cs == 0) {
#pragma unroll
            for (int i = 0; i < kTM; ++i) {
                const int f = f0 + ro.nl * kTM + i;
                if (f < n) rec[(size_t)f * W + dv] = den[i];
            }
        }
    }
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
// Masked intra-chunk weights of rows r0 .. r0+7 against keys s, s+1 (map
// coordinates transposed in qsT, ksT [d][C]): (q.k)^2 for the full map,
// sum_a (q_a.k_a)^2 for M_g, eps^2 m + eps s (|q|^2 + |k|^2) + s^2 sum_{a,b}
// (q_a.k_b)^2 for Sigma_g (Sec. 4.1, reduced PSD families; qn, kn the squared
// norms), the plain dot of the transformed vectors for the orthant map.
template <int KIND>
__device__ __forceinline__ void weight_tile(const float *qsT, const float *ksT, const float *qn,
                                            const float *kn, int C, int d, const MapSpec &mp,
                                            int r0, int s, float (&p)[kTM][2]) {
    const int g = KIND >= 0 ? 1 : (mp.kind == 1 || mp.kind == 2) ? mp.g : 1, m = d / g;
    const bool sq = KIND == 0 || (KIND < 0 && mp.kind != 3);
#pragma unroll
    for (int i = 0; i < kTM; ++i) p[i][0] = p[i][1] = 0.f;
    for (int a = 0; a < g; ++a) {
        const int blo = (KIND < 0 && mp.kind == 2) ? 0 : a, bhi = (KIND < 0 && mp.kind == 2) ? g : a + 1;
        for (int b = blo; b < bhi; ++b) {
            float pa[kTM][2] = {};
            const float *qp = qsT + (size_t)(a * m) * C + r0;
            const float *kp = ksT + (size_t)(b * m) * C + s;
#pragma unroll 2
            for (int i = 0; i < m; ++i) {
                const float4 q0 = *reinterpret_cast<const float4 *>(qp + i * C);
                const float4 q1 = *reinterpret_cast<const float4 *>(qp + i * C + 4);
                const float2 k2 = *reinterpret_cast<const float2 *>(kp + i * C);
                const float qv[kTM] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int r = 0; r < kTM; ++r) {
                    pa[r][0] = fmaf(qv[r], k2.x, pa[r][0]);
                    pa[r][1] = fmaf(qv[r], k2.y, pa[r][1]);
                }
            }
#pragma unroll
            for (int r = 0; r < kTM; ++r)
#pragma unroll
                for (int u = 0; u < 2; ++u) p[r][u] += sq ? pa[r][u] * pa[r][u] : pa[r][u];
        }
    }
    if (KIND < 0 && mp.kind == 2) {
#pragma unroll
        for (int r = 0; r < kTM; ++r)
#pragma unroll
            for (int u = 0; u < 2; ++u)
                p[r][u] = mp.eps * mp.eps * m + mp.eps * mp.scale * (qn[r0 + r] + kn[s + u]) +
                          mp.scale * mp.scale * p[r][u];
    }
}

// One block per (chunk, head, column slab): C rows (C / 8 row groups) x the
// slab's value columns; inner axis the n features of Psi(Q_c), then the chunk's
// keys in 32-key slabs from the last to the first.  Gated: psi(q_r) scaled by
// pre_r and the weight of key s <= r by prod_{u=s+1}^{r} gamma_u, a running
// product per row walked from s = r down (carried across the key slabs).
template <typename T, bool kGated, int TM, int KIND>
__global__ void __maxnreg__(112)
tiled_output_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    const float *__restrict__ gamma, const float *__restrict__ st,
                    T *__restrict__ out, int T_, int d, int dv, int C, int n, int NC, MapSpec mp,
                    int normalize) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, bh = blockIdx.y, cs = blockIdx.z;
    const int t0 = c * C, tc = min(C, T_ - t0);
    const int W = dv + 1, ng = C / TM;
    const int ncol = min(kSlabCols, dv - cs * kSlabCols), ncg = ncol / kTN;
    const Roles ro(ng, ncg);

    float *qsT = sm;                         // [d][C] query map coordinates, transposed
    float *ksT = qsT + d * C;                // [d][C] key map coordinates, transposed
    float *As = ksT + d * C;                 // [2][kKS][C]  psi_f(q_r) or masked weights
    float *Bs = As + 2 * kKS * C;            // [2][kKS][kSlabCols]  S_pre rows or v_s
    float *zs = Bs + 2 * kKS * kSlabCols;    // [2][kKS]     Z_pre or 1
    float *qn = zs + 2 * kKS;                // [C] squared norms (Sigma_g)
    float *kn = qn + C;
    float *gam = kn + C;                     // [C] gates, prefix and suffix products
    float *pre = gam + C;
    float *suf = pre + C;
    float *arun = suf + C;                   // [C] running intra-chunk decay per row
    float *dsh = arun + C;                   // [C] denominators
    float *fA = dsh + C;                     // [n] feature table
    float *fB = fA + n;
    int *fij = reinterpret_cast<int *>(fB + n);
    T *vr = reinterpret_cast<T *>(fij + n);  // [C][kSlabCols] value rows as stored

    // prefix-state rows of feature slab j (the slab's columns and Z) into buffer
    // j & 1, asynchronously: issued one slab ahead of its product
    const float *sp = st + ((size_t)bh * NC + c) * (size_t)n * W;
    const int nfs = (n + kKS - 1) / kKS;
    auto issue_state_slab = [&](int j) {
        float *B = Bs + (j & 1) * kKS * kSlabCols;
        float *z = zs + (j & 1) * kKS;
        const int f0 = j * kKS;
        for (int e = threadIdx.x; e < kKS * kSlabCols; e += blockDim.x) {
            const int kk = e / kSlabCols, cc = e % kSlabCols, f = f0 + kk;
            const bool ok = f < n && cc < ncol;
            cp_async4(B + e, ok ? sp + (size_t)f * W + cs * kSlabCols + cc : sp, ok);
        }
        if (threadIdx.x < kKS) {
            const int f = f0 + threadIdx.x;
            cp_async4(z + threadIdx.x, f < n ? sp + (size_t)f * W + dv : sp, f < n);
        }
        cp_async_commit();
    };
    issue_state_slab(0);

    const T *qc = q + ((size_t)bh * T_ + t0) * d;
    const T *kc = k + ((size_t)bh * T_ + t0) * d;
    const T *vc = v + ((size_t)bh * T_ + t0) * dv + cs * kSlabCols;
    for (int e = threadIdx.x; e < C * d; e += blockDim.x) {
        const int t = e % C, i = e / C;   // consecutive threads: consecutive tokens
        const bool ok = t < tc;
        qsT[e] = ok ? map_coord(to_f(qc[(size_t)t * d + i]), mp) : 0.f;
        ksT[e] = ok ? map_coord(to_f(kc[(size_t)t * d + i]), mp) : 0.f;
    }
    stage_values(vc, dv, tc, C, ncol, vr);
    if (kGated) chunk_gates(gamma + (size_t)bh * T_ + t0, tc, C, gam, pre, suf);
    for (int r = threadIdx.x; r < C; r += blockDim.x) arun[r] = 1.f;
    feature_table(0, n, n, d, mp, fij, fA, fB);
    __syncthreads();
    if (mp.kind == 2) {
        for (int r = threadIdx.x; r < C; r += blockDim.x) {
            float a = 0.f, b = 0.f;
            for (int i = 0; i < d; ++i) {
                a = fmaf(qsT[i * C + r], qsT[i * C + r], a);
                b = fmaf(ksT[i * C + r], ksT[i * C + r], b);
            }
            qn[r] = a;
            kn[r] = b;
        }
        // ordered before their first use by the slab barrier below
    }

    const bool orth = mp.kind == 3;
    const int terms = mp.kind == 2 ? mp.g : 1, step = mp.kind == 2 ? d / mp.g : 0;
    float acc[TM][kTN] = {};
    float den[TM] = {};
    const int nks = (tc + kKS - 1) / kKS;
    for (int j = 0; j < nfs + nks; ++j) {
        float *A = As + (j & 1) * kKS * C;
        float *B = Bs + (j & 1) * kKS * kSlabCols;
        float *z = zs + (j & 1) * kKS;
        const bool keys = j >= nfs;
        const int s0 = keys ? (nks - 1 - (j - nfs)) * kKS : 0;
        if (!keys) {
            const int f0 = j * kKS;
            const int nw = blockDim.x / 32, w = threadIdx.x / 32, lane = threadIdx.x % 32;
            for (int kk = w; kk < kKS; kk += nw) {   // one feature per warp, lanes over rows
                const int f = f0 + kk;
                float *arow = A + kk * C;
                if (f < n) {
                    const int ij = fij[f];
                    const float fa = fA[f], fb = fB[f];
                    for (int r = lane; r < C; r += 32) {
                        float x = psi_at<KIND>(qsT + r, C, ij, fa, fb, terms, step, orth);
                        if (kGated) x *= pre[r];
                        arow[r] = x;
                    }
                } else {
                    for (int r = lane; r < C; r += 32) arow[r] = 0.f;
                }
            }
        } else {
            for (int tile = threadIdx.x; tile < (C / kTM) * (kKS / 2); tile += blockDim.x) {
                const int r0 = (tile / (kKS / 2)) * kTM, kp = tile % (kKS / 2), s = s0 + 2 * kp;
                float p[kTM][2];
                weight_tile<KIND>(qsT, ksT, qn, kn, C, d, mp, r0, s, p);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float m8[kTM];
#pragma unroll
                    for (int i = 0; i < kTM; ++i)
                        m8[i] = (s + u <= r0 + i && s + u < tc) ? p[i][u] : 0.f;
                    float *dst = A + (2 * kp + u) * C + r0;
                    *reinterpret_cast<float4 *>(dst) = make_float4(m8[0], m8[1], m8[2], m8[3]);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(m8[4], m8[5], m8[6], m8[7]);
                }
            }
            for (int e = threadIdx.x; e < kKS * kSlabCols; e += blockDim.x)
                B[e] = to_f(vr[s0 * kSlabCols + e]);
            if (threadIdx.x < kKS) z[threadIdx.x] = s0 + (int)threadIdx.x < tc ? 1.f : 0.f;
        }
        cp_async_wait_all();   // this slab's state rows (issued last iteration) have landed
        __syncthreads();
        if (j + 1 < nfs) issue_state_slab(j + 1);   // its buffer's last readers are past the barrier
        if (kGated && keys) {
            for (int r = threadIdx.x; r < tc; r += blockDim.x) {
                if (r < s0) continue;
                float a = arun[r];
#pragma unroll 1
                for (int kk = min(kKS - 1, r - s0); kk >= 0; --kk) {
                    A[kk * C + r] *= a;
                    a *= gam[s0 + kk];
                }
                arun[r] = a;
            }
            __syncthreads();
        }
        const bool skip = keys && (ro.val ? ro.rg : ro.nl) * TM + TM - 1 < s0;   // all above the diagonal
        if (ro.val && !skip) slab_fma<TM>(A, C, B, ro.rg, ro.cg, acc);
        else if (ro.nrm && !skip) slab_den<TM>(A, C, z, ro.nl, den);
    }

    if (ro.nrm)
#pragma unroll
        for (int i = 0; i < TM; ++i) dsh[ro.nl * TM + i] = den[i];
    __syncthreads();
    if (ro.val) {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = ro.rg * TM + i;
            if (r >= tc) break;
            const float dn = dsh[r];
            const float inv = dn > 0.f ? 1.f / dn : 0.f;   // Eq. 20; a zero denominator gives 0
            float o[kTN];
#pragma unroll
            for (int jj = 0; jj < kTN; ++jj)
                o[jj] = normalize ? (dn > 0.f ? acc[i][jj] * inv : 0.f) : acc[i][jj];
            store4<T>(out + ((size_t)bh * T_ + t0 + r) * dv + cs * kSlabCols + ro.cg * kTN, o);
        }
    }
}

}  // namespace

namespace simt {

// Tiling of a state launch: n features in ntile tiles of ng <= 16 row groups,
// as even as the row groups allow.
static void state_tiling(int n, int &ntile, int &ng) {
    const int n8 = (n + kTM - 1) / kTM;
    ntile = (n8 + 15) / 16;
    ng = (n8 + ntile - 1) / ntile;
}

template <typename T>
cudaError_t state_launch(const FwdShape &s, const T *k, const T *v, const float *gamma,
                         float *st, float *cgate, const MapSpec &mp, cudaStream_t stream,
                         const char *stage) {
    const int n = mp.n(s.d), NC = s.NC(), BH = s.BH();
    int ntile, ng;
    state_tiling(n, ntile, ng);
    const int ncs = (s.dv + kSlabCols - 1) / kSlabCols;
    const int ncg = (s.dv < kSlabCols ? s.dv : kSlabCols) / kTN;
    const int FT = ng * kTM;
    const int threads = block_threads(ng, ncg);
    if (threads > kMaxThreads) return cudaErrorInvalidConfiguration;   // the 112-register budget
    const size_t smem = sizeof(float) * ((size_t)s.C * s.d + 2 * kKS * FT + 2 * kKS * kSlabCols +
                                         2 * kKS + 3 * s.C + 3 * (size_t)n) +
                        sizeof(T) * (size_t)s.C * kSlabCols;
    // the full map (and every gated call) and the orthant map with their feature and
    // weight forms fixed at compile time; the reduced maps read the map at run time
    auto kern = gamma          ? tiled_state_kernel<T, true, 0>
                : mp.kind == 0 ? tiled_state_kernel<T, false, 0>
                : mp.kind == 3 ? tiled_state_kernel<T, false, 3>
                               : tiled_state_kernel<T, false, -1>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    TraceScope tr(stage, stream);
    kern<<<dim3(NC, BH, ncs), threads, smem, stream>>>(
        k, v, gamma, st, cgate, s.T, s.d, s.dv, s.C, n, NC, ntile, ng, mp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t output_launch(const FwdShape &s, const T *q, const T *k, const T *v,
                          const float *gamma, const float *st, T *out, const MapSpec &mp,
                          int normalize, cudaStream_t stream, const char *stage) {
    const int n = mp.n(s.d), NC = s.NC(), BH = s.BH();
    const int ncs = (s.dv + kSlabCols - 1) / kSlabCols;
    const int ncg = (s.dv < kSlabCols ? s.dv : kSlabCols) / kTN;
    const int threads = block_threads(s.C / kTM, ncg);
    if (threads > kMaxThreads) return cudaErrorInvalidConfiguration;   // the 112-register budget
    const size_t smem = sizeof(float) * (2 * (size_t)s.d * s.C + 2 * kKS * s.C +
                                         2 * kKS * kSlabCols + 2 * kKS + 7 * s.C + 3 * (size_t)n) +
                        sizeof(T) * (size_t)s.C * kSlabCols;
    // 8-row thread tiles for every chunk length: 4 x 4 tiles (twice the threads
    // at C = 64) measured slower, bound by the shared-memory loads
    auto kern = gamma          ? tiled_output_kernel<T, true, kTM, 0>
                : mp.kind == 0 ? tiled_output_kernel<T, false, kTM, 0>
                : mp.kind == 3 ? tiled_output_kernel<T, false, kTM, 3>
                               : tiled_output_kernel<T, false, kTM, -1>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    TraceScope tr(stage, stream);
    kern<<<dim3(NC, BH, ncs), threads, smem, stream>>>(
        q, k, v, gamma, st, out, s.T, s.d, s.dv, s.C, n, NC, mp, normalize);
    return cudaGetLastError();
}

#define KATA_SIMT_INSTANTIATE(T)                                                              \
    template cudaError_t state_launch<T>(const FwdShape &, const T *, const T *, const float *, \
                                         float *, float *, const MapSpec &, cudaStream_t,      \
                                         const char *);                                        \
    template cudaError_t output_launch<T>(const FwdShape &, const T *, const T *, const T *,    \
                                          const float *, const float *, T *, const MapSpec &,  \
                                          int, cudaStream_t, const char *);
KATA_SIMT_INSTANTIATE(float)
KATA_SIMT_INSTANTIATE(__nv_bfloat16)
#undef KATA_SIMT_INSTANTIATE

}  // namespace simt

namespace {

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
    cudaError_t e = simt::state_launch<T>(s, k, v, nullptr, st, nullptr, mp, stream,
                                          "simt_chunk_state");
    if (e != cudaSuccess) return e;
    const int64_t E = (int64_t)n * (s.dv + 1);
    float *part_ws = st + (size_t)BH * NC * E;   // part totals of the two-level scan
    e = scan_exclusive_launch(st, BH, NC, E, "simt_scan", stream, so, s.dv + 1, nullptr,
                              part_ws);
    if (e != cudaSuccess) return e;

    return simt::output_launch<T>(s, q, k, v, nullptr, st, out, mp, 1, stream, "simt_output");
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
