// GatedKATA chunked forward on CUDA cores (fp32 FFMA).
//
// The gated recurrence of the pages' "multiplicative scalar state gate"
// variant (appendix on recurrent variants; Sec. 5.2):
//   S_t = gamma_t S_{t-1} + psi(k_t) v_t^T,  Z_t = gamma_t Z_{t-1} + psi(k_t),
// so write s reaches token t with the weight a_ts = prod_{r=s+1}^{t} gamma_r,
// read out as psi(q_t)^T S_t / psi(q_t)^T Z_t, or psi(q_t)^T S_t without the
// denominator.  In chunk form (chunk c = tokens c0 .. c0+L-1):
//
//   1. chunk state   S_loc[c] = sum_s suf_s psi(k_s) [v_s | 1]^T,
//                    suf_s = prod_{r=s+1}^{c0+L-1} gamma_r;  g_c = prod_{r in c} gamma_r
//   2. gated scan    S_pre[0] = 0,  S_pre[c+1] = g_c S_pre[c] + S_loc[c]
//   3. output        N_t = pre_t psi(q_t) [S_pre | Z_pre][c] + sum_{s<=t in c} a_ts w_ts [v_s | 1],
//                    pre_t = prod_{r=c0}^{t} gamma_r,  w_ts = (q_t . k_s)^2
//
// Every decay is a running product of the gates themselves (no logarithms), so
// gamma = 0 (a reset) and gamma = 1 are exact and nothing cancels.
// Workspace: per-chunk states [B*H][N_C][n][dv+1] fp32 (scanned in place),
// then the chunk gate products [B*H][N_C].
#include "kata_simt_common.cuh"

namespace kata {
namespace {

constexpr int kMaxC = 128;
using namespace simt;

// Gate products of the chunk starting at t0 with tc tokens, into shared memory:
// gam[t] = gamma, pre[t] = prod_{r<=t} gamma_r (from the chunk start),
// suf[t] = prod_{r>t} gamma_r (to the chunk end).  One thread, tc <= 128 steps.
__device__ __forceinline__ void chunk_gates(const float *__restrict__ g, int tc, float *gam,
                                            float *pre, float *suf) {
    if (threadIdx.x == 0) {
        float p = 1.f;
        for (int t = 0; t < tc; ++t) {
            gam[t] = g[t];
            p *= gam[t];
            pre[t] = p;
        }
        float s = 1.f;
        for (int t = tc - 1; t >= 0; --t) {
            suf[t] = s;
            s *= gam[t];
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- stage 1
template <typename T>
__global__ void __launch_bounds__(kFeatTile)
gated_state_kernel(const T *__restrict__ k, const T *__restrict__ v,
                   const float *__restrict__ gamma, float *__restrict__ st,
                   float *__restrict__ cgate, int T_, int d, int dv, int C, int n, int NC,
                   int nft) {
    extern __shared__ __align__(16) float sm[];
    __shared__ float gam[kMaxC], pre[kMaxC], suf[kMaxC];
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
    chunk_gates(gamma + (size_t)bh * T_ + t0, tc, gam, pre, suf);
    if (ft == 0 && cg == 0 && threadIdx.x == 0) cgate[(size_t)bh * NC + c] = pre[tc - 1];

    float acc[kStride];
#pragma unroll
    for (int jj = 0; jj < kStride; ++jj) acc[jj] = 0.f;
    const int f = ft * kFeatTile + threadIdx.x;
    if (f < n) {
        int i, j;
        vech_pair(f, d, i, j);
        const float cf = i == j ? 1.f : kSqrt2;
        for (int t = 0; t < tc; ++t) {
            const float a = ks[t * d + i] * ks[t * d + j] * cf * suf[t];   // decayed psi(k_t)_f
            fma_row32(a, vs + t * kColGroup, acc);
            acc[kColGroup] += a;
        }
    }
    // through shared memory so that each warp writes contiguous row segments
    store_state_rows(acc, sm, st + ((size_t)bh * NC + c) * (size_t)n * W, ft, cg, cols, n, dv);
}

// ---------------------------------------------------------------- stage 2
// Exclusive gated prefix over chunks, per (b, h, element), in place:
// run = 0; per chunk c: store run, then run = g_c run + S_loc[c].  Four
// consecutive elements per thread (E is a multiple of 4 for every supported d).
// With state_out set, the inclusive total (the state after the last token) of
// element e = f * W + col goes to state_out[bh][f][col] or z_out[bh][f].
__global__ void __launch_bounds__(256)
gated_scan_kernel(float *__restrict__ st, const float *__restrict__ cgate, int NC, int64_t E,
                  float *__restrict__ state_out, float *__restrict__ z_out, int W) {
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t E4 = E >> 2;
    if (e4 >= E4) return;
    float4 *p = reinterpret_cast<float4 *>(st + (size_t)blockIdx.y * NC * E) + e4;
    const float *gc = cgate + (size_t)blockIdx.y * NC;
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
                const float g = gc[c + j];
                p[(size_t)j * E4] = run;
                run.x = fmaf(g, run.x, x[j].x);
                run.y = fmaf(g, run.y, x[j].y);
                run.z = fmaf(g, run.z, x[j].z);
                run.w = fmaf(g, run.w, x[j].w);
            }
        }
        p += (size_t)8 * E4;
    }
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

// ---------------------------------------------------------------- stage 3
// One block per (chunk, head, column group); thread r owns output row r.
template <typename T>
__global__ void __launch_bounds__(128)
gated_output_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    const float *__restrict__ gamma, const float *__restrict__ st,
                    T *__restrict__ out, int T_, int d, int dv, int C, int n, int NC,
                    int normalize) {
    extern __shared__ __align__(16) float sm[];
    __shared__ float gam[kMaxC], pre[kMaxC], suf[kMaxC];
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
    chunk_gates(gamma + (size_t)bh * T_ + t0, tc, gam, pre, suf);

    float acc[kStride];
#pragma unroll
    for (int jj = 0; jj < kStride; ++jj) acc[jj] = 0.f;

    // inter-chunk term psi(q_r) . [S_pre | Z_pre], features in packed order
    const float *sp = st + ((size_t)bh * NC + c) * (size_t)n * W;
    int fi = 0, fj = 0;
    for (int f0 = 0; f0 < n; f0 += kStageRows) {
        const int nf = min(kStageRows, n - f0);
        __syncthreads();
        stage_state_rows(sp, stg, f0, nf, cg, cols, dv);
        __syncthreads();
        for (int fr = 0; fr < nf; ++fr) {
            const float a = qsT[fi * C + r] * qsT[fj * C + r] * (fi == fj ? 1.f : kSqrt2);
            const float *sr = stg + fr * kRow;
            fma_row32(a, sr, acc);
            acc[kColGroup] = fmaf(a, sr[kColGroup], acc[kColGroup]);
            if (++fj == d) fj = ++fi;
        }
    }

    if (r < tc) {
        // the state before the chunk decays by the gates of tokens c0 .. r
        const float dec = pre[r];
#pragma unroll
        for (int jj = 0; jj < kStride; ++jj) acc[jj] *= dec;
        // intra-chunk: s = r, r-1, ..., with a_rs = prod_{u=s+1}^{r} gamma_u
        float a = 1.f;
        for (int s = r; s >= 0; --s) {
            float dot = 0.f;
            for (int i = 0; i < d; ++i) dot = fmaf(qsT[i * C + r], ks[s * d + i], dot);
            const float w = a * dot * dot;
            fma_row32(w, vs + s * kColGroup, acc);
            acc[kColGroup] += w;
            a *= gam[s];
        }
        const float den = acc[kColGroup];
        const float inv = den > 0.f ? 1.f / den : 0.f;
        T *orow = out + ((size_t)bh * T_ + t0 + r) * dv + cg * kColGroup;
#pragma unroll
        for (int jj = 0; jj < kColGroup; ++jj)
            if (jj < cols)
                orow[jj] = from_f<T>(normalize ? (den > 0.f ? acc[jj] * inv : 0.f) : acc[jj]);
    }
}

template <typename T>
cudaError_t gated_forward_t(const FwdShape &s, const T *q, const T *k, const T *v,
                            const float *gamma, T *out, float *st, cudaStream_t stream,
                            const StateOut &so, int normalize) {
    const int n = s.n(), NC = s.NC(), BH = s.BH();
    const int nft = (n + kFeatTile - 1) / kFeatTile;
    const int ncg = (s.dv + kColGroup - 1) / kColGroup;
    float *cgate = st + (size_t)BH * NC * n * (s.dv + 1);

    size_t sm1 = sizeof(float) * (size_t)(s.C * s.d + s.C * kColGroup);
    sm1 = sm1 > sizeof(float) * kFeatTile * kStride ? sm1 : sizeof(float) * kFeatTile * kStride;
    cudaFuncSetAttribute(gated_state_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm1);
    {
        TraceScope tr("gated_chunk_state", stream);
        gated_state_kernel<T><<<dim3(NC, BH, nft * ncg), kFeatTile, sm1, stream>>>(
            k, v, gamma, st, cgate, s.T, s.d, s.dv, s.C, n, NC, nft);
    }
    const int64_t E = (int64_t)n * (s.dv + 1);
    if (E % 4 != 0 || (so.state && !so.z)) return cudaErrorInvalidValue;
    {
        TraceScope tr("gated_scan", stream);
        gated_scan_kernel<<<dim3((unsigned)((E / 4 + 255) / 256), BH), 256, 0, stream>>>(
            st, cgate, NC, E, so.state, so.z, s.dv + 1);
    }
    const size_t sm3 = sizeof(float) *
                       (size_t)(2 * s.d * s.C + s.C * kColGroup + kStageRows * kRow);
    cudaFuncSetAttribute(gated_output_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm3);
    {
        TraceScope tr("gated_output", stream);
        gated_output_kernel<T><<<dim3(NC, BH, ncg), s.C, sm3, stream>>>(
            q, k, v, gamma, st, out, s.T, s.d, s.dv, s.C, n, NC, normalize);
    }
    return cudaGetLastError();
}

}  // namespace

size_t gated_workspace_bytes(const FwdShape &s) {
    return sizeof(float) * (size_t)s.BH() * (size_t)s.NC() * ((size_t)s.n() * (s.dv + 1) + 1);
}

cudaError_t gated_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                          const float *gamma, void *out, void *workspace, cudaStream_t stream,
                          const StateOut &so, int normalize) {
    if (s.C > kMaxC) return cudaErrorInvalidValue;
    float *st = static_cast<float *>(workspace);
    if (s.dtype == 0)
        return gated_forward_t<float>(s, (const float *)q, (const float *)k, (const float *)v,
                                      gamma, (float *)out, st, stream, so, normalize);
    return gated_forward_t<__nv_bfloat16>(s, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                          (const __nv_bfloat16 *)v, gamma,
                                          (__nv_bfloat16 *)out, st, stream, so, normalize);
}

}  // namespace kata
