// KATA-Sigma_2 at d = 64 on the d = 32 tensor path: the finalize pass.
//
// The map (Sec. 4.1, "two reduced PSD families") cuts u in R^64 into halves
// u_1, u_2 of width m = 32 and lifts psi(u) = eps I + s (u_1 u_1^T + u_2 u_2^T).
// Its weight expands, with |u|^2 = |u_1|^2 + |u_2|^2, into
//
//   <psi(q), psi(k)>_F = s^2 sum_{a,b} (q_a . k_b)^2 + eps s (|q|^2 + |k|^2) + eps^2 m.
//
// The four (a, b) terms are full-map attentions of 32-wide sub-heads (query
// half a against key half b); the tensor path runs them as four sub-heads and
// leaves their numerators N_ab(t) and denominators D_ab(t) in fp32.  The rest
// is a linear attention with the features (eps^2 m + eps s |q|^2, eps s) of
// the query and (1, |k|^2) of the key:
//
//   N_eps(t) = c_t sum_{s<=t} v_s + eps s sum_{s<=t} |k_s|^2 v_s,
//   D_eps(t) = c_t (t + 1)       + eps s sum_{s<=t} |k_s|^2,     c_t = eps^2 m + eps s |q_t|^2,
//
// and o_t = (s^2 sum N_ab + N_eps) / (s^2 sum D_ab + D_eps), zero where the
// denominator is not positive.  The prefix sums run in 128-token chunks: one
// pass sums each chunk, the segment scan of the tensor path makes the sums
// exclusive across chunks, and the finalize pass walks each chunk in order.
#include <cuda_bf16.h>

#include "kata_internal.cuh"

namespace kata {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kChunk = 128;
constexpr int kDim = 64;                 // d = dv = 64
constexpr int kRec = 2 * kDim + 4;       // [sum v | sum |k|^2 v | sum |k|^2 | 3 unused]
constexpr int kThreads = 64;             // one thread per value column

// |x|^2 of one 64-wide bf16 row, summed in fp32 in a fixed order.
__device__ __forceinline__ float sq_norm(const bf16 *row) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kDim / 8; ++i) {
        const uint4 w = p[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(u[e] << 16), hi = __uint_as_float(u[e] & 0xFFFF0000u);
            acc = fmaf(lo, lo, acc);
            acc = fmaf(hi, hi, acc);
        }
    }
    return acc;
}

// Chunk sums of v, |k|^2 v and |k|^2: one CTA per (chunk, head).
__global__ void __launch_bounds__(kThreads)
sigma_chunk_sums_kernel(const bf16 *__restrict__ k, const bf16 *__restrict__ v,
                        float *__restrict__ rec, int T, int NC) {
    __shared__ float kk[kChunk];
    const int c = blockIdx.x, bh = blockIdx.y, col = threadIdx.x;
    const int t0 = c * kChunk, n = min(kChunk, T - t0);
    const size_t base = (size_t)bh * T + t0;
    for (int t = col; t < n; t += kThreads) kk[t] = sq_norm(k + (base + t) * kDim);
    __syncthreads();
    float sv = 0.f, skv = 0.f, sk = 0.f;
    for (int t = 0; t < n; ++t) {
        const float x = __bfloat162float(v[(base + t) * kDim + col]);
        sv += x;
        skv = fmaf(kk[t], x, skv);
        sk += kk[t];
    }
    float *r = rec + ((size_t)bh * NC + c) * kRec;
    r[col] = sv;
    r[kDim + col] = skv;
    if (col < 4) r[2 * kDim + col] = col == 0 ? sk : 0.f;
}

// Output: the sub-head partials plus the eps terms, walking each chunk from its
// exclusive prefix.  part: N [BH * 4][T][64], then D [BH * 4][T].
__global__ void __launch_bounds__(kThreads)
sigma_finalize_kernel(const float *__restrict__ part, const float *__restrict__ rec,
                      const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                      const bf16 *__restrict__ v, bf16 *__restrict__ out, int BH, int T, int NC,
                      float s2, float es, float e2m) {
    __shared__ float kk[kChunk], qq[kChunk];
    const int c = blockIdx.x, bh = blockIdx.y, col = threadIdx.x;
    const int t0 = c * kChunk, n = min(kChunk, T - t0);
    const size_t base = (size_t)bh * T + t0;
    for (int t = col; t < n; t += kThreads) {
        kk[t] = sq_norm(k + (base + t) * kDim);
        qq[t] = sq_norm(q + (base + t) * kDim);
    }
    __syncthreads();
    const float *r = rec + ((size_t)bh * NC + c) * kRec;
    float sv = r[col], skv = r[kDim + col], sk = r[2 * kDim];
    const float *pd = part + (size_t)BH * 4 * T * kDim;
    // 8 tokens at a time: every load of the group is issued before the running
    // sums use the first, so the walk is not paced by one load latency per token
    constexpr int kGroup = 8;
    for (int t8 = 0; t8 < n; t8 += kGroup) {
        float xs[kGroup], ns[kGroup], ds[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int t = min(t8 + u, n - 1);
            xs[u] = __bfloat162float(v[(base + t) * kDim + col]);
            ns[u] = 0.f;
            ds[u] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const size_t row = ((size_t)bh * 4 + j) * T + t0 + t;
                ns[u] += part[row * kDim + col];
                ds[u] += pd[row];
            }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int t = t8 + u;
            if (t >= n) break;
            sv += xs[u];
            skv = fmaf(kk[t], xs[u], skv);
            sk += kk[t];
            const float ct = fmaf(es, qq[t], e2m);
            const float num = fmaf(s2, ns[u], fmaf(ct, sv, es * skv));
            const float den = fmaf(s2, ds[u], fmaf(ct, (float)(t0 + t + 1), es * sk));
            out[(base + t) * kDim + col] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
        }
    }
}

}  // namespace

size_t sigma_workspace_bytes(const FwdShape &s) {
    const size_t nc = (size_t)(s.T + kChunk - 1) / kChunk;
    return sizeof(float) * (size_t)s.BH() * nc * kRec;
}

cudaError_t sigma_finalize_launch(const FwdShape &s, const float *part, float *ws, const void *q,
                                  const void *k, const void *v, void *out, const MapSpec &map,
                                  cudaStream_t stream) {
    if (s.d != kDim || s.dv != kDim || s.dtype != 1 || map.kind != 2 || map.g != 2)
        return cudaErrorInvalidValue;
    const int NC = (s.T + kChunk - 1) / kChunk;
    const dim3 grid(NC, s.BH());
    {
        TraceScope tr("tc_sigma_sums", stream);
        sigma_chunk_sums_kernel<<<grid, kThreads, 0, stream>>>((const bf16 *)k, (const bf16 *)v, ws,
                                                               s.T, NC);
    }
    cudaError_t e = scan_exclusive_launch(ws, s.BH(), NC, kRec, "tc_sigma_scan", stream);
    if (e != cudaSuccess) return e;
    const float eps = map.eps, sc = map.scale;
    const int m = s.d / map.g;
    {
        TraceScope tr("tc_sigma_finalize", stream);
        sigma_finalize_kernel<<<grid, kThreads, 0, stream>>>(
            part, ws, (const bf16 *)q, (const bf16 *)k, (const bf16 *)v, (bf16 *)out, s.BH(), s.T,
            NC, sc * sc, eps * sc, eps * eps * (float)m);
    }
    return cudaGetLastError();
}

}  // namespace kata
