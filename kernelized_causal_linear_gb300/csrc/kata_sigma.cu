// KATA-Sigma_g on the tensor paths: the eps terms and the finalize pass.
//
// The map (Sec. 4.1, "two reduced PSD families") cuts u into g blocks u_a of
// width m = d / g and lifts psi(u) = eps I + s sum_a u_a u_a^T.  Its weight
// expands, with |u|^2 = sum_a |u_a|^2, into
//
//   <psi(q), psi(k)>_F = s^2 sum_{a,b} (q_a . k_b)^2 + eps s (|q|^2 + |k|^2) + eps^2 m.
//
// The (a, b) terms are full-map attentions; the tensor paths leave their
// numerators N(t) and denominators D(t) in fp32 partials:
//   Sigma_2 at d = 64: four crosswise d = 32 sub-heads (query half a, key half b);
//   Sigma_1 at d = 32: the d = 32 full map, one sub-head;
//   Sigma_1 at d = 64: the d = 64 full map, whose four feature groups each leave
//   a partial numerator, with one denominator.
// The rest is a linear attention with the features (eps^2 m + eps s |q|^2,
// eps s) of the query and (1, |k|^2) of the key:
//
//   N_eps(t) = c_t sum_{s<=t} v_s + eps s sum_{s<=t} |k_s|^2 v_s,
//   D_eps(t) = c_t (t + 1)       + eps s sum_{s<=t} |k_s|^2,     c_t = eps^2 m + eps s |q_t|^2,
//
// and o_t = (s^2 sum N + N_eps) / (s^2 sum D + D_eps), zero where the
// denominator is not positive.  The prefix sums run in 128-token chunks: one
// pass sums each chunk, the chunk scan makes the sums exclusive across chunks,
// and the finalize pass walks each chunk in order.
#include <cuda_bf16.h>

#include "kata_internal.cuh"

namespace kata {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kChunk = 128;
constexpr int kDv = 64;                  // value columns
constexpr int kRec = 2 * kDv + 4;        // [sum v | sum |k|^2 v | sum |k|^2 | 3 unused]
static_assert(kRec == kSigmaRec, "the record layout StateOut::eps_totals documents");
constexpr int kThreads = 64;             // one thread per value column

// |x|^2 of one D-wide bf16 row, summed in fp32 in a fixed order.
template <int D>
__device__ __forceinline__ float sq_norm(const bf16 *row) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
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
template <int D>
__global__ void __launch_bounds__(kThreads)
sigma_chunk_sums_kernel(const bf16 *__restrict__ k, const bf16 *__restrict__ v,
                        float *__restrict__ rec, int T, int NC) {
    __shared__ float kk[kChunk];
    const int c = blockIdx.x, bh = blockIdx.y, col = threadIdx.x;
    const int t0 = c * kChunk, n = min(kChunk, T - t0);
    const size_t base = (size_t)bh * T + t0;
    for (int t = col; t < n; t += kThreads) kk[t] = sq_norm<D>(k + (base + t) * D);
    __syncthreads();
    float sv = 0.f, skv = 0.f, sk = 0.f;
    for (int t = 0; t < n; ++t) {
        const float x = __bfloat162float(v[(base + t) * kDv + col]);
        sv += x;
        skv = fmaf(kk[t], x, skv);
        sk += kk[t];
    }
    float *r = rec + ((size_t)bh * NC + c) * kRec;
    r[col] = sv;
    r[kDv + col] = skv;
    if (col < 4) r[2 * kDv + col] = col == 0 ? sk : 0.f;
}

// Output: the partials plus the eps terms, walking each chunk from its
// exclusive prefix.  Partial j of head bh at token t is row
// bh * head_rows + j * part_rows + t of N (64 floats a row) and of D, summed
// over NN numerator and ND denominator partials in the order j = 0, 1, ...
struct PartLayout {
    const float *n, *d;
    int64_t n_head, n_part, d_head, d_part;
};
template <int D, int NN, int ND>
__global__ void __launch_bounds__(kThreads)
sigma_finalize_kernel(PartLayout pl, const float *__restrict__ rec, const bf16 *__restrict__ q,
                      const bf16 *__restrict__ k, const bf16 *__restrict__ v,
                      bf16 *__restrict__ out, int T, int NC, float s2, float es, float e2m) {
    __shared__ float kk[kChunk], qq[kChunk];
    const int c = blockIdx.x, bh = blockIdx.y, col = threadIdx.x;
    const int t0 = c * kChunk, n = min(kChunk, T - t0);
    const size_t base = (size_t)bh * T + t0;
    for (int t = col; t < n; t += kThreads) {
        kk[t] = sq_norm<D>(k + (base + t) * D);
        qq[t] = sq_norm<D>(q + (base + t) * D);
    }
    __syncthreads();
    const float *r = rec + ((size_t)bh * NC + c) * kRec;
    float sv = r[col], skv = r[kDv + col], sk = r[2 * kDv];
    const size_t nrow = (size_t)bh * pl.n_head + t0, drow = (size_t)bh * pl.d_head + t0;
    // 8 tokens at a time: every load of the group is issued before the running
    // sums use the first, so the walk is not paced by one load latency per token
    constexpr int kGroup = 8;
    for (int t8 = 0; t8 < n; t8 += kGroup) {
        float xs[kGroup], ns[kGroup], ds[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int t = min(t8 + u, n - 1);
            xs[u] = __bfloat162float(v[(base + t) * kDv + col]);
            ns[u] = 0.f;
            ds[u] = 0.f;
#pragma unroll
            for (int j = 0; j < NN; ++j) ns[u] += pl.n[(nrow + (size_t)j * pl.n_part + t) * kDv + col];
#pragma unroll
            for (int j = 0; j < ND; ++j) ds[u] += pl.d[drow + (size_t)j * pl.d_part + t];
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
            out[(base + t) * kDv + col] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
        }
    }
}

template <int D, int NN, int ND>
void launch_finalize(dim3 grid, cudaStream_t stream, const PartLayout &pl, const float *rec,
                     const void *q, const void *k, const void *v, void *out, int T, int NC,
                     float s2, float es, float e2m) {
    sigma_finalize_kernel<D, NN, ND><<<grid, kThreads, 0, stream>>>(
        pl, rec, (const bf16 *)q, (const bf16 *)k, (const bf16 *)v, (bf16 *)out, T, NC, s2, es, e2m);
}

}  // namespace

size_t sigma_workspace_bytes(const FwdShape &s) {
    const size_t nc = (size_t)(s.T + kChunk - 1) / kChunk;
    return sizeof(float) * (size_t)s.BH() * nc * kRec;
}

cudaError_t sigma_finalize_launch(const FwdShape &s, SigmaParts parts, const float *part,
                                  float *ws, const void *q, const void *k, const void *v, void *out,
                                  const MapSpec &map, cudaStream_t stream, float *eps_totals) {
    if (s.dv != kDv || s.dtype != 1 || map.kind != 2) return cudaErrorInvalidValue;
    const bool sub4 = parts == SigmaParts::Sub4 && s.d == 64 && map.g == 2;
    const bool sub1 = parts == SigmaParts::Sub1 && s.d == 32 && map.g == 1;
    const bool wide = parts == SigmaParts::Wide && s.d == 64 && map.g == 1;
    if (!sub4 && !sub1 && !wide) return cudaErrorInvalidValue;
    const int NC = (s.T + kChunk - 1) / kChunk;
    const dim3 grid(NC, s.BH());
    {
        TraceScope tr("tc_sigma_sums", stream);
        if (s.d == 64)
            sigma_chunk_sums_kernel<64><<<grid, kThreads, 0, stream>>>((const bf16 *)k, (const bf16 *)v,
                                                                       ws, s.T, NC);
        else
            sigma_chunk_sums_kernel<32><<<grid, kThreads, 0, stream>>>((const bf16 *)k, (const bf16 *)v,
                                                                       ws, s.T, NC);
    }
    cudaError_t e = scan_exclusive_launch(ws, s.BH(), NC, kRec, "tc_sigma_scan", stream, StateOut{}, 0,
                                          eps_totals);
    if (e != cudaSuccess) return e;
    const float eps = map.eps, sc = map.scale;
    const float s2 = sc * sc, es = eps * sc, e2m = eps * eps * (float)(s.d / map.g);
    const int64_t T = s.T, rows = (int64_t)s.BH() * T;
    TraceScope tr("tc_sigma_finalize", stream);
    if (sub4) {   // N [BH * 4][T][64], then D [BH * 4][T]
        const PartLayout pl{part, part + rows * 4 * kDv, 4 * T, T, 4 * T, T};
        launch_finalize<64, 4, 4>(grid, stream, pl, ws, q, k, v, out, s.T, NC, s2, es, e2m);
    } else if (sub1) {   // N [BH][T][64], then D [BH][T]
        const PartLayout pl{part, part + rows * kDv, T, 0, T, 0};
        launch_finalize<32, 1, 1>(grid, stream, pl, ws, q, k, v, out, s.T, NC, s2, es, e2m);
    } else {   // N [4][BH][T][64], then D [BH][T]
        const PartLayout pl{part, part + rows * 4 * kDv, T, rows, T, 0};
        launch_finalize<64, 4, 1>(grid, stream, pl, ws, q, k, v, out, s.T, NC, s2, es, e2m);
    }
    return cudaGetLastError();
}

}  // namespace kata
