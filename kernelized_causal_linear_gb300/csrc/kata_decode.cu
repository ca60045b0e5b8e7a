// Single-token recurrent decode step of KATA (Sec. 2, Eq. 2 additive
// recurrence; App. D.1 "Plain KATA"):
//
//   S += psi(k) v^T,  z += psi(k),  o = psi(q)^T S / psi(q)^T z
//
// in place, update then read.  The step streams the fp32 state once (read and
// write of S and z), so it is bound by HBM bandwidth: one block per (b, h),
// 256 threads, 16-byte vector accesses, and the psi(q)^T S reduction folded
// into the same sweep so S is touched exactly once.
//
// The GatedKATA step (the pages' multiplicative scalar state gate) is the same
// sweep with S = gamma S + psi(k) v^T, z = gamma z + psi(k) (gamma per head), read
// out with or without the denominator: a compile-time variant, so the plain step
// carries no gate multiply.  A reduced map (KATA-M_g, KATA-Sigma_g, the orthant
// map) changes only the lift: its packed features from kata_map.cuh, its state
// width n.
#include "kata_dispatch.cuh"
#include "kata_map.cuh"

namespace kata {
namespace {

constexpr int kThreads = 256;

template <typename T, int DV4, bool kGated>
__global__ void __launch_bounds__(kThreads)
decode_kernel(float *__restrict__ S, float *__restrict__ z, const T *__restrict__ q,
              const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ out, int d,
              int n, const float *__restrict__ gamma, int normalize, MapSpec mp) {
    extern __shared__ float sm[];
    float *pk = sm;                 // psi(k) [n]
    float *pq = pk + n;             // psi(q) [n]
    __shared__ float qs[64], ks[64];
    __shared__ __align__(16) float vs[4 * DV4];
    __shared__ __align__(16) float part[kThreads * 4];
    __shared__ float dpart[kThreads / 32];

    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    constexpr int dv = 4 * DV4;
    const float g = kGated ? gamma[bh] : 1.f;
    if (tid < d) {
        qs[tid] = to_f(q[(size_t)bh * d + tid]);
        ks[tid] = to_f(k[(size_t)bh * d + tid]);
    }
    if (tid < dv) vs[tid] = to_f(v[(size_t)bh * dv + tid]);
    __syncthreads();

    // lift both vectors, update z and accumulate the denominator psi(q).z
    float den = 0.f;
    float *zb = z + (size_t)bh * n;
    for (int f = tid; f < n; f += kThreads) {
        float a, b;
        if (mp.kind == 0) {   // the rank-one lift
            int i, j;
            vech_pair(f, d, i, j);
            const float cf = (i == j) ? 1.f : kSqrt2;
            a = ks[i] * ks[j] * cf;
            b = qs[i] * qs[j] * cf;
        } else {              // a reduced map's packed feature f
            const Feat ft = map_feature(f, d, mp);
            a = ft(ks, 1);
            b = ft(qs, 1);
        }
        pk[f] = a;
        pq[f] = b;
        const float zn = kGated ? fmaf(g, zb[f], a) : zb[f] + a;
        zb[f] = zn;
        den = fmaf(b, zn, den);
    }
    __syncthreads();

    // state sweep: thread owns column quad c4 for rows f = tid/DV4 + m*(256/DV4)
    const int c4 = tid % DV4;
    constexpr int kRowStep = kThreads / DV4;
    const float4 vv = reinterpret_cast<const float4 *>(vs)[c4];
    float4 *Sb = reinterpret_cast<float4 *>(S + (size_t)bh * n * dv);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int f = tid / DV4;
    for (; f + 3 * kRowStep < n; f += 4 * kRowStep) {
        float4 s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] = Sb[(size_t)(f + u * kRowStep) * DV4 + c4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float a = pk[f + u * kRowStep];
            const float b = pq[f + u * kRowStep];
            s[u].x = fmaf(a, vv.x, kGated ? g * s[u].x : s[u].x);
            s[u].y = fmaf(a, vv.y, kGated ? g * s[u].y : s[u].y);
            s[u].z = fmaf(a, vv.z, kGated ? g * s[u].z : s[u].z);
            s[u].w = fmaf(a, vv.w, kGated ? g * s[u].w : s[u].w);
            Sb[(size_t)(f + u * kRowStep) * DV4 + c4] = s[u];
            acc.x = fmaf(b, s[u].x, acc.x);
            acc.y = fmaf(b, s[u].y, acc.y);
            acc.z = fmaf(b, s[u].z, acc.z);
            acc.w = fmaf(b, s[u].w, acc.w);
        }
    }
    for (; f < n; f += kRowStep) {
        float4 s = Sb[(size_t)f * DV4 + c4];
        const float a = pk[f], b = pq[f];
        s.x = fmaf(a, vv.x, kGated ? g * s.x : s.x);
        s.y = fmaf(a, vv.y, kGated ? g * s.y : s.y);
        s.z = fmaf(a, vv.z, kGated ? g * s.z : s.z);
        s.w = fmaf(a, vv.w, kGated ? g * s.w : s.w);
        Sb[(size_t)f * DV4 + c4] = s;
        acc.x = fmaf(b, s.x, acc.x);
        acc.y = fmaf(b, s.y, acc.y);
        acc.z = fmaf(b, s.z, acc.z);
        acc.w = fmaf(b, s.w, acc.w);
    }

    // reductions: denominator over all threads, numerator over threads of a quad
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if ((tid & 31) == 0) dpart[tid >> 5] = den;
    reinterpret_cast<float4 *>(part)[tid] = acc;
    __syncthreads();
    if (tid < dv) {
        float dsum = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) dsum += dpart[w];
        const int cq = tid / 4, lane4 = tid % 4;
        float num = 0.f;
        for (int r = 0; r < kRowStep; ++r) num += part[(r * DV4 + cq) * 4 + lane4];
        out[(size_t)bh * dv + tid] =
            from_f<T>((!kGated || normalize) ? (dsum > 0.f ? num / dsum : 0.f) : num);
    }
}

template <typename T, int DV4>
void decode_go(float *S, float *z, const T *q, const T *k, const T *v, T *out, int BH, int d,
               int n, size_t sm, cudaStream_t stream, const float *gamma, int normalize,
               const MapSpec &mp) {
    if (gamma)
        decode_kernel<T, DV4, true><<<BH, kThreads, sm, stream>>>(S, z, q, k, v, out, d, n, gamma,
                                                                 normalize, mp);
    else
        decode_kernel<T, DV4, false><<<BH, kThreads, sm, stream>>>(S, z, q, k, v, out, d, n,
                                                                  nullptr, 1, mp);
}

template <typename T>
cudaError_t decode_t(float *S, float *z, const T *q, const T *k, const T *v, T *out, int BH,
                     int d, int dv, cudaStream_t stream, const float *gamma, int normalize,
                     const MapSpec &mp) {
    const int n = mp.n(d);
    const size_t sm = sizeof(float) * 2 * (size_t)n;
    TraceScope tr(gamma ? "decode_gated" : mp.kind ? "decode_map" : "decode", stream);
    switch (dv) {
        case 16: decode_go<T, 4>(S, z, q, k, v, out, BH, d, n, sm, stream, gamma, normalize, mp); break;
        case 32: decode_go<T, 8>(S, z, q, k, v, out, BH, d, n, sm, stream, gamma, normalize, mp); break;
        case 64: decode_go<T, 16>(S, z, q, k, v, out, BH, d, n, sm, stream, gamma, normalize, mp); break;
        case 128: decode_go<T, 32>(S, z, q, k, v, out, BH, d, n, sm, stream, gamma, normalize, mp); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t decode_any(float *S, float *z, const void *q, const void *k, const void *v, void *out,
                       int BH, int d, int dv, int dtype, cudaStream_t stream, const float *gamma,
                       int normalize, const MapSpec &mp) {
    if (dtype == 0)
        return decode_t<float>(S, z, (const float *)q, (const float *)k, (const float *)v,
                               (float *)out, BH, d, dv, stream, gamma, normalize, mp);
    return decode_t<__nv_bfloat16>(S, z, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                   (const __nv_bfloat16 *)v, (__nv_bfloat16 *)out, BH, d, dv,
                                   stream, gamma, normalize, mp);
}

}  // namespace

cudaError_t decode_launch(float *S, float *z, const void *q, const void *k, const void *v,
                          void *out, int BH, int d, int dv, int dtype, cudaStream_t stream,
                          const float *gamma, int normalize) {
    return decode_any(S, z, q, k, v, out, BH, d, dv, dtype, stream, gamma, normalize, MapSpec{});
}

cudaError_t decode_map_launch(float *S, float *z, const void *q, const void *k, const void *v,
                              void *out, int BH, int d, int dv, int dtype, const MapSpec &map,
                              cudaStream_t stream) {
    return decode_any(S, z, q, k, v, out, BH, d, dv, dtype, stream, nullptr, 1, map);
}

}  // namespace kata
