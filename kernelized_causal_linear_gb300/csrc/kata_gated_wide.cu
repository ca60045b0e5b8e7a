// GatedKATA at d = 64 on the tensor cores (bf16, dv = 64).
//
// The gated recurrence (the pages' "multiplicative scalar state gate",
// S_t = gamma_t S_{t-1} + psi(k_t) v_t^T) weighs write s at token t by
// prod_{r=s+1}^{t} gamma_r.  At d = 64 its outputs come from the gated
// quadratic form (kata_quad.cu), which evaluates that definition tile by tile
// on the tensor cores; nothing is approximated.
//
// The state after the last token is
//   S_T = sum_s A_s psi(k_s) v_s^T,   z_T = sum_s A_s psi(k_s),
//   A_s = prod_{r=s+1}^{T-1} gamma_r,
// and psi is quadratic, so A_s psi(k_s) = psi(sqrt(A_s) k_s): the plain state of
// the d = 64 chunked tensor path (kata_tc64.cu) on the keys sqrt(A_s) k_s is the
// gated state.  The quadratic form's prep pass already leaves K'_s = sqrt(a_s) k_s
// (a_s the gates after s to the end of its 128-token tile) and each tile's gate
// product; suffix_scale_kernel multiplies K' by the square root of the product of
// the later tiles' gates.  The chunked pass's own output is not used.
#include "kata_internal.cuh"

#include <cuda_bf16.h>

namespace kata {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kTileT = 128;   // tokens per tile of the quadratic form's prep
constexpr int kDim = 64;

// K''_s = sqrt(prod of the gates of the tiles after s's tile) K'_s for the 128
// tokens of tile c of head bh.  Grid (tiles, heads), 128 threads.
__global__ void __launch_bounds__(128)
suffix_scale_kernel(const bf16 *__restrict__ kc, const float *__restrict__ gtile,
                    bf16 *__restrict__ kpp, int T, int NT) {
    __shared__ float wprod[4];
    const int c = blockIdx.x, bh = blockIdx.y;
    const float *gt = gtile + (size_t)bh * NT;
    float after = 1.f;
    for (int cc = c + 1 + threadIdx.x; cc < NT; cc += blockDim.x) after *= gt[cc];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) after *= __shfl_xor_sync(0xffffffffu, after, o);
    if ((threadIdx.x & 31) == 0) wprod[threadIdx.x >> 5] = after;
    __syncthreads();
    const float sc = sqrtf(wprod[0] * wprod[1] * wprod[2] * wprod[3]);
    const int rows = min(kTileT, T - c * kTileT);
    const size_t base = ((size_t)bh * T + (size_t)c * kTileT) * kDim;
    const uint4 *src = reinterpret_cast<const uint4 *>(kc + base);
    uint4 *dst = reinterpret_cast<uint4 *>(kpp + base);
    for (int e = threadIdx.x; e < rows * (kDim / 8); e += blockDim.x) {
        uint4 u = src[e];
        uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(w[k] << 16) * sc;
            const float hi = __uint_as_float(w[k] & 0xFFFF0000u) * sc;
            const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
            w[k] = *reinterpret_cast<const uint32_t *>(&p);
        }
        dst[e] = u;
    }
}

}  // namespace

bool gated_wide_supported(const FwdShape &s, int cc_major, int cc_minor, int num_sms,
                          bool with_state) {
    if (s.d != kDim || s.dv != kDim || s.dtype != 1 || s.T > kGatedWideMaxT) return false;
    if (!quad_supported(s, cc_major, cc_minor)) return false;
    return !with_state || tc64_supported(s, cc_major, cc_minor, num_sms);
}

size_t gated_wide_workspace_bytes(const FwdShape &s, bool with_state) {
    const size_t q = (quad_gated_workspace_bytes(s) + 255) & ~(size_t)255;
    if (!with_state) return q;
    const size_t rows = (size_t)s.BH() * s.T * kDim * sizeof(bf16);   // K'' and a scratch output
    return q + 2 * rows + tc64_workspace_bytes(s, true);
}

cudaError_t gated_wide_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                               const float *gamma, void *out, void *workspace, cudaStream_t stream,
                               const StateOut &so, int normalize) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // the quadratic form's workspace: K' [BH][T][d] bf16 | lam2 [BH][T] | tile gate products [BH][NT]
    cudaError_t e = quad_forward(s, q, k, v, out, stream, gamma, normalize, ws);
    if (e != cudaSuccess || so.state == nullptr) return e;
    const int NT = (s.T + kTileT - 1) / kTileT;
    const size_t nrow = (size_t)s.BH() * s.T * kDim;
    const bf16 *kc = reinterpret_cast<const bf16 *>(ws);
    const float *gtile = reinterpret_cast<const float *>(kc + nrow) + (size_t)s.BH() * s.T;
    uint8_t *rest = ws + ((quad_gated_workspace_bytes(s) + 255) & ~(size_t)255);
    bf16 *kpp = reinterpret_cast<bf16 *>(rest);
    bf16 *oscratch = kpp + nrow;
    {
        TraceScope tr("tc_gated_suffix_scale", stream);
        suffix_scale_kernel<<<dim3(NT, s.BH()), 128, 0, stream>>>(kc, gtile, kpp, s.T, NT);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return tc64_forward(s, q, kpp, v, oscratch, oscratch + nrow, stream, so);
}

}  // namespace kata
