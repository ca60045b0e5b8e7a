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
// gamma = 0 (a reset) and gamma = 1 are exact and nothing cancels.  Stages 1
// and 3 are the tiled kernels of the plain path (kata_simt.cu) with the gates
// switched on; stage 2 is here.
// Workspace: per-chunk states [B*H][N_C][n][dv+1] fp32 (scanned in place),
// then the chunk gate products [B*H][N_C].
#include "kata_simt_common.cuh"

namespace kata {
namespace {

constexpr int kMaxC = 128;

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

template <typename T>
cudaError_t gated_forward_t(const FwdShape &s, const T *q, const T *k, const T *v,
                            const float *gamma, T *out, float *st, cudaStream_t stream,
                            const StateOut &so, int normalize) {
    const int n = s.n(), NC = s.NC(), BH = s.BH();
    const int64_t E = (int64_t)n * (s.dv + 1);
    if (E % 4 != 0 || (so.state && !so.z)) return cudaErrorInvalidValue;
    float *cgate = st + (size_t)BH * NC * n * (s.dv + 1);
    cudaError_t e = simt::state_launch<T>(s, k, v, gamma, st, cgate, MapSpec{}, stream,
                                          "gated_chunk_state");
    if (e != cudaSuccess) return e;
    {
        TraceScope tr("gated_scan", stream);
        gated_scan_kernel<<<dim3((unsigned)((E / 4 + 255) / 256), BH), 256, 0, stream>>>(
            st, cgate, NC, E, so.state, so.z, s.dv + 1);
    }
    return simt::output_launch<T>(s, q, k, v, gamma, st, out, MapSpec{}, normalize, stream,
                                  "gated_output");
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
