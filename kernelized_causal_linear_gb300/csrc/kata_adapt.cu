// bf16 shapes the tensor-core kernels do not take directly (d = 16, or dv in
// {16, 32, 128}), run on them through scratch copies.
//
// The kernels are written for d in {32, 64} and dv = 64.  Every forward they
// compute (the chunked form, Sec. 4.1 Eq. 17-20; the quadratic form, Eq. 2; and
// both with the scalar state gate) is exact under two rewritings:
//   - q and k padded with zero columns to d = 32: psi of the padded row holds
//     psi of the row plus zeros, so every weight (q . k)^2 is unchanged, and the
//     state's features for index pairs (i, j) with i, j < 16 are the state of
//     the unpadded rows (the others are zero);
//   - v cut into 64-column parts (the last one zero-padded): an output column
//     depends on its own v column and on weights that every part shares, so
//     the parts are independent forwards whose outputs are the columns of the
//     result, and whose states are the state's column blocks (z, which holds no
//     v, is the same in each).  Gates act on the weights only.
// A part's output and state go to scratch; their real columns and features are
// copied to the caller's buffers.  With dv = 64 (d = 16) the one part is v
// itself and its output is out.
#include "kata_dispatch.cuh"

#include <cuda_bf16.h>

namespace kata {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kPartDv = 64;

// Rows of bf16: dst[r][dcol .. dcol + width) = src[r][scol .. scol + width), and,
// with zero_rest, the rest of each dst row zero.  One thread per 16-byte piece
// (strides, column offsets and widths are multiples of 8 elements).
__global__ void __launch_bounds__(256)
copy_cols_kernel(const bf16 *__restrict__ src, int sstride, int scol, int width,
                 bf16 *__restrict__ dst, int dstride, int dcol, int64_t rows, int zero_rest) {
    const int per = (zero_rest ? dstride : width) / 8;   // pieces written per row
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * per) return;
    const int64_t r = e / per;
    const int p = (int)(e % per);
    const int c = zero_rest ? 8 * p : dcol + 8 * p;   // dst column of the piece
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (c >= dcol && c < dcol + width)
        u = *reinterpret_cast<const uint4 *>(src + (size_t)r * sstride + scol + (c - dcol));
    *reinterpret_cast<uint4 *>(dst + (size_t)r * dstride + c) = u;
}

cudaError_t copy_cols(const void *src, int sstride, int scol, int width, void *dst, int dstride,
                      int dcol, int64_t rows, bool zero_rest, cudaStream_t stream) {
    const int64_t n = rows * ((zero_rest ? dstride : width) / 8);
    if (n == 0) return cudaSuccess;
    copy_cols_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        (const bf16 *)src, sstride, scol, width, (bf16 *)dst, dstride, dcol, rows, zero_rest ? 1 : 0);
    return cudaGetLastError();
}

// State of one v part in the core's layout (sp [BH][np][64], zp [BH][np], np
// the packed features of dimension dc) to the caller's (state [BH][n][dv],
// z [BH][n], n those of d <= dc): feature f = (i, j) of dimension d sits at
// i*dc - i*(i-1)/2 + (j - i) in the core's order.  Grid (n, BH), 64 threads.
__global__ void __launch_bounds__(64)
state_gather_kernel(const float *__restrict__ sp, const float *__restrict__ zp, int np, int dc,
                    int d, float *__restrict__ state, float *__restrict__ z, int n, int dv, int col,
                    int width, int write_z) {
    const int f = blockIdx.x, bh = blockIdx.y;
    int i, j;
    vech_pair(f, d, i, j);
    const int fp = i * dc - i * (i - 1) / 2 + (j - i);
    const float *src = sp + ((size_t)bh * np + fp) * kPartDv;
    float *dst = state + ((size_t)bh * n + f) * dv + col;
    for (int c = threadIdx.x; c < width; c += blockDim.x) dst[c] = src[c];
    if (write_z && threadIdx.x == 0) z[(size_t)bh * n + f] = zp[(size_t)bh * np + fp];
}

// The shapes taken through the rewritings: bf16, d in {16, 32, 64}, dv in
// {16, 32, 64, 128}, other than the kernels' own (d in {32, 64}, dv = 64).
bool adapted_shape(const FwdShape &s) {
    if (s.dtype != 1 || (s.d != 16 && s.d != 32 && s.d != 64)) return false;
    if (s.dv != 16 && s.dv != 32 && s.dv != 64 && s.dv != 128) return false;
    return s.d == 16 || s.dv != kPartDv;
}

FwdShape core_shape(const FwdShape &s) {
    FwdShape c = s;
    c.d = s.d == 16 ? 32 : s.d;
    c.dv = kPartDv;
    return c;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

// Scratch of the rewritings: [padded q, k when d = 16] [one v part] [its
// output] [its state and z when exported], each from a 256-byte boundary; the
// core's workspace follows.
struct AdaptLayout {
    size_t qk, v, o, st, total;
};

AdaptLayout layout(const FwdShape &s, bool with_state) {
    const FwdShape c = core_shape(s);
    const size_t rows = (size_t)s.BH() * s.T;
    AdaptLayout L;
    L.qk = s.d == 16 ? 2 * round256(rows * c.d * sizeof(bf16)) : 0;
    L.v = s.dv == kPartDv ? 0 : round256(rows * kPartDv * sizeof(bf16));
    L.o = L.v;
    L.st = with_state ? round256((size_t)s.BH() * c.n() * kPartDv * sizeof(float)) +
                            round256((size_t)s.BH() * c.n() * sizeof(float))
                      : 0;
    L.total = L.qk + L.v + L.o + L.st;
    return L;
}

// Runs run(qc, kc, vc, oc, state_out, core_workspace) once per 64-column part
// of v on the core shape, around the copies described at the top.
template <class Run>
cudaError_t run_parts(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                      void *workspace, cudaStream_t stream, const StateOut &so, Run run) {
    if ((size_t)s.BH() * s.T == 0) return cudaSuccess;
    const FwdShape c = core_shape(s);
    const bool with_state = so.state != nullptr;
    const AdaptLayout L = layout(s, with_state);
    const int64_t rows = (int64_t)s.BH() * s.T;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *qp = ws, *kp = ws + L.qk / 2;
    uint8_t *vp = ws + L.qk, *op = vp + L.v;
    float *sp = reinterpret_cast<float *>(op + L.o);
    float *zp = sp + round256((size_t)s.BH() * c.n() * kPartDv * sizeof(float)) / sizeof(float);
    void *cw = ws + L.total;
    cudaError_t e = cudaSuccess;
    const void *qc = q, *kc = k;
    if (s.d == 16) {
        {
            TraceScope tr("tc_adapt_pad", stream);
            if ((e = copy_cols(q, s.d, 0, s.d, qp, c.d, 0, rows, true, stream)) != cudaSuccess)
                return e;
        }
        {
            TraceScope tr("tc_adapt_pad", stream);
            if ((e = copy_cols(k, s.d, 0, s.d, kp, c.d, 0, rows, true, stream)) != cudaSuccess)
                return e;
        }
        qc = qp;
        kc = kp;
    }
    StateOut cso;
    if (with_state) {
        cso.state = sp;
        cso.z = zp;
    }
    const bool whole = s.dv == kPartDv;   // v and out serve as the one part directly
    for (int col = 0; col < s.dv; col += kPartDv) {
        const int w = s.dv - col < kPartDv ? s.dv - col : kPartDv;
        if (!whole) {
            TraceScope tr("tc_adapt_v_part", stream);
            if ((e = copy_cols(v, s.dv, col, w, vp, kPartDv, 0, rows, true, stream)) != cudaSuccess)
                return e;
        }
        if ((e = run(qc, kc, whole ? v : (const void *)vp, whole ? out : (void *)op, cso, cw)) !=
            cudaSuccess)
            return e;
        if (!whole) {
            TraceScope tr("tc_adapt_out_part", stream);
            if ((e = copy_cols(op, kPartDv, 0, w, out, s.dv, col, rows, false, stream)) != cudaSuccess)
                return e;
        }
        if (with_state) {
            TraceScope tr("tc_adapt_state_part", stream);
            state_gather_kernel<<<dim3(s.n(), s.BH()), 64, 0, stream>>>(
                sp, zp, c.n(), c.d, s.d, so.state, so.z, s.n(), s.dv, col, w, col == 0 ? 1 : 0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace

// ---- copies for the parts of the reduced maps (kata_api.cu) ------------------
__global__ void __launch_bounds__(64)
state_cols_kernel(const float *__restrict__ sp, const float *__restrict__ zp, int n,
                  float *__restrict__ state, float *__restrict__ z, int dv, int col, int width,
                  int write_z) {
    const int f = blockIdx.x, bh = blockIdx.y;
    const float *src = sp + ((size_t)bh * n + f) * kPartDv;
    float *dst = state + ((size_t)bh * n + f) * dv + col;
    for (int c = threadIdx.x; c < width; c += blockDim.x) dst[c] = src[c];
    if (write_z && threadIdx.x == 0) z[(size_t)bh * n + f] = zp[(size_t)bh * n + f];
}

cudaError_t part_copy_cols(const void *src, int sstride, int scol, int width, void *dst, int dstride,
                           int dcol, int64_t rows, bool zero_rest, cudaStream_t stream) {
    return copy_cols(src, sstride, scol, width, dst, dstride, dcol, rows, zero_rest, stream);
}

cudaError_t part_copy_state(const float *sp, const float *zp, int n, float *state, float *z, int BH,
                            int dv, int col, int width, bool write_z, cudaStream_t stream) {
    if (n == 0 || BH == 0) return cudaSuccess;
    state_cols_kernel<<<dim3(n, BH), 64, 0, stream>>>(sp, zp, n, state, z, dv, col, width,
                                                      write_z ? 1 : 0);
    return cudaGetLastError();
}

// ---- plain chunked forward ---------------------------------------------------
FwdKernels adapt_kernels(const FwdShape &s, int cc_major, int cc_minor, int num_sms) {
    if (!adapted_shape(s)) return FwdKernels::Simt;
    const FwdShape c = core_shape(s);
    if (tc_supported(c, cc_major, cc_minor)) return FwdKernels::Tc32Adapt;
    if (tc64_supported(c, cc_major, cc_minor, num_sms)) return FwdKernels::Tc64Adapt;
    return FwdKernels::Simt;
}

size_t adapt_workspace_bytes(const FwdShape &s, FwdKernels core, int num_sms, bool with_state) {
    const FwdShape c = core_shape(s);
    return layout(s, with_state).total +
           (core == FwdKernels::Tc32Adapt ? tc_workspace_bytes(c, num_sms, with_state)
                                          : tc64_workspace_bytes(c, with_state));
}

cudaError_t adapt_forward(const FwdShape &s, FwdKernels core, const void *q, const void *k,
                          const void *v, void *out, void *workspace, int num_sms,
                          cudaStream_t stream, const StateOut &so) {
    const FwdShape c = core_shape(s);
    return run_parts(s, q, k, v, out, workspace, stream, so,
                     [&](const void *qc, const void *kc, const void *vc, void *oc,
                         const StateOut &cso, void *cw) {
                         return core == FwdKernels::Tc32Adapt
                                    ? tc_forward(c, qc, kc, vc, oc, cw, num_sms, stream, cso)
                                    : tc64_forward(c, qc, kc, vc, oc, cw, stream, cso);
                     });
}

// ---- GatedKATA chunked forward -------------------------------------------------
GatedCore adapt_gated_core(const FwdShape &s, int cc_major, int cc_minor, int num_sms,
                           bool with_state) {
    if (!adapted_shape(s)) return GatedCore::None;
    const FwdShape c = core_shape(s);
    if (tc_supported(c, cc_major, cc_minor)) return GatedCore::Tc32;
    if (gated_wide_supported(c, cc_major, cc_minor, num_sms, with_state)) return GatedCore::Wide;
    return GatedCore::None;
}

size_t adapt_gated_workspace_bytes(const FwdShape &s, GatedCore core, int num_sms,
                                   bool with_state) {
    const FwdShape c = core_shape(s);
    return layout(s, with_state).total +
           (core == GatedCore::Tc32 ? tc_gated_workspace_bytes(c, num_sms, with_state)
                                    : gated_wide_workspace_bytes(c, with_state));
}

cudaError_t adapt_gated_forward(const FwdShape &s, GatedCore core, const void *q, const void *k,
                                const void *v, const float *gamma, void *out, void *workspace,
                                int num_sms, cudaStream_t stream, const StateOut &so,
                                int normalize) {
    const FwdShape c = core_shape(s);
    return run_parts(s, q, k, v, out, workspace, stream, so,
                     [&](const void *qc, const void *kc, const void *vc, void *oc,
                         const StateOut &cso, void *cw) {
                         return core == GatedCore::Tc32
                                    ? tc_forward_gated(c, qc, kc, vc, gamma, oc, cw, num_sms,
                                                       stream, cso, normalize)
                                    : gated_wide_forward(c, qc, kc, vc, gamma, oc, cw, stream, cso,
                                                         normalize);
                     });
}

// ---- quadratic form, plain or gated -------------------------------------------
bool adapt_quad_supported(const FwdShape &s, int cc_major, int cc_minor) {
    return adapted_shape(s) && quad_supported(core_shape(s), cc_major, cc_minor);
}

size_t adapt_quad_workspace_bytes(const FwdShape &s, bool gated) {
    return layout(s, false).total + (gated ? quad_gated_workspace_bytes(core_shape(s)) : 0);
}

cudaError_t adapt_quad_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                               void *out, void *workspace, cudaStream_t stream, const float *gamma,
                               int normalize) {
    const FwdShape c = core_shape(s);
    return run_parts(s, q, k, v, out, workspace, stream, StateOut{},
                     [&](const void *qc, const void *kc, const void *vc, void *oc, const StateOut &,
                         void *cw) {
                         return quad_forward(c, qc, kc, vc, oc, stream, gamma, normalize,
                                             gamma ? cw : nullptr);
                     });
}

}  // namespace kata
