// Forward dispatch shared by the API entry points (kata_api.cu, kata_noalloc.cu)
// and the scratch-copy route of kata_adapt.cu: which kernel family a shape runs
// on, its workspace and its launch.  Not included by the kernels' own files.
#pragma once
#include "kata_internal.cuh"

namespace kata {

// ---- plain forward dispatch: kata_api.cu ------------------------------------
// The kernel family a plain (full-map) chunked forward runs on, its workspace
// size and its launch; shared by kata_fwd_chunked and kata_fwd_chunked_noalloc
// so that both take the same path for the same shape.
// Tc32Adapt / Tc64Adapt: a bf16 shape the tensor-core kernels do not take
// directly (d = 16, or dv != 64) run on them through scratch copies
// (kata_adapt.cu).
enum class FwdKernels { Simt, Tc32, Tc64, Tc32Adapt, Tc64Adapt };
FwdKernels select_fwd_kernels(const FwdShape &s, int cc_major, int cc_minor, int num_sms);
size_t fwd_workspace_bytes(const FwdShape &s, FwdKernels kn, int num_sms, bool with_state = false);
cudaError_t fwd_launch(const FwdShape &s, FwdKernels kn, const void *q, const void *k,
                       const void *v, void *out, void *workspace, int num_sms,
                       cudaStream_t stream, const StateOut &so = StateOut{});

// ---- other bf16 shapes on the tensor-core kernels: kata_adapt.cu -----------
// d = 16 and dv in {16, 32, 128} run on the kernels of d = 32 or 64, dv = 64
// with q, k padded to d = 32 and v cut into 64-column parts.  Each selector
// answers for those shapes only (Simt / None / false for the kernels' own).
// Plain chunked: Tc32Adapt or Tc64Adapt.
FwdKernels adapt_kernels(const FwdShape &s, int cc_major, int cc_minor, int num_sms);
size_t adapt_workspace_bytes(const FwdShape &s, FwdKernels core, int num_sms, bool with_state);
cudaError_t adapt_forward(const FwdShape &s, FwdKernels core, const void *q, const void *k,
                          const void *v, void *out, void *workspace, int num_sms,
                          cudaStream_t stream, const StateOut &so);
// GatedKATA chunked: the d = 32 gated segments or the d = 64 gated route.
enum class GatedCore { None, Tc32, Wide };
GatedCore adapt_gated_core(const FwdShape &s, int cc_major, int cc_minor, int num_sms,
                           bool with_state);
size_t adapt_gated_workspace_bytes(const FwdShape &s, GatedCore core, int num_sms,
                                   bool with_state);
cudaError_t adapt_gated_forward(const FwdShape &s, GatedCore core, const void *q, const void *k,
                                const void *v, const float *gamma, void *out, void *workspace,
                                int num_sms, cudaStream_t stream, const StateOut &so,
                                int normalize);
// Quadratic form (gamma non-null: gated).
bool adapt_quad_supported(const FwdShape &s, int cc_major, int cc_minor);
size_t adapt_quad_workspace_bytes(const FwdShape &s, bool gated);
cudaError_t adapt_quad_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                               void *out, void *workspace, cudaStream_t stream, const float *gamma,
                               int normalize);

// ---- decode step under a reduced map: kata_decode.cu -------------------------
// S [BH][n][dv], z [BH][n] with n = map.n(d), features in map_feature's order.
cudaError_t decode_map_launch(float *S, float *z, const void *q, const void *k, const void *v,
                              void *out, int BH, int d, int dv, int dtype, const MapSpec &map,
                              cudaStream_t stream);

// Copies for running a reduced map's dv = 64 route on 64-column parts of v
// (kata_api.cu): columns of bf16 rows as copy_cols of kata_adapt.cu (zero_rest:
// the rest of each destination row zero), and a part's state sp [BH][n][64],
// zp [BH][n] into columns col .. col + width of state [BH][n][dv] (z as well
// when write_z).
cudaError_t part_copy_cols(const void *src, int sstride, int scol, int width, void *dst, int dstride,
                           int dcol, int64_t rows, bool zero_rest, cudaStream_t stream);
cudaError_t part_copy_state(const float *sp, const float *zp, int n, float *state, float *z, int BH,
                            int dv, int col, int width, bool write_z, cudaStream_t stream);

}  // namespace kata
