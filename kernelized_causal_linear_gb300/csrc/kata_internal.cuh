// Internal declarations shared by the translation units of libkata.
// Not part of the public ABI (include/kata.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kata {

// Shape of one forward call, validated by the API layer.
struct FwdShape {
    int B, H, T, d, dv, C, dtype;
    int BH() const { return B * H; }
    int n() const { return d * (d + 1) / 2; }
    int NC() const { return (T + C - 1) / C; }
};

// Element conversion for the two input types.
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Packed position f -> (i, j), i <= j, of the upper-triangle row-major order
// f(i,j) = i*d - i*(i-1)/2 + (j - i) used by the rank-one PSD lift.
__device__ __forceinline__ void vech_pair(int f, int d, int &i, int &j) {
    int row = 0, start = 0;
    while (start + (d - row) <= f) {
        start += d - row;
        ++row;
    }
    i = row;
    j = row + (f - start);
}

constexpr float kSqrt2 = 1.41421356237309515f;

// ---- tracing: kata_trace.cu ------------------------------------------------
// Brackets one kernel launch with CUDA events on `stream` while tracing is on.
class TraceScope {
  public:
    TraceScope(const char *stage, cudaStream_t stream);
    ~TraceScope();
    TraceScope(const TraceScope &) = delete;
    TraceScope &operator=(const TraceScope &) = delete;

  private:
    const char *stage_;
    cudaStream_t stream_;
    cudaEvent_t start_ = nullptr;
};

// Feature map of the forward ([KATA] Sec. 4.1, the full rank-one map and the two
// reduced PSD families): the vector is cut into g blocks of width m = d / g.
//   kind 0: psi(u) = u u^T (g = 1);
//   kind 1 (M_g): psi(u) = (u_1 u_1^T, ..., u_g u_g^T), g m(m+1)/2 features;
//   kind 2 (Sigma_g): psi(u) = eps I + scale * sum_a u_a u_a^T, m(m+1)/2 features.
// Packing per matrix: upper triangle row-major, sqrt(2) off the diagonal.
struct MapSpec {
    int kind = 0, g = 1;
    float eps = 0.f, scale = 1.f;
    __host__ __device__ int m(int d) const { return d / g; }
    __host__ __device__ int n(int d) const {
        const int w = d / g;
        return kind == 1 ? g * w * (w + 1) / 2 : kind == 2 ? w * (w + 1) / 2 : kind == 3 ? d
                                                                                 : d * (d + 1) / 2;
    }
};

// Optional export of the state after the last token, in the decode layout:
// state [BH][n][dv] and z [BH][n] fp32, row-major vech order with sqrt(2) on the
// off-diagonal entries.  Both null: no export.
struct StateOut {
    float *state = nullptr;
    float *z = nullptr;
    // A Sigma map's eps terms (tensor routes): the inclusive totals of their chunk
    // sums per head, [BH][kSigmaRec] = [sum v (64) | sum |k|^2 v (64) | sum |k|^2 | 3 unused].
    float *eps_totals = nullptr;
};
constexpr int kSigmaRec = 2 * 64 + 4;

// ---- CUDA-core (SIMT) path: kata_simt.cu ----------------------------------
size_t simt_workspace_bytes(const FwdShape &s, const MapSpec &map = MapSpec{});
cudaError_t simt_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                         void *out, void *workspace, cudaStream_t stream,
                         const StateOut &so = StateOut{}, const MapSpec &map = MapSpec{});
cudaError_t lift_launch(const void *x, float *phi, int64_t rows, int d, int dtype,
                        cudaStream_t stream, const MapSpec &map = MapSpec{});
// Exclusive prefix in place along axis 1 of data[BH][n][E] (fp32).  With
// so.state set, E = nf * W holds nf rows of W = dv + 1 values and the inclusive
// totals go to so.state[BH][nf][dv] (columns 0..dv-1) and so.z[BH][nf] (column dv).
// With totals set, the inclusive totals go to totals[BH][E] as they are.
// part_ws (BH * (n / 16 + 1) * E floats) allows the two-level form of the scan.
cudaError_t scan_exclusive_launch(float *data, int BH, int n, int64_t E, const char *stage,
                                  cudaStream_t stream, const StateOut &so = StateOut{},
                                  int W = 0, float *totals = nullptr, float *part_ws = nullptr);

// ---- decode: kata_decode.cu -----------------------------------------------
cudaError_t decode_launch(float *S, float *z, const void *q, const void *k, const void *v,
                          void *out, int BH, int d, int dv, int dtype, cudaStream_t stream,
                          const float *gamma = nullptr, int normalize = 1);

// ---- GatedKATA chunked forward on CUDA cores: kata_gated.cu ----------------
size_t gated_workspace_bytes(const FwdShape &s);
cudaError_t gated_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                          const float *gamma, void *out, void *workspace, cudaStream_t stream,
                          const StateOut &so, int normalize);

// ---- tcgen05 path: kata_tc.cu ---------------------------------------------
bool tc_supported(const FwdShape &s, int cc_major, int cc_minor);
// nsub > 1: the head's q/k columns are nsub sub-heads of width d / nsub, each run
// as a d / nsub head (KATA-M_2 at d = 64); their numerators and denominators are
// summed.  sigma: KATA-Sigma_2 at d = 64 (nsub = 4, the four sub-heads pair
// query half a with key half b) or KATA-Sigma_1 at d = 32 (nsub = 1, the full
// map); the map's eps terms are added in the finalize pass (kata_sigma.cu).
// With sub-heads or eps terms, so receives the full-map (d = 32) state of every
// key sub-head: [BH * nsub] of them (two per head when crosswise) in the decode
// layout, and so.eps_totals the eps sums; map_state_compose forms the map's.
size_t tc_workspace_bytes(const FwdShape &s, int num_sms, bool with_state = false, int nsub = 1,
                          const MapSpec *sigma = nullptr);
cudaError_t tc_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                       void *out, void *workspace, int num_sms, cudaStream_t stream,
                       const StateOut &so = StateOut{}, int nsub = 1,
                       const MapSpec *sigma = nullptr);
// GatedKATA on the d = 32 tensor path (bf16, dv = 64): the same segments, with
// the gates folded into the keys, a gated segment scan and the running state
// decayed by each chunk's gate product.  normalize 0 drops the denominator.
size_t tc_gated_workspace_bytes(const FwdShape &s, int num_sms, bool with_state);
cudaError_t tc_forward_gated(const FwdShape &s, const void *q, const void *k, const void *v,
                             const float *gamma, void *out, void *workspace, int num_sms,
                             cudaStream_t stream, const StateOut &so, int normalize);
// GatedKATA at d = 64 on the tensor cores (kata_gated_wide.cu): the output from
// the gated quadratic form, the state after the last token (when asked) from
// the plain d = 64 chunked tensor path on the keys scaled by the square root of
// the gates after them.  Up to kGatedWideMaxT tokens (the quadratic form's cost
// per token grows with T; ~13 ns per token and head at that bound).
constexpr int kGatedWideMaxT = 262144;
bool gated_wide_supported(const FwdShape &s, int cc_major, int cc_minor, int num_sms,
                          bool with_state);
size_t gated_wide_workspace_bytes(const FwdShape &s, bool with_state);
cudaError_t gated_wide_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                               const float *gamma, void *out, void *workspace, cudaStream_t stream,
                               const StateOut &so, int normalize);
// KATA-M_4 at d = 64: q and k rows padded to four 32-wide blocks [u_a | 0], run
// as four d = 32 sub-heads (nsub = 4) whose numerators and denominators add.
// so: the four padded sub-heads' d = 32 states, as tc_forward with nsub = 4.
size_t tc_m4_workspace_bytes(const FwdShape &s, int num_sms, bool with_state = false);
cudaError_t tc_forward_m4(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                          void *workspace, int num_sms, cudaStream_t stream,
                          const StateOut &so = StateOut{});
// KATA-Sigma_g finalize (kata_sigma.cu): the scratch it needs after the
// partials, and the pass that sums them with the eps terms.  The partials'
// layouts: Sub4, the four crosswise d = 32 sub-heads of Sigma_2 at d = 64
// (N [BH * 4][T][64], then D [BH * 4][T]); Sub1, Sigma_1 at d = 32 as one
// d = 32 sub-head (N [BH][T][64], then D [BH][T]); Wide, Sigma_1 at d = 64 on the
// d = 64 path (N [4][BH][T][64] of its feature groups, then D [BH][T]).
enum class SigmaParts { Sub4, Sub1, Wide };
size_t sigma_workspace_bytes(const FwdShape &s);
// eps_totals: if set, receives the inclusive totals of the eps chunk sums.
cudaError_t sigma_finalize_launch(const FwdShape &s, SigmaParts parts, const float *part,
                                  float *ws, const void *q, const void *k, const void *v, void *out,
                                  const MapSpec &map, cudaStream_t stream,
                                  float *eps_totals = nullptr);
// The state of a reduced map from the full-map states its tensor route leaves
// (kata_map_state.cu): src [BH * nsrc][n(dsrc)][64] and z [BH * nsrc][n(dsrc)]
// in the decode layout, to the map's state [BH][n][64] and z [BH][n] in the
// packed order of its lift.
//   KATA-M_g: source a (of nsrc = g) is block a's full map, in the first
//     m = d / g coordinates of its dsrc (the rest zero padding); the map's block
//     a takes the features of those m coordinates.
//   KATA-Sigma_g: the sources are the full maps of the key blocks (nsrc = g,
//     dsrc = m); psi = eps I + s sum_a u_a u_a^T gives
//     S = s sum_a S_a + eps [f diagonal] sum_t v_t and z = s sum_a z_a + eps [f diagonal] T,
//     sum_t v_t from eps_totals.
cudaError_t map_state_compose(const float *src_state, const float *src_z, int nsrc, int dsrc,
                              const MapSpec &map, int d, const float *eps_totals, int T,
                              float *state, float *z, int BH, cudaStream_t stream);
// Reads and clears the sticky device error word of the tensor-core kernels
// (nonzero: a bounded wait expired); -1 if it could not be read.
int tc_take_error();
void tc_arm_stall();   // test hook: the next segment-state launch issues no loads
int pair_take_error();
// Segments per head of the d = 32 tensor path and the tokens in each (all but
// the last); the output of a segment starts from the scan's prefix state.
int tc_segments(const FwdShape &s, int num_sms, int *seg_tokens);

// ---- tcgen05 path at d = 64 (state split over four CTAs): kata_tc64.cu -----
bool tc64_supported(const FwdShape &s, int cc_major, int cc_minor, int num_sms);
// sigma (KATA-Sigma_1 at d = 64, eps I + s u u^T): the full map's numerators and
// denominator stay in fp32 and the finalize pass of kata_sigma.cu adds the
// map's eps terms; so then receives the full map's state and so.eps_totals the
// eps sums, for map_state_compose.
size_t tc64_workspace_bytes(const FwdShape &s, bool with_state = false,
                            const MapSpec *sigma = nullptr);
cudaError_t tc64_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                         void *out, void *workspace, cudaStream_t stream,
                         const StateOut &so = StateOut{}, const MapSpec *sigma = nullptr);
int tc64_take_error();

// ---- quadratic (flash-style) forward: kata_quad.cu ------------------------
bool quad_supported(const FwdShape &s, int cc_major, int cc_minor);
// gamma non-null: the GatedKATA weights (gamma [BH][T]; ws of
// quad_gated_workspace_bytes; normalize 0 drops the denominator).
cudaError_t quad_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                         void *out, cudaStream_t stream, const float *gamma = nullptr,
                         int normalize = 1, void *ws = nullptr);
size_t quad_gated_workspace_bytes(const FwdShape &s);
// Per 128-token chunk of every head: the keys scaled by the square root of the
// gates after them to the end of their chunk (kp, bf16 [BH][T][d]), the
// chunk-local inclusive cumulative log2 of the gates (lam2 [BH][T], a gate below
// 2^-126 counted as 2^-126) and each chunk's gate product (gtile [BH][NC]).
cudaError_t gate_prep_launch(const void *k, const float *gamma, void *kp, float *lam2, float *gtile,
                             int BH, int T, int d, cudaStream_t stream);
int quad_take_error();

}  // namespace kata
