/*
 * kata.h -- C ABI of libkata: causal kernelized linear attention with the
 * rank-one PSD feature map (KATA) on NVIDIA GB300 (sm_103a).
 *
 * Method: "Kernelized Linear Attention: Breaking the Capacity Wall with
 * Symmetric Cones" (KATA, arXiv 2607.17419v1).
 *
 *   psi(x) = vech(x x^T) in R^n, n = d(d+1)/2            (Sec. 3.1, Sec. 4.1)
 *            upper triangle, row-major, i <= j:
 *              f(i,j) = i*d - i*(i-1)/2 + (j - i),
 *              psi_f = x_i^2 (i == j),  sqrt(2) x_i x_j (i < j),
 *            so that psi(q) . psi(k) = (q . k)^2 >= 0.
 *   o_t    = psi(q_t)^T S_t / psi(q_t)^T Z_t,              (Sec. 2, Eq. 2)
 *            S_t = sum_{s<=t} psi(k_s) v_s^T, Z_t = sum_{s<=t} psi(k_s)
 *          = sum_{s<=t} (q_t.k_s)^2 v_s / sum_{s<=t} (q_t.k_s)^2.
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense, row-major, contiguous, in the caller's memory.  The
 *     library never frees or keeps a pointer it is given.
 *   - q, k are [B][H][T][d]; v and out are [B][H][T][dv]; all of q, k, v and
 *     out have the element type `dtype` (KATA_F32 or KATA_BF16).
 *   - Every device pointer must be 16-byte aligned.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and is asynchronous unless stated otherwise.
 *   - Accumulation is fp32.  A row whose denominator is exactly zero (its query
 *     orthogonal to every key so far) is written as zeros.
 *   - Return value: KATA_OK (0) or a negative kata_status.  Argument errors are
 *     detected on the host before any work is enqueued, and leave every
 *     output untouched.  KATA_ERR_CUDA reports a CUDA runtime error from a
 *     launch or allocation (the CUDA error state is cleared first).
 *   - There is no CPU fallback: unsupported shapes return
 *     KATA_ERR_UNSUPPORTED.
 */
#ifndef KATA_H_
#define KATA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef enum {
    KATA_OK = 0,
    KATA_ERR_ARG = -1,         /* null pointer, misaligned pointer, bad size */
    KATA_ERR_UNSUPPORTED = -2, /* valid but unsupported shape or dtype       */
    KATA_ERR_CUDA = -3,        /* CUDA runtime error                         */
    KATA_ERR_ALLOC = -4,       /* device workspace allocation failed         */
    KATA_ERR_TIMEOUT = -5,     /* a bounded device-side wait expired         */
    KATA_ERR_SCRATCH_LIMIT = -6 /* shape needs more scratch than the fixed
                                   buffer of kata_fwd_chunked_noalloc holds    */
} kata_status;

/* Capacity of the fixed device scratch array of kata_fwd_chunked_noalloc. */
#define KATA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Element types of q, k, v and out. */
typedef enum { KATA_F32 = 0, KATA_BF16 = 1 } kata_dtype;

/* Implementation a forward call runs on (see kata_fwd_path). */
typedef enum {
    KATA_PATH_NONE = 0, /* the shape is rejected                                 */
    KATA_PATH_SIMT = 1, /* fp32 CUDA-core kernels (used for KATA_F32 inputs)     */
    KATA_PATH_TC = 2    /* tcgen05 tensor-core kernels (bf16 inputs, sm_103a)    */
} kata_path;

/* Feature map of kata_fwd_chunked_map ([KATA] Sec. 4.1): the full rank-one map,
 * the two reduced PSD families, and the orthant map of the pages' linear-state
 * baselines (kernel appendix; one feature per coordinate). */
typedef enum {
    KATA_MAP_FULL = 0,   /* psi(u) = u u^T                                        */
    KATA_MAP_BLOCK = 1,  /* KATA-M_g: psi(u) = (u_1 u_1^T, ..., u_g u_g^T)         */
    KATA_MAP_SUM = 2,    /* KATA-Sigma_g: psi(u) = eps I + scale sum_a u_a u_a^T    */
    KATA_MAP_ORTHANT = 3 /* psi(u)_i = max(u_i, 0) + eps, n = d (g = 1, scale 1)   */
} kata_map;

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *kata_stream_t;

/* n = d(d+1)/2, the packed width of the lift (Sec. 4.1); -1 if d < 1. */
int kata_feature_dim(int d);

/* Packed feature width of a map with g blocks of width m = d/g: d(d+1)/2
 * (full), g m(m+1)/2 (KATA-M_g), m(m+1)/2 (KATA-Sigma_g) or d (orthant) -- the
 * pages' state sizes over d_v (Sec. 4.1); -1 for an invalid map, d or g. */
int kata_map_feature_dim(int map, int d, int g);

/* Static human-readable text for a status code. */
const char *kata_status_str(int status);

/*
 * kata_fwd_chunked -- causal KATA forward in the exact O(T) chunked-state
 * form (Sec. 4.1, Eq. 17-20; App. D.2, Algorithm 1; App. E.1 three-stage
 * pipeline): per chunk of C tokens, the masked squared-score intra-chunk term
 * (Psi(Q)Psi(K)^T .* M = (Q K^T)^2 .* M, M lower-triangular with the
 * diagonal), the chunk state Psi(K)^T [V | 1], an exclusive prefix scan of the
 * states over chunks, and the normalised output O = diag(D)^-1 N.
 *
 *   q, k  [B][H][T][d]   device, dtype, read only
 *   v     [B][H][T][dv]  device, dtype, read only
 *   out   [B][H][T][dv]  device, dtype, written (may not alias the inputs)
 *   B, H, T >= 1; d in {16, 32, 64}; dv in {16, 32, 64, 128};
 *   C in {32, 64, 128}: the chunk of Eq. 17-20.  T need not be a multiple of
 *   C: the last chunk is zero-padded (Algorithm 1), padded rows are dropped.
 *
 * The output is the same function for every C (Eq. 17-20 regroup one sum);
 * C changes only the rounding.  bf16 inputs run on the tensor-core path, which
 * rounds the lifted features and the chunk-state prefix to bf16 as MMA
 * operands (fp32 accumulation), for every d and dv.  At d = 64 each head's
 * chunks run in order on four CTAs (fewer than 38 heads leave SMs idle; the
 * quadratic form, which kata_fwd takes there, is then faster for longer T).  Its
 * kernels take d = 32 or 64 with dv = 64; other head
 * sizes run on them through scratch copies: q and k padded with zero columns
 * to d = 32 (d = 16), v cut into 64-column parts (dv = 16, 32 zero-padded; dv =
 * 128 as two parts, each a full pass of the kernels).  Both are exact
 * rewritings of Eq. 17-20.  fp32 inputs run on CUDA cores in fp32
 * (kata_fwd_path tells which).
 *
 * Scratch: per-call device workspace (kata_fwd_workspace_size bytes) taken
 * from the device's stream-ordered memory pool and released on `stream`.
 * Returns KATA_ERR_ALLOC if that allocation fails.
 */
int kata_fwd_chunked(const void *q, const void *k, const void *v, void *out, int B, int H,
                     int T, int d, int dv, int C, int dtype, kata_stream_t stream);

/*
 * kata_fwd_chunked_state -- kata_fwd_chunked plus the state after the last
 * token, so that a prefill hands off to kata_decode_step: S_T = sum_{t<T}
 * psi(k_t) v_t^T and z_T = sum_{t<T} psi(k_t) (Eq. 17 at the end of the last
 * chunk; App. D.1 "Plain KATA" state), in the decode layout.
 *
 *   q, k, v, out, B, H, T, d, dv, C, dtype, stream: as kata_fwd_chunked
 *   state  [B][H][n][dv]  device, fp32, written (n = d(d+1)/2)
 *   z      [B][H][n]      device, fp32, written
 *
 * Features are in the row-major upper-triangle order of kata_lift with sqrt(2)
 * on the off-diagonal entries (the layout kata_decode_step reads), whatever
 * order the forward uses inside.  state and z must be 16-byte aligned and may
 * not overlap each other or the other buffers (KATA_ERR_ARG).  The state is
 * accumulated in fp32; on the tensor-core path its terms are products of the
 * bf16-rounded lifted keys with v.  Other errors as kata_fwd_chunked.
 */
int kata_fwd_chunked_state(const void *q, const void *k, const void *v, void *out, float *state,
                           float *z, int B, int H, int T, int d, int dv, int C, int dtype,
                           kata_stream_t stream);

/*
 * kata_fwd_chunked_map -- the chunked forward with a reduced PSD feature map
 * ([KATA] Sec. 4.1, "two reduced PSD families"; the eps I term and scale of the
 * Sigma configuration).  q and k are cut into g blocks u_a of width m = d/g:
 *
 *   KATA_MAP_BLOCK (KATA-M_g):     psi(u) = (u_1 u_1^T, ..., u_g u_g^T),
 *                                  <psi(q), psi(k)> = sum_a (q_a . k_a)^2;
 *   KATA_MAP_SUM   (KATA-Sigma_g): psi(u) = eps I + scale sum_a u_a u_a^T,
 *                                  <psi(q), psi(k)> = eps^2 m + eps scale
 *                                  (|q|^2 + |k|^2) + scale^2 sum_{a,b} (q_a . k_b)^2;
 *   KATA_MAP_FULL with g = 1:      kata_fwd_chunked;
 *   KATA_MAP_ORTHANT with g = 1:   psi(u)_i = max(u_i, 0) + eps, n = d,
 *                                  <psi(q), psi(k)> = sum_i (q_i^+ + eps)(k_i^+ + eps)
 *                                  (the pages' linear-state family; eps = 1e-6 in
 *                                  their configuration; scale must be 1).
 *
 * Eq. 17-20 with this psi: states of kata_map_feature_dim(map, d, g) x (dv + 1).
 *   map, g: g in {1, 2, 4} dividing d; KATA_MAP_FULL and KATA_MAP_ORTHANT need g = 1.
 *   eps >= 0 and scale > 0, finite; KATA_MAP_FULL and KATA_MAP_BLOCK need
 *   eps = 0 and scale = 1 (KATA_ERR_ARG otherwise).
 * Other arguments, layouts, scratch and errors as kata_fwd_chunked.  With bf16
 * inputs, d = 64 and dv = 64, two maps run on the tensor cores as d = 32
 * sub-heads whose fp32 numerators and denominators add:
 *   KATA-M_2: two sub-heads, (q_a . k_a)^2 for a = 1, 2;
 *   KATA-Sigma_2: four sub-heads, (q_a . k_b)^2 for every (a, b), scaled by
 *   scale^2, plus the eps terms as a linear attention with the query features
 *   (eps^2 m + eps scale |q|^2, eps scale) and the key features (1, |k|^2),
 *   summed in fp32 in 128-token chunks.
 *   KATA-M_4: four sub-heads on the 16-wide blocks, each zero-padded to 32
 *   columns in scratch (the zero coordinates add nothing to (q_a . k_a)^2).
 * KATA-M_2 at d = 32 runs as M_2 at d = 64 on the rows [u_1 0 | u_2 0] (copied
 * to scratch), i.e. two zero-padded d = 32 sub-heads.  KATA-Sigma_1 (eps I +
 * s u u^T, m = d) at d = 32 and d = 64 runs as the full map on the tensor path of
 * that d, its numerators and denominator kept in fp32, scaled by scale^2, plus
 * the same eps terms.
 * With bf16 inputs and dv = 64, the other maps with at most 192 packed features
 * (KATA-Sigma_4 at d = 64; Sigma_2, Sigma_4 and M_4 at d = 32; every map at
 * d = 16; the orthant map) run on the tensor cores with their features written
 * out: psi of every q and k row in two bf16 parts (psi = hi + lo to ~2^-16),
 * per 128-token chunk the state Psi(K)^T V from the hi part and an fp32 record
 * [n][dv + 1], the chunk scan, and per chunk the output with the intra-chunk
 * weights Psi(Q) Psi(K)^T from the hi and lo parts (the weights are signed sums
 * that can be much smaller than the features; bf16 parts alone would leave
 * them ~2^-9 |psi(q)| |psi(k)| off) and Psi(Q) S_pre from the hi part.  Scratch
 * per token and head: 8 n bytes of features plus the records, about 260 n
 * bytes per 128-token chunk.  bf16 with dv in {16, 32, 128} runs the dv = 64
 * route of the map on 64-column parts of v (the last one zero-padded; an
 * output column depends only on its own v column), the parts' outputs copied
 * back.  The other reduced maps run on CUDA cores in fp32 (bf16 inputs are
 * widened; the output is written in the input type).  kata_fwd_path_map tells
 * which.
 */
int kata_fwd_chunked_map(const void *q, const void *k, const void *v, void *out, int B, int H,
                         int T, int d, int dv, int C, int dtype, int map, int g, float eps,
                         float scale, kata_stream_t stream);

/*
 * kata_fwd_chunked_map_state -- kata_fwd_chunked_map plus the state after the
 * last token under the map (Eq. 2's recurrence with the map's psi, at the end of
 * the last chunk), for kata_decode_step_map to continue:
 *   state [B][H][n][dv] fp32 = sum_t psi(k_t) v_t^T, z [B][H][n] fp32 =
 *   sum_t psi(k_t), n = kata_map_feature_dim(map, d, g), features in the packed
 *   order of kata_lift_map (each matrix row-major over its upper triangle,
 *   sqrt(2) off the diagonal, M_g's matrices block by block).
 * state and z 16-byte aligned, not overlapping each other or the other buffers
 * (KATA_ERR_ARG).  The routes built from full-map heads (M_2, Sigma_2, M_4 and
 * Sigma_1 at d = 64; M_2 and Sigma_1 at d = 32) compose the map's state from
 * their heads' full-map states: M_g's blocks are its sub-heads' (the first
 * m = d / g coordinates of a zero-padded one), and Sigma_g's is
 * scale (S_1 + ... + S_g) + eps sum_t v_t on the diagonal features (z the same
 * with T), S_a the full-map state of key block a;
 * the explicit-feature path exports its scanned records (products of the bf16
 * hi feature parts with v, accumulated in fp32).  Other arguments and errors as
 * kata_fwd_chunked_map.
 */
int kata_fwd_chunked_map_state(const void *q, const void *k, const void *v, void *out,
                               float *state, float *z, int B, int H, int T, int d, int dv, int C,
                               int dtype, int map, int g, float eps, float scale,
                               kata_stream_t stream);

/*
 * kata_decode_step_map -- one decode step under a map, in place:
 *   S += psi(k) v^T, z += psi(k), o = psi(q)^T S / psi(q)^T z (0 where the
 *   denominator is not positive), psi the map's packed features.
 * Layouts, alignment, ownership and errors as kata_decode_step with
 * n = kata_map_feature_dim(map, d, g); map, g, eps, scale as kata_fwd_chunked_map.
 */
int kata_decode_step_map(float *state, float *z, const void *q, const void *k, const void *v,
                         void *out, int B, int H, int d, int dv, int dtype, int map, int g,
                         float eps, float scale, kata_stream_t stream);

/*
 * kata_fwd_quadratic -- the quadratic (flash-style) form of the same forward:
 * o_t = sum_{s<=t} (q_t . k_s)^2 v_s / sum_{s<=t} (q_t . k_s)^2 evaluated tile
 * by tile, with no state ([KATA] Sec. 2 Eq. 2 directly; the pages' O(T^2)
 * kernel).  O(T^2) work against the chunked form's O(T n dv): the faster form
 * while T is short against n = d(d+1)/2.  The weights are non-negative, so no
 * running maximum is kept.
 *   q, k, v, out, B, H, T, d, dv, dtype, stream: as kata_fwd_chunked (no C).
 *   Supported: bf16 on sm_103a (KATA_ERR_UNSUPPORTED otherwise).  The kernel
 *   takes d in {32, 64} with dv = 64 and needs no workspace; the other head
 *   sizes (d = 16, dv in {16, 32, 128}) run on it as kata_fwd_chunked runs them
 *   (q, k padded to d = 32, v in 64-column parts, one pass per part), with a
 *   workspace for those copies allocated and freed stream-ordered inside the
 *   call (KATA_ERR_ALLOC if that fails).  Rounding as the tensor-core chunked
 *   path (P in bf16 as an MMA operand, fp32 accumulation and denominators).
 */
int kata_fwd_quadratic(const void *q, const void *k, const void *v, void *out, int B, int H,
                       int T, int d, int dv, int dtype, kata_stream_t stream);

/*
 * kata_fwd_quadratic_gated -- GatedKATA (see kata_fwd_chunked_gated for the
 * recurrence and the two readouts) in the quadratic form on the tensor cores:
 * every causal pair weighted by prod_{r=s+1}^{t} gamma_r (q_t . k_s)^2, tile by
 * tile with no state.  The gate products are folded into the keys of the tiles
 * below the diagonal (K'_s = sqrt(c_s) k_s, c_s <= 1 the gates after s to the
 * end of its 128-token tile), a per-row and a per-tile factor, and on the
 * diagonal tile into 2^(l_t - l_s) from the tile-local cumulative log2 of the
 * gates (a gate below 2^-126 counts as 2^-126 there: a zero gate leaves a
 * weight of at most 2^-126 on the writes before it within the tile).
 *   gamma [B][H][T] fp32 device, 16-byte aligned, values in [0, 1].
 *   normalize 0 or 1 as kata_fwd_chunked_gated.
 * Supported shapes, rounding and other arguments as kata_fwd_quadratic.
 * Workspace (scaled keys, cumulative log2 gates, tile gate products;
 * B H T (2 d + 4) bytes and a little more) is allocated and freed
 * stream-ordered inside the call.
 */
int kata_fwd_quadratic_gated(const void *q, const void *k, const void *v, const float *gamma,
                             void *out, int B, int H, int T, int d, int dv, int dtype,
                             int normalize, kata_stream_t stream);

/*
 * kata_fwd_chunked_gated -- GatedKATA, the pages' "multiplicative scalar state
 * gate" variant ([KATA] appendix on recurrent variants; Sec. 5.2): a gate
 * gamma_t in [0, 1] inside the recurrence,
 *   S_t = gamma_t S_{t-1} + psi(k_t) v_t^T,  Z_t = gamma_t Z_{t-1} + psi(k_t),
 * so write s reaches token t with the weight prod_{r=s+1}^{t} gamma_r (q_t . k_s)^2;
 *   normalize = 1: out_t = psi(q_t)^T S_t / psi(q_t)^T Z_t (the convex readout of
 *                  Prop. 1 over the gated weights; a zero denominator gives 0);
 *   normalize = 0: out_t = psi(q_t)^T S_t (the no-denominator readout of the
 *                  pages' MQAR configuration).
 * Computed in the chunked form of Eq. 17-20 with the chunk's gate products
 * folded into the state, the scan and the output.  bf16 inputs with d = 32 and
 * dv = 64 take the tensor cores (kata_fwd_path_gated reports which path a
 * shape takes): the d = 32 segments of kata_fwd_chunked, with the keys scaled by
 * the square root of the gates after them (to the end of their 128-token chunk
 * for the running state, to the end of their piece for the segment sums, as
 * bf16), the queries by the square root of the gates from their chunk's start,
 * a gated segment scan, the running state and Gram decayed by each chunk's gate
 * product in TMEM, and the intra-chunk weights multiplied by 2^(l_t - l_s) from
 * the chunk-local cumulative log2 of the gates (a gate below 2^-126 counts as
 * 2^-126 there: a zero gate leaves a weight of at most 2^-126 on the writes
 * before it within the chunk).  bf16 inputs with d = 64, dv = 64 and T <= 262144
 * take the tensor cores as well.  The other bf16 head sizes (d = 16, dv in {16,
 * 32, 128}) run on these two routes as kata_fwd_chunked runs them (q, k padded
 * to d = 32, v in 64-column parts; gates act on the weights only, so each part
 * is one gated forward), under the same bounds.  The output comes from the gated quadratic form
 * (kata_fwd_quadratic_gated), which evaluates the same weights tile by tile.
 * The state is sum_s A_s psi(k_s) v_s^T, A_s the product of the gates after s,
 * and psi is quadratic, so the state comes from the chunked d = 64 tensor path
 * run on the keys sqrt(A_s) k_s (rounded to bf16).  Other shapes run on CUDA
 * cores in fp32 FFMA.
 *
 *   gamma    [B][H][T] fp32 device, read only, 16-byte aligned; values in [0, 1]
 *            (not checked on the device: other values give the recurrence's
 *            arithmetic as written; gamma = 0 resets the state exactly).
 *   state, z both null, or both set: [B][H][n][dv] and [B][H][n] fp32 device,
 *            written with the gated state after the last token, in the layout
 *            kata_decode_step_gated reads.
 *   normalize 0 or 1 (KATA_ERR_ARG otherwise).
 * q, k, v, out, B, H, T, d, dv, C, dtype, stream: as kata_fwd_chunked.
 * Workspace: allocated and freed stream-ordered inside the call.
 */
int kata_fwd_chunked_gated(const void *q, const void *k, const void *v, const float *gamma,
                           void *out, float *state, float *z, int B, int H, int T, int d, int dv,
                           int C, int dtype, int normalize, kata_stream_t stream);

/* kata_fwd_path_gated -- the path kata_fwd_chunked_gated takes for a shape
 * without the state export: KATA_PATH_TC (tensor cores), KATA_PATH_SIMT (CUDA
 * cores) or KATA_PATH_NONE (invalid shape or no device); the same with the
 * state exported. */
int kata_fwd_path_gated(int B, int H, int T, int d, int dv, int C, int dtype);

/*
 * kata_fwd_chunked_noalloc -- the same forward as kata_fwd_chunked (same
 * arguments, layouts, paths and results), for callers that cannot allocate
 * device memory where they run it: code whose device memory is owned by a
 * framework pool that forbids other allocators, hosts that must not allocate
 * after start-up, and replays of pre-recorded GPU work that may not contain
 * allocations.  The paper has no counterpart; this is an interface choice.
 *
 * It allocates nothing.  Its scratch is one fixed device array of
 * KATA_NOALLOC_SCRATCH_BYTES (32 MiB) that is part of the library's device
 * image.  It is reserved when that device code is loaded: with the default
 * lazy loading, at this entry point's first call on a device; with eager
 * module loading (CUDA_MODULE_LOADING=EAGER), on every device context of the
 * process.  It stays reserved until the process exits.
 *
 * It takes the kernel family kata_fwd_chunked takes for the shape (see
 * kata_fwd_path) and needs the scratch kata_fwd_workspace_size reports; a
 * shape that needs more than the array returns KATA_ERR_SCRATCH_LIMIT before
 * any device work.  Every bf16 shape with d = 32 and dv = 64 fits on a
 * 152-SM GPU.  The d = 64 tensor path needs about 1 KB per token and head
 * (B*H*T up to roughly 32 K).  The scratch copies of the other head sizes add,
 * per token and head, 128 bytes for q and k padded to d = 32 (d = 16) and 256
 * bytes for one 64-column part of v and its output (dv != 64): B*H*T up to
 * about 256 K for d = 16 with dv = 64, 128 K for d = 32 with dv != 64 and 85 K
 * for d = 16 with dv != 64.  The CUDA-core path needs
 * B*H*(NC + NC/16 + 1)*n*(dv+1)*4 bytes with NC = ceil(T/C).
 *
 * The first call on each device (with that device current) looks up the
 * array's device address, which may load device code; make that first call
 * before any stream capture starts.  All calls share the array and it keeps
 * the last call's contents; no content has to start at zero, because each
 * call writes every byte it later reads.  Calls whose work overlaps on the
 * GPU (e.g. two streams without ordering) race on the array: order them.
 */
int kata_fwd_chunked_noalloc(const void *q, const void *k, const void *v, void *out, int B,
                             int H, int T, int d, int dv, int C, int dtype,
                             kata_stream_t stream);

/* Bytes of device workspace kata_fwd_chunked allocates for this shape, written
 * to *bytes.  Same argument checks as kata_fwd_chunked; no device work. */
int kata_fwd_workspace_size(int B, int H, int T, int d, int dv, int C, int dtype,
                            size_t *bytes);

/* Which implementation kata_fwd_chunked_map selects for this shape and map on
 * the current device (a kata_path value); KATA_PATH_NONE if it would reject it. */
int kata_fwd_path_map(int B, int H, int T, int d, int dv, int C, int dtype, int map, int g);

/* How kata_fwd_chunked cuts each head along the sequence on the current device:
 * returns the number of segments (>= 1) and writes the tokens of every segment
 * but the last to *seg_tokens (may be NULL); a negative kata_status for a shape
 * it would reject.  Segments are processed in parallel, each starting from the
 * exclusive prefix state of the segments before it ([KATA] Sec. 4.2, the scan
 * over chunks); the CUDA-core and d = 64 paths use one segment of T tokens.
 * For diagnostics and tests (the first rows after a segment start take the
 * scanned state); no device work. */
int kata_fwd_segments(int B, int H, int T, int d, int dv, int C, int dtype, int *seg_tokens);

/* Which implementation kata_fwd_chunked selects for this shape on the current
 * device (a kata_path value); KATA_PATH_NONE if it would reject the call.
 * Queries the device's compute capability, nothing else. */
int kata_fwd_path(int B, int H, int T, int d, int dv, int C, int dtype);

/* Which form kata_fwd runs for a shape on the current device. */
typedef enum {
    KATA_FORM_NONE = 0,       /* the shape is rejected                           */
    KATA_FORM_CHUNKED = 1,    /* kata_fwd_chunked                                */
    KATA_FORM_QUADRATIC = 2   /* kata_fwd_quadratic                              */
} kata_form;

/*
 * kata_fwd -- the forward in whichever exact form is faster for the shape:
 * the quadratic form (kata_fwd_quadratic) where it is supported and faster,
 * else the chunked form (kata_fwd_chunked).  At d = 32 (and d = 16, which runs
 * the d = 32 kernels) the quadratic form is faster up to T = 6144.  At d = 64 the
 * chunked kernels walk each head's chunks in order, so the bound depends on the
 * head count: the quadratic form is taken while B H T < 420000 x ceil(4 B H /
 * SMs) (T = 8192 at 128 heads, T = 26000 at 16, T = 420000 at one head; fitted to
 * GB300 timings of both forms).  Both compute the same o_t; they differ in rounding
 * only.  Arguments, layouts and errors as kata_fwd_chunked (C is used by the
 * chunked form).  kata_fwd_form tells which form a shape takes.
 */
int kata_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int T, int d,
             int dv, int C, int dtype, kata_stream_t stream);
int kata_fwd_form(int B, int H, int T, int d, int dv, int C, int dtype);

/*
 * kata_fwd_gated -- GatedKATA in whichever exact form is faster for the shape:
 * the gated quadratic form (kata_fwd_quadratic_gated) where it is supported and
 * T <= 10240 (d = 16 or 32) or T <= 65536 (d = 64), else the gated chunked form
 * (kata_fwd_chunked_gated, no state export).  The bounds come from the
 * measured per-token costs of both forms on GB300 (bf16, dv = 64): the
 * quadratic form's grows with T (1.1 ns per token and head at T = 8192, 1.9 at
 * 16384, d = 32); the chunked form's does not (1.3 ns at d = 32 on the tensor
 * cores).  At d = 64 the chunked call takes its output from the same gated
 * quadratic kernel up to T = 262144.  Arguments,
 * layouts, ownership and errors as kata_fwd_chunked_gated with state = z = NULL
 * (gamma [B][H][T] fp32 device; normalize 0 or 1).  kata_fwd_gated_form tells
 * which form a shape takes (a kata_form value).
 */
int kata_fwd_gated(const void *q, const void *k, const void *v, const float *gamma, void *out,
                   int B, int H, int T, int d, int dv, int C, int dtype, int normalize,
                   kata_stream_t stream);
int kata_fwd_gated_form(int B, int H, int T, int d, int dv, int C, int dtype);

/*
 * kata_fwd_chunked_host -- the same forward with HOST buffers: allocates
 * device buffers from the stream-ordered pool, copies q, k, v host->device,
 * runs kata_fwd_chunked, copies out device->host and waits for `stream`.
 * Pointers are host memory (pinned memory gives asynchronous copies).
 * Synchronous: returns after out holds the result.
 */
int kata_fwd_chunked_host(const void *q, const void *k, const void *v, void *out, int B,
                          int H, int T, int d, int dv, int C, int dtype,
                          kata_stream_t stream);

/*
 * kata_decode_step -- one recurrent decode step per (b, h) (Sec. 2, Eq. 2
 * additive recurrence; App. D.1 "Plain KATA"), updating the state in place and
 * then reading it out, so the step's own key is included as in Eq. 2:
 *   S += psi(k) v^T;  z += psi(k);  out = psi(q)^T S / psi(q)^T z.
 *
 *   state [B][H][n][dv] fp32 device, read and written (n = d(d+1)/2, packed in
 *         the order of psi above; a prefill state in this layout continues it)
 *   z     [B][H][n]     fp32 device, read and written
 *   q, k  [B][H][d]     device, dtype
 *   v     [B][H][dv]    device, dtype
 *   out   [B][H][dv]    device, dtype, written
 *   B, H >= 1; d in {16, 32, 64}; dv in {16, 32, 64, 128}.
 * No workspace.
 */
int kata_decode_step(float *state, float *z, const void *q, const void *k, const void *v,
                     void *out, int B, int H, int d, int dv, int dtype,
                     kata_stream_t stream);

/*
 * kata_decode_step_gated -- one GatedKATA step per (b, h), in place (the
 * recurrence of kata_fwd_chunked_gated at one token):
 *   S = gamma S + psi(k) v^T;  z = gamma z + psi(k);
 *   out = psi(q)^T S / psi(q)^T z (normalize = 1) or psi(q)^T S (normalize = 0).
 *   gamma [B][H] fp32 device, read only, 16-byte aligned, values in [0, 1].
 * Other arguments as kata_decode_step.
 */
int kata_decode_step_gated(float *state, float *z, const void *q, const void *k, const void *v,
                           const float *gamma, void *out, int B, int H, int d, int dv,
                           int dtype, int normalize, kata_stream_t stream);

/*
 * kata_lift -- the feature lift alone (Sec. 3.1 rank-one PSD map, packed as
 * in Sec. 4.1): phi[r][f] = psi(x_r)_f for rows r < rows.  The forward fuses
 * this lift into its kernels and never writes phi to memory; this entry point
 * exposes it for tests and for building states.
 *
 *   x   [rows][d]  device, dtype, read only
 *   phi [rows][n]  fp32 device, written
 *   rows >= 1; 1 <= d <= 64.
 */
int kata_lift(const void *x, float *phi, int64_t rows, int d, int dtype,
              kata_stream_t stream);

/* kata_lift_map -- the packed lift of a map (as kata_fwd_chunked_map defines
 * it) for rows of x: phi [rows][kata_map_feature_dim(map, d, g)] fp32.  Map
 * arguments as kata_fwd_chunked_map, other arguments as kata_lift. */
int kata_lift_map(const void *x, float *phi, int64_t rows, int d, int dtype, int map, int g,
                  float eps, float scale, kata_stream_t stream);

/*
 * kata_sync_status -- waits for `stream`, then reports and clears the sticky
 * device-side error word: KATA_ERR_TIMEOUT if a tensor-core kernel gave up a
 * bounded wait (it records the error and exits instead of hanging; its output
 * is then incomplete), KATA_OK otherwise.  No counterpart in the paper.
 */
int kata_sync_status(kata_stream_t stream);

/*
 * kata_test_arm_stall -- test hook for the failure path that kata_sync_status
 * reports.  It arms a host-side flag that the next launch of the tensor path's
 * segment-state kernel (a bf16 d = 32, dv = 64 call of kata_fwd_chunked that
 * cuts its heads into two or more segments) consumes: that launch issues no
 * tile loads, so every wait on the tiles runs out its bounded limit (about
 * 2 s per wave of CTAs), the kernel leaves through its abort path with no
 * copy or MMA in flight and its TMEM released, and the next kata_sync_status
 * returns KATA_ERR_TIMEOUT.  That call's output is undefined; later calls are
 * unaffected.  Returns KATA_OK.  No counterpart in the paper.
 */
int kata_test_arm_stall(void);

/*
 * Tracing (no counterpart in the paper; measurement support).  Between
 * kata_trace_begin and kata_trace_end, every kernel the library launches is
 * bracketed by two CUDA events recorded on the stream it is launched on.
 * kata_trace_end waits for those events, then reports per stage the number of
 * launches and their summed device time, and switches tracing off.  Stages
 * are named after the kernels ("chunk_state", "scan", "output", "decode",
 * "lift", ...).  Tracing is process-wide and off by default.
 */
typedef struct {
    char name[32];
    int launches;
    double total_ms;
} kata_trace_stage;

/* Start tracing (clears earlier records). */
int kata_trace_begin(void);

/* Stop tracing; writes up to max_stages entries to stages (may be NULL when
 * max_stages is 0) and the number of distinct stages seen to *n_stages.
 * Returns KATA_ERR_CUDA if an event could not be read. */
int kata_trace_end(kata_trace_stage *stages, int max_stages, int *n_stages);

#ifdef __cplusplus
}
#endif

#endif /* KATA_H_ */
