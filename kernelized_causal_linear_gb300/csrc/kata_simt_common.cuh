// Shared pieces of the CUDA-core (fp32 FFMA) chunked kernels: the plain and
// reduced-map path (kata_simt.cu) and GatedKATA (kata_gated.cu).  Both run the
// chunk-state and output contractions of the chunk form ([KATA] Sec. 4.1,
// Eq. 17-20) as register-tiled products in kata_simt.cu:
//
//   chunk state  [S_loc | z_loc] = Psi(K_c)^T [V_c | 1]       (features x columns)
//   output       [N | D] = Psi(Q_c) [S_pre | Z_pre] + P [V_c | 1]  (rows x columns)
//
// Each product walks its inner axis in 32-deep slabs staged in shared memory
// (double-buffered): features of Psi(Q_c) formed on the fly from the staged
// rows, then the masked weights P of each 32-key slab.  A thread accumulates an
// 8 x 4 tile (8 rows, 4 value columns); one extra warp accumulates the
// normaliser column for 8 rows per lane.
#pragma once
#include "kata_internal.cuh"

namespace kata {
namespace simt {

// gamma non-null selects the GatedKATA weights (gamma [BH][T]): the state
// kernel decays every key to the chunk end and writes the chunk gate products
// cgate [BH][NC]; the output kernel decays the prefix state by the gates from
// the chunk start and every intra-chunk weight by the gates between its key
// and its query.  normalize 0 drops the denominator.  n = mp.n(s.d).
template <typename T>
cudaError_t state_launch(const FwdShape &s, const T *k, const T *v, const float *gamma,
                         float *st, float *cgate, const MapSpec &mp, cudaStream_t stream,
                         const char *stage);
template <typename T>
cudaError_t output_launch(const FwdShape &s, const T *q, const T *k, const T *v,
                          const float *gamma, const float *st, T *out, const MapSpec &mp,
                          int normalize, cudaStream_t stream, const char *stage);

}  // namespace simt
}  // namespace kata
