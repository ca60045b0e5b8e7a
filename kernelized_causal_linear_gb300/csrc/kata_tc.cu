// tcgen05 tensor-core path of the KATA chunked forward (bf16 inputs, sm_103a).
//
// The method (KATA paper, Sec. 4.1 Eq. 17-20, App. D.2 Algorithm 1) walks the
// chunks of a head in order, carrying the state (S, Z).  To fill 152 SMs at
// small batch (B*H = 16 heads for T = 131072), each head is cut into G
// segments of whole 128-token chunks, and the exclusive scan over chunks of
// Eq. 17 (Sec. 4.2) is done at two levels:
//
//   1. seg_state_kernel   per (piece of a segment, head): the state sum
//                         Psi(K)^T V over the piece's chunks (tcgen05, fp32
//                         accumulators in TMEM) and its key Gram matrix K^T K;
//                         a segment is cut into m pieces when that fills more
//                         SMs.                                         [Eq. 17]
//   2. exclusive scan     of the piece records (CUDA cores); segment g's
//                         prefix is the record of its first piece.
//   3. seg_output_kernel  per (segment, head): starts from the segment's prefix
//                         state, held in TMEM in fp32, and walks its chunks:
//                           P   = (Q K^T)^2 .* M            (intra, Eq. 18)
//                           N   = P V + Psi(Q) S_pre        (Eq. 18)
//                           D   = P 1 + q^T G_pre q         (Eq. 19)
//                           O   = N / D                     (Eq. 20)
//                           S  += Psi(K)^T V, G += K^T K    (Eq. 17)
//                         all contractions on tcgen05 with operands in shared
//                         memory (TMA-fed for q, k, v tiles) and accumulators
//                         in TMEM.
//
// Both tensor kernels are warp-specialised: one warp issues TMA copies, one
// issues MMAs (one thread), and the other warps lift features, build P and
// convert accumulators; they hand buffers to each other through mbarriers, so
// the tensor pipe never waits on a __syncthreads.
//
// Normaliser.  Z = sum psi(k) is kept as the unpacked d x d matrix
// G = sum k k^T: psi(q).Z = <q q^T, G>_F = q^T G q (Sec. 3.1 Frobenius
// identity), which costs a d-column MMA instead of a ones column padded to 16
// in every state MMA, and keeps the fp32 state (5 x 64 TMEM columns) plus all
// accumulators inside the 512 TMEM columns of one SM.
//
// Feature order.  The forward never exports its state, so it uses its own
// order of the features of psi (the grouped layout described above lift_rect:
// cross-group 8 x 8 rectangles, then within-group triangles), with two
// features per 32-bit bf16 pair.  The sqrt(2) of the off-diagonal entries is
// applied as a factor 2 on the key side only (psi_q = q_i q_j, psi_k =
// 2 k_i k_j for i < j, k_i^2 on the diagonal), which keeps psi(q).psi(k) =
// (q.k)^2 and makes every lifted entry an exactly rounded bf16 product.
// Padded entries are zero.
//
// Chunk.  The tensor path uses 128-token chunks (the MMA tile height) for
// every requested C; Eq. 17-20 give the same function for any chunk size, so
// C only changes rounding.
//
// Variants of the output kernel: the sub-head form (M_2, M_4, Sigma_2 at d = 64
// as d = 32 sub-heads whose fp32 N and D are summed afterwards) and the gated
// form (GatedKATA: keys scaled by the gates, the running state decayed per
// chunk); both are described at the kernel.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "kata_tc_common.cuh"

namespace kata {

__device__ int g_tc_error = 0;   // sticky: bounded waits that expired

namespace {

__device__ __forceinline__ void flag_error(int code) { atomicOr(&g_tc_error, code); }


// ================================================================= kernel 1
// Segment state of one (segment, head): S_seg = sum over the segment's tokens of
// psi_k(k) v^T (all feature blocks, fp32 in TMEM) and G_seg = K^T K.
//   warp 0: TMA (K and V tiles, 2 stages)
//   warps 1-2: MMA issue, split so that one thread's barrier waits never idle
//     the tensor pipe: warp 1 the Gram and state blocks 0-1, warp 2 blocks 2-4
//   warps 3-10: key lift into a 4-slot ring (two warps per 32 tokens, each
//   lifting half of every block), then the epilogue (warps 3-6)
// stall (a test hook): the producer issues no tile loads, so every wait on the
// tiles expires and the kernel leaves through its abort path with no copy or
// MMA in flight.
constexpr int kStateRing = 4;
template <int D, int DV>
__global__ void __launch_bounds__(352, 1)
seg_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 float *__restrict__ seg, int NCt, int Lc, int m_pieces, int NR, int nsub,
                 int stall) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32 && C::NBLK == 5, "layouts below are written for d = 32, dv = 64");
    constexpr int kStage = C::QK_TILE + C::V_TILE;
    constexpr int kRing = kStateRing;
    constexpr int kLiftWarps = 8, kWarpLift = 3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *ring = sm + 2 * kStage;                     // [kRing][32 KB]: psi_k block
    __shared__ __align__(8) uint64_t tile_full[2], tile_empty[2], lift_full[kRing],
        lift_empty[kRing], done_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    // piece p of segment g: chunks g Lc + [p Lc / m, (p + 1) Lc / m) of the head
    const int piece = blockIdx.x, bh = blockIdx.y;
    const int g = piece / m_pieces, p = piece % m_pieces;
    // sub-head bh of nsub per head: columns D * (bh % nsub) .. of head bh / nsub
    const int hz = bh / nsub, hx = (bh % nsub) * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = g * Lc + (p * Lc) / m_pieces;
    const int nch = max(0, min(NCt, g * Lc + ((p + 1) * Lc) / m_pieces) - c0);
    const Sync sy{&abort_flag};
    float *rec = seg + ((size_t)bh * NR + piece) * C::E;
    if (nch == 0) {   // an empty piece (a short last segment) sums to zero
        for (int e = threadIdx.x; e < C::E; e += blockDim.x) rec[e] = 0.f;
        return;
    }

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tile_full[i], 1);
            mbar_init(&tile_empty[i], 2 + kLiftWarps);   // 2 MMA commits + lift warps
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&lift_full[i], kLiftWarps);
            mbar_init(&lift_empty[i], 1);                // the MMA thread of that block
        }
        mbar_init(&done_bar, 2);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base, tG = tmem_base + C::NBLK * DV;

    if (warp == 0) {
        // ---------------- TMA producer
        if (elect_lane0()) {
            for (int i = 0; i < (stall ? 0 : nch); ++i) {
                const int st = i & 1, use = i >> 1;
                if (use >= 1 && !sy.wait(&tile_empty[st], use - 1)) break;
                uint8_t *tk = sm + st * kStage;
                const int t0 = (c0 + i) * kTile;
                mbar_arrive_expect_tx(&tile_full[st], kStage);
                tma_load_3d(tk, &tm_k, hx, t0, hz, &tile_full[st]);
                tma_load_3d(tk + C::QK_TILE, &tm_v, 0, t0, hz, &tile_full[st]);
                if (i + 1 < nch) {   // warm L2 with the next chunk's tiles
                    tma_prefetch_3d(&tm_k, hx, t0 + kTile, hz);
                    tma_prefetch_3d(&tm_v, 0, t0 + kTile, hz);
                }
            }
        }
    } else if (warp < kWarpLift) {
        // ---------------- MMA issue: warp 1 = Gram + blocks 0-1, warp 2 = blocks 2-4
        if (elect_lane0()) {
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            // base descriptors: K tile as MN-major A/B of the Gram, lifted keys as
            // MN-major A and V as MN-major B of the state update
            const uint64_t dK = smem_desc(smem_u32(sm), 8192, 512, kSw64);
            const uint64_t dV = smem_desc(smem_u32(sm + C::QK_TILE), 16384, 1024, kSw128);
            const uint64_t dR = smem_desc(smem_u32(ring), 16384, 1024, kSw128);
            const bool first = warp == 1;
            const int b_lo = first ? 0 : 2, b_hi = first ? 2 : C::NBLK;
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                ok = sy.wait(&tile_full[st], i >> 1);
                if (!ok) break;
                tc_fence_after();
                if (first) {
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        const uint64_t a = desc_add(dK, st * kStage + ks * 1024);
                        mma_ss(tG, a, a, kIdGram, (i > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                for (int b = b_lo; b < b_hi && ok; ++b) {
                    const int gb = i * C::NBLK + b, rs = gb % kRing;
                    ok = sy.wait(&lift_full[rs], gb / kRing);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = desc_add(dR, rs * 32768), b0 = desc_add(dV, st * kStage);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + b * DV, desc_add(a0, ks * 2048), desc_add(b0, ks * 2048), kIdState,
                               (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&lift_empty[rs]);
                }
                mma_commit(&tile_empty[st]);
            }
            mma_commit(&done_bar);
        }
    } else {
        // ---------------- lift warps: token t, half h of every block
        const int lw = warp - kWarpLift;
        const int t = (lw & 3) * 32 + lane, h = lw >> 2;
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int st = i & 1;
            ok = __all_sync(0xffffffffu, sy.wait(&tile_full[st], i >> 1));
            if (!ok) break;
            PackedRow<D> r;
            tile_row_packed<D>(sm + st * kStage, t, r);
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&tile_empty[st]);
            for (int b = 0; b < C::NBLK && ok; ++b) {
                const int gb = i * C::NBLK + b, rs = gb % kRing, use = gb / kRing;
                if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&lift_empty[rs], use - 1));
                if (!ok) break;
                lift_block<2>(b, h, r, kTwo2, block_row(ring + rs * 32768, t));
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&lift_full[rs]);
            }
        }
        // ---------------- epilogue (warps 3-6): state and Gram rows to the segment record
        ok = __all_sync(0xffffffffu, sy.wait(&done_bar, 0));
        tc_fence_after();
        if (ok && h == 0) {
            const int quarter = warp & 3;
            const int lrow = quarter * 32 + lane;
            const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
            for (int b = 0; b < C::NBLK; ++b) {
                float4 *d4 = reinterpret_cast<float4 *>(rec + (size_t)(b * 128 + lrow) * DV);
                uint32_t v[64];
                tmem_ld64(tS + lsel + b * DV, v);
#pragma unroll
                for (int e = 0; e < DV / 4; ++e)
                    d4[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                        __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            }
            if (quarter == 0) {   // Gram rows 0..D-1 are TMEM lanes 0..D-1
                float *gd = rec + (size_t)C::NBLK * 128 * DV + (size_t)lane * D;
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tG + lsel + c, v);
                    float4 *d4 = reinterpret_cast<float4 *>(gd + c);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        d4[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                            __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) flag_error(1);
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Lift role of the output kernel: the q (or k) row of token t into both
// 64-feature atom columns of each block, through a 2-stage ring whose slots
// are 64 KB apart.  Kept out of line so that its registers are allocated apart
// from the other roles of the kernel.
// lam2 (gated queries): the chunk-local cumulative log2 of the gates of this
// head's tokens from chunk c0 on; the query row of token t is scaled by the
// square root of the gates from its chunk's start to t before it is lifted.
template <int D, int NB, bool kScaleQ>
__device__ __noinline__ void output_lift_role(const uint8_t *tile, uint8_t *ring, int t, bool key,
                                              int nch, uint64_t *chunk_full, uint64_t *qk_empty,
                                              uint64_t *block_ready, uint64_t *block_empty,
                                              volatile int *abort, const float *lam2, int nvalid) {
    const Sync sy{abort};
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
        ok = __all_sync(0xffffffffu, sy.wait(&chunk_full[i & 1], i >> 1));
        if (!ok) break;
        PackedRow<D> r;
        tile_row_packed<D>(tile, t, r);
        __syncwarp();
        if (elect_lane0()) mbar_arrive(qk_empty);
        if (kScaleQ && lam2 != nullptr) {
            const int ta = min(i * kTile + t, nvalid - 1);
            const float sc = exp2f(0.5f * lam2[ta]);
#pragma unroll
            for (int m = 0; m < D / 2; ++m)
                r.w[m] = pack_bf16(__uint_as_float(r.w[m] << 16) * sc,
                                   __uint_as_float(r.w[m] & 0xFFFF0000u) * sc);
        }
        for (int b = 0; b < NB && ok; ++b) {
            const int gb = i * NB + b, ls = gb & 1, use = gb >> 1;
            if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&block_empty[ls], use - 1));
            if (!ok) break;
            lift_block_rt(b, r, key ? kTwo2 : kOne2, block_row_rt(ring + ls * 65536, t));
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&block_ready[ls]);
        }
    }
}

// ================================================================= kernel 3
// Segment output: walk the segment's chunks with the running state in TMEM.
//   warp 0: TMA (Q, K tiles: 1 stage; V tile: 2 stages; the next chunk's
//     tiles are prefetched into L2)
//   warp 1: output MMAs (Q G_pre, Q K^T quarters, psi_q S_pre, P V)
//   warp 2: state MMAs (K^T K, psi_k^T V).  Two issuing threads keep the
//     tensor pipe fed while either one waits on a barrier.
//   warps 3-6 ("convert warps", lane quarter = warp % 4): S_run -> S_pre in
//     bf16, one 128-feature block at a time, into a 2-slot shared-memory ring
//   warps 7-10 ("P warps", lane quarter = warp % 4): P = (Q K^T)^2 masked, one
//     32-key quarter at a time, written back to TMEM in bf16 as the A operand
//     of P V; denominators; Gram -> bf16; output epilogue
//   warps 11-18: query/key lift into a 2-stage ring; each thread lifts one
//     token's row of one side (query or key) into both atom columns of a block
// TMEM: S_run [0,320) | G [320,352) | Q G_pre [352,384) | Q K^T quarter [384,416) |
//       P slots [416,432) [432,448) | output accumulator [448,512)
// kSub: sub-head form (KATA-M_2, KATA-Sigma_2): the epilogue writes the fp32
// numerator and the denominator of the sub-head for a finalize pass instead of O.
// cross: the nsub = 4 sub-heads of a head pair query half j / 2 with key half
// j % 2 (KATA-Sigma_2); otherwise sub-head j takes half j of both.  The segment
// prefixes then come from the key half's records (2 per head).
// kGated (GatedKATA, S_t = gamma_t S_{t-1} + psi(k_t) v_t^T): in chunk c with
// gate product g_c, cumulative log2 gates l_t from the chunk's start, and a_s the
// gates after s to the chunk's end,
//   S_run <- g_c S_run + sum_s psi(sqrt(a_s) k_s) v_s^T   (keys from tm_kg),
//   G     <- g_c G     + sum_s a_s k_s k_s^T,
//   N_t = psi(sqrt(b_t) q_t) . S_pre + sum_{s<=t} 2^(l_t - l_s) (q_t . k_s)^2 v_s,
//   D_t = b_t q_t^T G_pre q_t      + sum_{s<=t} 2^(l_t - l_s) (q_t . k_s)^2,
// b_t = 2^l_t.  The convert warps decay S_run block by block as they read it,
// the P warps decay G as they read it; O = N / D, or N when !normalize.
// kFin: fin receives the state after the head's last token.  S_run starts from
// the segment's exclusive prefix, so after the last segment's last chunk it is
// the head's whole state, and so is G (gated: S_run is decayed before each
// chunk's update and G's decay for the next chunk is 1 after the last one, so
// both are the gated totals); that CTA writes both in the record layout to
// fin[sbh] (crosswise: the query-half-0 sub-heads, one per key half).  A
// compile-time variant, so the kernel without it carries no export code.
struct OutGate {
    const float *lam2;     // [BH][T] chunk-local cumulative log2 of the gates
    const float *gchunk;   // [BH][NC] gate product of each 128-token chunk
    int normalize;
};
template <int D, int DV, bool kSub, bool kGated, bool kFin = false>
__global__ void __launch_bounds__(608, 1)
seg_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kg,
                  bf16 *__restrict__ out, const float *__restrict__ seg, int T, int NCt, int Lc,
                  int m_pieces, int NR, int nsub, int cross, float *__restrict__ part, OutGate ga,
                  float *__restrict__ fin) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32 && C::NBLK == 5, "layouts below are written for d = 32, dv = 64");
    constexpr int NB = C::NBLK;
    constexpr int kLastK = (C::NF - (NB - 1) * 128 + 15) / 16;   // K steps of the last block
    constexpr int kLiftWarps = 8, kTmemWarps = 4;
    constexpr int kWarpP = 7, kWarpLift = 11;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tq = sm;                                   // Q tile, 8 KB (64-byte swizzle)
    uint8_t *tk = sm + C::QK_TILE;                      // K tile, 8 KB
    // gated: the scaled K tile follows K.  The Gram MMA (M = 128, MN-major) reads
    // its operand as four 8 KB atoms 8 KB apart, i.e. 24 KB past the tile it
    // names, which here are the V tiles (the real rows are the first 32).
    uint8_t *tkg = sm + 2 * C::QK_TILE;
    uint8_t *tv = sm + (kGated ? 3 : 2) * C::QK_TILE;   // V tiles [2][16 KB]
    uint8_t *lring = tv + 2 * C::V_TILE;                // [2][psi_q 32 KB | psi_k 32 KB]
    uint8_t *spre = lring + 2 * 65536;                  // S_pre blocks [2][16 KB]
    uint8_t *gram = spre + 2 * 16384;                   // G_pre bf16, 2 KB
    // chunk_full[s]: the Q, K, V tiles of a chunk in stage s have landed and G_pre
    //   for it is in `gram` (TMA + P warps).
    // block_ready[s] / block_empty[s]: ring slot s holds psi_q, psi_k and S_pre of
    //   one block (lift + convert warps) / both MMA threads are done with it.
    __shared__ __align__(8) uint64_t chunk_full[2], qk_empty, v_empty[2], xs_full, p_full[2],
        p_empty[2], block_ready[2], block_empty[2], state_done[NB], o_full, o_empty, gram_done,
        qg_done, fin_bar[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int g = blockIdx.x, bh = blockIdx.y;
    // sub-head bh of nsub per head: q/k columns D * (bh % nsub) .. of head bh / nsub
    // (one sub-head per head, nsub = 1, unless kSub)
    const int hz = kSub ? bh / nsub : bh, j = kSub ? bh % nsub : 0;
    const bool xc = kSub && cross;
    const int qx = (xc ? j >> 1 : j) * D, kx = (xc ? j & 1 : j) * D;
    const int sbh = xc ? hz * 2 + (j & 1) : bh;   // records of this sub-head's keys
    float *const frec = (kFin && g == (int)gridDim.x - 1 && (!xc || (j >> 1) == 0))
                            ? fin + (size_t)sbh * C::E
                            : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;
    const Sync sy{&abort_flag};
    // gated: this segment's cumulative log2 gates (valid for nvalid tokens) and chunk gate products
    const float *lam2 = kGated ? ga.lam2 + (size_t)bh * T + (size_t)c0 * kTile : nullptr;
    const float *gch = kGated ? ga.gchunk + (size_t)bh * NCt + c0 : nullptr;
    const int nvalid = T - c0 * kTile;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&qk_empty, 2 + kLiftWarps + kTmemWarps);   // 2 MMA commits, lift warps, P warps
        for (int i = 0; i < 2; ++i) {
            mbar_init(&chunk_full[i], 1 + kTmemWarps);         // TMA arrive + P warps (G_pre)
            mbar_init(&v_empty[i], 2);
            mbar_init(&block_ready[i], kLiftWarps + kTmemWarps);   // lift + convert warps
            mbar_init(&block_empty[i], 2);
            mbar_init(&p_full[i], kTmemWarps);
            mbar_init(&p_empty[i], 1);
            mbar_init(&fin_bar[i], 1);
        }
        mbar_init(&xs_full, 1);
        for (int b = 0; b < NB; ++b) mbar_init(&state_done[b], 1);
        mbar_init(&o_full, 1);
        mbar_init(&o_empty, kTmemWarps);
        mbar_init(&gram_done, 1);
        mbar_init(&qg_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base, tG = tmem_base + 320, tQG = tmem_base + 352;
    const uint32_t tXs = tmem_base + 384, tP = tmem_base + 416, tXo = tmem_base + 448;

    if (warp == 0) {
        // ================= TMA producer
        if (elect_lane0()) {
            for (int i = 0; i < nch; ++i) {
                const int t0 = (c0 + i) * kTile;
                const int st = i & 1, use = i >> 1;
                if (i >= 1 && !sy.wait(&qk_empty, i - 1)) break;
                if (use >= 1 && !sy.wait(&v_empty[st], use - 1)) break;
                mbar_arrive_expect_tx(&chunk_full[st],
                                      (kGated ? 3 : 2) * C::QK_TILE + C::V_TILE);
                tma_load_3d(tq, &tm_q, qx, t0, hz, &chunk_full[st]);
                tma_load_3d(tk, &tm_k, kx, t0, hz, &chunk_full[st]);
                if constexpr (kGated) tma_load_3d(tkg, &tm_kg, 0, t0, hz, &chunk_full[st]);
                tma_load_3d(tv + st * C::V_TILE, &tm_v, 0, t0, hz, &chunk_full[st]);
                if (i + 1 < nch) {   // warm L2 with the next chunk's tiles
                    tma_prefetch_3d(&tm_q, qx, t0 + kTile, hz);
                    tma_prefetch_3d(&tm_k, kx, t0 + kTile, hz);
                    tma_prefetch_3d(&tm_v, 0, t0 + kTile, hz);
                }
            }
        }
    } else if (warp == 1) {
        // ================= output MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdQK = idesc_bf16(128, 32, false, false);
            constexpr uint32_t kIdQG = idesc_bf16(128, D, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
            // base descriptors, built once; each MMA only offsets the start address
            const uint64_t dQ = smem_desc(smem_u32(tq), 16, 512, kSw64);        // K-major A
            const uint64_t dKb = smem_desc(smem_u32(tk), 16, 512, kSw64);       // K-major B
            const uint64_t dGr = smem_desc(smem_u32(gram), 16, 512, kSw64);     // K-major B
            const uint64_t dSp = smem_desc(smem_u32(spre), 16384, 1024, kSw128); // MN-major B
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);  // MN-major B
            const uint64_t dLq = smem_desc(smem_u32(lring), 16, 1024, kSw128);  // K-major A
            auto qk_quarter = [&](int q) {   // Xs = Q K[32q .. 32q+31]^T
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tXs, desc_add(dQ, ks * 32), desc_add(dKb, q * 2048 + ks * 32), kIdQK,
                           ks > 0);
                mma_commit(&xs_full);
            };
            auto pv_quarter = [&](int n, uint32_t vo) {   // Xo += P_q V[32q .. 32q+31]
                const int q = n & 3, slot = n & 1;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_ts(tXo, tP + slot * 16 + ks * 8, desc_add(dV0, vo + (2 * q + ks) * 2048),
                           kIdPV, 1u);
                mma_commit(&p_empty[slot]);
            };
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t vo = st * C::V_TILE;     // byte offset of this chunk's V tile
                // tiles and G_pre of this chunk (the P warps read quarter 3 of the
                // previous chunk's Q K^T before building its P, waited for below)
                ok = sy.wait(&chunk_full[st], i >> 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tQG, desc_add(dQ, ks * 32), desc_add(dGr, ks * 32), kIdQG, ks > 0);
                mma_commit(&qg_done);
                qk_quarter(0);
#pragma unroll 1
                for (int b = 0; b < NB && ok; ++b) {
                    const int gb = i * NB + b, ls = gb & 1;
                    if (b > 0) {
                        // P of quarter b - 1 was built while block b - 1 ran: queue
                        // Q K^T quarter b and P V of quarter b - 1 ahead of this
                        // block's MMAs, so that quarter b's P is built while they run
                        const int n = 4 * i + b - 1;
                        ok = sy.wait(&p_full[n & 1], n >> 1);
                        if (!ok) break;
                        tc_fence_after();
                        if (b < 4) {
                            qk_quarter(b);
                            if (b == 3) mma_commit(&qk_empty);
                        }
                        pv_quarter(n, vo);
                    }
                    ok = sy.wait(&block_ready[ls], gb >> 1) &&
                         (b != 0 || i == 0 || sy.wait(&o_empty, i - 1));
                    if (!ok) break;
                    tc_fence_after();
                    // Xo (+)= psi_q S_pre for this block
                    const uint64_t a0 = desc_add(dLq, ls * 65536), b0 = desc_add(dSp, ls * 16384);
                    if (b < NB - 1) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ss(tXo, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32),
                                   desc_add(b0, ks * 2048), kIdPV, (b > 0 || ks > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < kLastK; ++ks)
                            mma_ss(tXo, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32),
                                   desc_add(b0, ks * 2048), kIdPV, 1u);
                    }
                    mma_commit(&block_empty[ls]);
                }
                if (!ok) break;
                mma_commit(&o_full);
                mma_commit(&v_empty[st]);
            }
            mma_commit(&fin_bar[0]);
            sy.wait(&fin_bar[0], 0);
        }
    } else if (warp == 2) {
        // ================= state MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            const uint64_t dKg = smem_desc(smem_u32(kGated ? tkg : tk), 8192, 512, kSw64); // MN-major (Gram)
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);  // MN-major B
            const uint64_t dLk = smem_desc(smem_u32(lring + 32768), 16384, 1024, kSw128); // MN-major A
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t vo = st * C::V_TILE;
                // G += K^T K, after the P warps have read G_pre for this chunk
                ok = sy.wait(&chunk_full[st], i >> 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    const uint64_t a = desc_add(dKg, ks * 1024);
                    mma_ss(tG, a, a, kIdGram, 1u);
                }
                mma_commit(&gram_done);
                mma_commit(&qk_empty);
#pragma unroll 1
                for (int b = 0; b < NB && ok; ++b) {
                    const int gb = i * NB + b, ls = gb & 1;
                    // S_run block b += psi_k^T V once the convert warps have read it
                    ok = sy.wait(&block_ready[ls], gb >> 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = desc_add(dLk, ls * 65536), b0 = desc_add(dV0, vo);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + b * DV, desc_add(a0, ks * 2048), desc_add(b0, ks * 2048), kIdState, 1u);
                    mma_commit(&state_done[b]);
                    mma_commit(&block_empty[ls]);
                }
                if (!ok) break;
                mma_commit(&v_empty[st]);
            }
            mma_commit(&fin_bar[1]);
            sy.wait(&fin_bar[1], 0);
        }
    } else if (warp < kWarpP) {
        // ================= convert warps: S_run block -> bf16 S_pre slot
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        {   // initial state: the segment's exclusive prefix (zero for g == 0)
            const float *pre = g > 0 ? seg + ((size_t)sbh * NR + (size_t)g * m_pieces) * C::E : nullptr;
            for (int b = 0; b < NB; ++b) {
#pragma unroll
                for (int c = 0; c < DV; c += 8) {
                    uint32_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        v[e] = pre ? __float_as_uint(pre[(size_t)(b * 128 + row) * DV + c + e]) : 0u;
                    tmem_st8(tS + lsel + b * DV + c, v);
                }
            }
            tmem_st_wait();
        }
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
#pragma unroll 1
            for (int b = 0; b < NB && ok; ++b) {
                const int gb = i * NB + b, ss = gb & 1, use = gb >> 1;
                bool w = (use == 0 || sy.wait(&block_empty[ss], use - 1)) &&
                         (i == 0 || sy.wait(&state_done[b], i - 1));
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                tc_fence_after();
                if (quarter * 32 < C::NF - b * 128) {   // rows past the real features are never read
                    const uint32_t srow = smem_u32(spre + ss * 16384 + (row >> 3) * 1024 + (row & 7) * 128);
                    const float gc = kGated ? gch[i] : 1.f;
#pragma unroll
                    for (int c32 = 0; c32 < DV; c32 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tS + lsel + b * DV + c32, v);
                        if constexpr (kGated) {   // S_run <- g_c S_run before this chunk's update
                            uint32_t dv32[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) dv32[e] = __float_as_uint(__uint_as_float(v[e]) * gc);
                            tmem_st32(tS + lsel + b * DV + c32, dv32);
                        }
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int chunk = (c32 >> 3) + cc;
                            st_shared_v4(srow + ((chunk ^ (row & 7)) << 4),
                                         pack_bf16(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1])),
                                         pack_bf16(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3])),
                                         pack_bf16(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5])),
                                         pack_bf16(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7])));
                        }
                    }
                    fence_proxy_async_smem();
                    if constexpr (kGated) tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&block_ready[ss]);
            }
        }
        // the final state: each block once its last state MMA is done
        for (int b = 0; kFin && b < NB && ok && frec != nullptr; ++b) {
            ok = __all_sync(0xffffffffu, sy.wait(&state_done[b], nch - 1));
            if (!ok) break;
            tc_fence_after();
            if (quarter * 32 >= C::NF - b * 128) continue;   // no real features in these rows
            float4 *dst = reinterpret_cast<float4 *>(frec + (size_t)(b * 128 + row) * DV);
#pragma unroll
            for (int c32 = 0; c32 < DV; c32 += 32) {
                uint32_t v[32];
                tmem_ld32(tS + lsel + b * DV + c32, v);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[c32 / 4 + e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            }
        }
    } else if (warp < kWarpLift) {
        // ================= P warps: lane quarter q owns query rows 32q..32q+31
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        // P for key quarter n % 4 of chunk n / 4 into P slot n % 2; adds this row's weights to dsum
        auto build_p = [&](int n, float &dsum) -> bool {
            const int q = n & 3, slot = n & 1;
            bool w = sy.wait(&xs_full, n) && (n < 2 || sy.wait(&p_empty[slot], (n >> 1) - 1));
            w = __all_sync(0xffffffffu, w);
            if (!w) return false;
            tc_fence_after();
            // every key of the quarter comes after this warp's rows: P is zero
            // (kept out of the gated kernel, where this branch measured slower)
            if (!kGated && quarter < q) {
                const uint32_t pz[16] = {};
                tmem_st16(tP + lsel + slot * 16, pz);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&p_full[slot]);
                return true;
            }
            uint32_t v[32];
            tmem_ld32(tXs + lsel, v);
            // gated: key s weighs 2^(l_t - l_s) for query t (lane s % 32 holds l_s)
            float lt = 0.f, lk = 0.f;
            if constexpr (kGated) {
                const int cb = (n >> 2) * kTile;
                lt = lam2[min(cb + row, nvalid - 1)];
                lk = lam2[min(cb + 32 * q + lane, nvalid - 1)];
            }
            uint32_t pw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s = 32 * q + 2 * j;
                float x0 = __uint_as_float(v[2 * j]), x1 = __uint_as_float(v[2 * j + 1]);
                x0 *= x0;
                x1 *= x1;
                if constexpr (kGated) {
                    x0 *= exp2f(lt - __shfl_sync(0xffffffffu, lk, 2 * j));
                    x1 *= exp2f(lt - __shfl_sync(0xffffffffu, lk, 2 * j + 1));
                }
                const float w0 = s <= row ? x0 : 0.f;
                const float w1 = s + 1 <= row ? x1 : 0.f;
                dsum += w0;
                dsum += w1;
                pw[j] = pack_bf16(w0, w1);
            }
            tmem_st16(tP + lsel + slot * 16, pw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&p_full[slot]);
            return true;
        };
        auto epilogue = [&](int i, float dsum) -> bool {   // O = N / D for chunk i
            bool w = __all_sync(0xffffffffu, sy.wait(&o_full, i));
            if (!w) return false;
            tc_fence_after();
            if constexpr (kSub) {   // sub-heads: N (fp32) and D, summed over sub-heads later
                const int t = (c0 + i) * kTile + row;
                float *dst = part + ((size_t)bh * T + t) * DV;
#pragma unroll
                for (int c32 = 0; c32 < DV; c32 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tXo + lsel + c32, v);
                    if (t < T)
#pragma unroll
                        for (int e = 0; e < 4; ++e) st_global_v8(dst + c32 + 8 * e, v + 8 * e);
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&o_empty);
                if (t < T) part[(size_t)gridDim.y * T * DV + (size_t)bh * T + t] = dsum;
                return true;
            }
            const float inv = (kGated && !ga.normalize) ? 1.f : dsum > 0.f ? 1.f / dsum : 0.f;
            uint32_t o[DV / 2];   // the row in bf16 pairs
#pragma unroll
            for (int c32 = 0; c32 < DV; c32 += 32) {
                uint32_t v[32];
                tmem_ld32(tXo + lsel + c32, v);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    o[c32 / 2 + e] = pack_bf16(__uint_as_float(v[2 * e]) * inv,
                                               __uint_as_float(v[2 * e + 1]) * inv);
            }
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&o_empty);
            const int t0 = (c0 + i) * kTile;
            if (t0 + row < T) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * T + t0 + row) * DV);
#pragma unroll
                for (int c = 0; c < DV / 8; ++c)
                    dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
            return true;
        };
        // gscale (gated): the factor G is left with in TMEM for the next Gram update;
        // gout: also the fp32 rows of G there
        auto gram_to_smem = [&](bool from_tmem, const float *pre, float gscale, float *gout) {
            // G rows i = lane (quarter 0 only): bf16 [D][D] K-major, 64-byte swizzle
            if (quarter != 0) return;
            float gv[D];
            if (from_tmem) {
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tG + lsel + c, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) gv[c + e] = __uint_as_float(v[e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < D; ++e) gv[e] = pre ? pre[lane * D + e] : 0.f;
            }
            if (kFin && gout != nullptr) {
                float4 *go = reinterpret_cast<float4 *>(gout + lane * D);
#pragma unroll
                for (int e = 0; e < D / 4; ++e)
                    go[e] = make_float4(gv[4 * e], gv[4 * e + 1], gv[4 * e + 2], gv[4 * e + 3]);
            }
#pragma unroll
            for (int chunk = 0; chunk < D / 8; ++chunk) {
                uint4 u;
                u.x = pack_bf16(gv[8 * chunk + 0], gv[8 * chunk + 1]);
                u.y = pack_bf16(gv[8 * chunk + 2], gv[8 * chunk + 3]);
                u.z = pack_bf16(gv[8 * chunk + 4], gv[8 * chunk + 5]);
                u.w = pack_bf16(gv[8 * chunk + 6], gv[8 * chunk + 7]);
                *reinterpret_cast<uint4 *>(gram + (lane >> 3) * 512 + (lane & 7) * 64 +
                                           ((chunk ^ ((lane >> 1) & 3)) << 4)) = u;
            }
            if (!from_tmem || (kGated && gscale != 1.f)) {
#pragma unroll
                for (int c = 0; c < D; c += 8) {
                    uint32_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(gv[c + e] * gscale);
                    tmem_st8(tG + lsel + c, v);
                }
                tmem_st_wait();
            }
        };
        // inter-chunk denominator q^T G_pre q (Q G_pre from TMEM, q from the Q
        // tile), then this chunk's Gram -> bf16 for the next chunk
        auto d_inter = [&](int i, float &dsum) -> bool {
            bool w = __all_sync(0xffffffffu, sy.wait(&chunk_full[i & 1], i >> 1) &&
                                                 sy.wait(&qg_done, i) && sy.wait(&gram_done, i));
            if (!w) return false;
            tc_fence_after();
            PackedRow<D> r;
            tile_row_packed<D>(tq, row, r);
            uint32_t v[32];
            tmem_ld32(tQG + lsel, v);
            float di = 0.f;
#pragma unroll
            for (int m = 0; m < D / 2; ++m) {
                di = fmaf(__uint_as_float(v[2 * m]), __uint_as_float(r.w[m] << 16), di);
                di = fmaf(__uint_as_float(v[2 * m + 1]), __uint_as_float(r.w[m] & 0xFFFF0000u), di);
            }
            if constexpr (kGated) di *= exp2f(lam2[min(i * kTile + row, nvalid - 1)]);   // b_t
            dsum += di;
            // after the last chunk, G is the head's whole Gram
            gram_to_smem(true, nullptr, (kGated && i + 1 < nch) ? gch[i + 1] : 1.f,
                         kFin && frec != nullptr && i == nch - 1 ? frec + (size_t)NB * 128 * DV : nullptr);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) {
                mbar_arrive(&chunk_full[(i + 1) & 1]);   // G_pre of chunk i + 1
                mbar_arrive(&qk_empty);
            }
            return true;
        };

        {   // initial Gram: the segment's exclusive prefix (zero for g == 0)
            const float *pre = g > 0 ? seg + ((size_t)sbh * NR + (size_t)g * m_pieces) * C::E : nullptr;
            gram_to_smem(false, pre ? pre + (size_t)NB * 128 * DV : nullptr, kGated ? gch[0] : 1.f, nullptr);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&chunk_full[0]);
        }
        bool ok = true;
        float dprev = 0.f;
        for (int i = 0; i <= nch && ok; ++i) {   // chunk i's P and denominators, chunk i-1's output
            if (i > 0) ok = epilogue(i - 1, dprev);
            if (i == nch) break;
            float dsum = 0.f;
#pragma unroll 1
            for (int q = 0; q < 4 && ok; ++q) {
                ok = build_p(4 * i + q, dsum);
                if (ok && q == 0) ok = d_inter(i, dsum);
            }
            dprev = dsum;
        }
    } else {
        // ================= lift warps: token t, side (0 query, 1 key)
        const int lw = warp - kWarpLift;
        const int side = lw >> 2;
        output_lift_role<D, NB, kGated>(side ? (kGated ? tkg : tk) : tq, lring + side * 32768, (lw & 3) * 32 + lane,
                                side != 0, nch, chunk_full, &qk_empty, block_ready, block_empty,
                                &abort_flag, side ? nullptr : lam2, nvalid);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) flag_error(2);
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ================================================================= state export
// The inclusive state of a head (a segment record summed over all segments:
// S in the grouped layout, 5 blocks x 128 features x DV, then the Gram
// G = sum k k^T) in the decode layout: state[f][c] and z[f] for the row-major
// upper-triangle feature f of (i, j), sqrt(2) on the off-diagonal entries.
// The grouped layout carries a factor 2 on the key side off the diagonal, so
// those rows are scaled by 1/sqrt(2); z_f is G_ij (sqrt(2) G_ij for i < j).
// Grid (NBLK + 1, heads), 128 threads: CTA b < NBLK moves feature block b (one
// thread per feature slot), CTA NBLK the Gram into z.
template <int D, int DV>
__global__ void __launch_bounds__(128)
state_export_kernel(const float *__restrict__ total, float *__restrict__ state,
                    float *__restrict__ z) {
    using C = Cfg<D, DV>;
    constexpr int kN = D * (D + 1) / 2;
    const int b = blockIdx.x, bh = blockIdx.y, p = threadIdx.x;
    const float *rec = total + (size_t)bh * C::E;
    float *st = state + (size_t)bh * kN * DV;
    if (b < C::NBLK) {
        int i = 0, j = 0;
        if (!grouped_slot_pair(b, p, i, j)) return;
        const int f = i * D - i * (i - 1) / 2 + (j - i);
        const float sc = i == j ? 1.f : 0.70710678118654752f;
        const float4 *src = reinterpret_cast<const float4 *>(rec + (size_t)(b * 128 + p) * DV);
        float4 *dst = reinterpret_cast<float4 *>(st + (size_t)f * DV);
#pragma unroll 4
        for (int e = 0; e < DV / 4; ++e) {
            const float4 x = src[e];
            dst[e] = make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc);
        }
        return;
    }
    const float *gram = rec + (size_t)C::NBLK * 128 * DV;
    for (int e = p; e < D * D; e += blockDim.x) {
        const int i = e / D, j = e % D;
        if (j < i) continue;
        z[(size_t)bh * kN + i * D - i * (i - 1) / 2 + (j - i)] =
            i == j ? gram[e] : kSqrt2 * gram[e];
    }
}

// ================================================================= host side
// Sub-heads (KATA-M_2 at d = 64): O = (N_0 + N_1) / (D_0 + D_1) in bf16 (zero
// where the sum of denominators is not positive), summed in sub-head order.
// part: N [BH * nsub][T][64] fp32, then D [BH * nsub][T].  One thread per four
// output values.
__global__ void __launch_bounds__(256)
sub_finalize_kernel(const float *__restrict__ part, bf16 *__restrict__ out, int64_t rows, int T,
                    int nsub) {
    const int64_t n4 = rows * 16;   // 64 values per row
    const float *dd = part + (size_t)rows * nsub * 64;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e >> 4, bh = row / T, t = row % T;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
        for (int a = 0; a < nsub; ++a) {
            const int64_t r = (bh * nsub + a) * T + t;
            const float4 x = reinterpret_cast<const float4 *>(part + r * 64)[e & 15];
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
            den += dd[r];
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(out) + 2 * e;
        o[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        o[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
}

constexpr int kSmemState = 2 * (Cfg<32, 64>::QK_TILE + Cfg<32, 64>::V_TILE) + kStateRing * 32768 + 2048;
constexpr int kSmemOutput = 2 * Cfg<32, 64>::QK_TILE + 2 * Cfg<32, 64>::V_TILE + 2 * 65536 +
                            2 * 16384 + 2048 + 2048;
constexpr int kSmemOutputGated = kSmemOutput + Cfg<32, 64>::QK_TILE;   // + the scaled K tile

// GatedKATA segment sums come from the keys scaled to the end of their piece:
// per chunk c of a summed piece, k''_s = sqrt(P_c) k'_s, where k'_s carries the
// gates after s to the end of chunk c and P_c is the product of the gates of the
// piece's later chunks.  The first chunk of each segment also writes the gate
// products of the segment's m pieces (the gated scan's multipliers; an empty
// piece has product 1).  Grid (summed chunks, heads), 128 threads.
__global__ void __launch_bounds__(128)
gated_piece_prep_kernel(const bf16 *__restrict__ kc, const float *__restrict__ gch,
                        bf16 *__restrict__ kpc, float *__restrict__ pgate, int T, int NCt, int Lc,
                        int m_pieces, int npieces, int NR) {
    __shared__ float wprod[4];
    const int c = blockIdx.x, bh = blockIdx.y;
    const int g = c / Lc, cs = g * Lc;
    const float *gc = gch + (size_t)bh * NCt;
    auto piece_lo = [&](int p) { return min(NCt, cs + (p * Lc) / m_pieces); };
    int p = 0;
    while (p + 1 < m_pieces && piece_lo(p + 1) <= c) ++p;
    const int lo = piece_lo(p), hi = piece_lo(p + 1);   // the piece's chunks
    // product of the gates of the piece's chunks after c, over the block
    float after = 1.f;
    for (int cc = c + 1 + threadIdx.x; cc < hi; cc += blockDim.x) after *= gc[cc];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) after *= __shfl_xor_sync(0xffffffffu, after, o);
    if ((threadIdx.x & 31) == 0) wprod[threadIdx.x >> 5] = after;
    __syncthreads();
    after = wprod[0] * wprod[1] * wprod[2] * wprod[3];
    if (c == lo && threadIdx.x == 0)   // the piece's gate product
        pgate[(size_t)bh * NR + g * m_pieces + p] = gc[c] * after;
    if (c == cs)   // empty pieces of the segment multiply by 1
        for (int pp = threadIdx.x; pp < m_pieces; pp += blockDim.x)
            if (piece_lo(pp) == piece_lo(pp + 1)) pgate[(size_t)bh * NR + g * m_pieces + pp] = 1.f;
    if (c == 0)   // the record past the pieces (the last segment's prefix) multiplies nothing
        for (int r = npieces + threadIdx.x; r < NR; r += blockDim.x) pgate[(size_t)bh * NR + r] = 1.f;
    const float sc = sqrtf(after);
    const int rows = min(kTile, T - c * kTile);
    const size_t base = ((size_t)bh * T + (size_t)c * kTile) * 32;
    const uint4 *src = reinterpret_cast<const uint4 *>(kc + base);
    uint4 *dst = reinterpret_cast<uint4 *>(kpc + base);
    for (int e = threadIdx.x; e < rows * 4; e += blockDim.x) {
        uint4 u = src[e];
        uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_bf16(__uint_as_float(w[k] << 16) * sc, __uint_as_float(w[k] & 0xFFFF0000u) * sc);
        dst[e] = u;
    }
}

// Exclusive gated prefix of the piece records in place: run = 0; per record r,
// store run, then run = pg_r run + rec_r (the affine maps (g, S) compose as
// (g, S) o (g', S') = (g g', g' S + S')).  Inclusive totals to totals[BH][E].
__global__ void __launch_bounds__(256)
gated_record_scan_kernel(float *__restrict__ rec, const float *__restrict__ pgate, int NR, int64_t E,
                         float *__restrict__ totals) {
    const int64_t e4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e4 >= E / 4) return;
    const int bh = blockIdx.y;
    float4 *p = reinterpret_cast<float4 *>(rec + (size_t)bh * NR * E) + e4;
    const float *pg = pgate + (size_t)bh * NR;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < NR; ++r) {
        const float4 x = p[(size_t)r * (E / 4)];
        const float gr = pg[r];
        p[(size_t)r * (E / 4)] = run;
        run = make_float4(fmaf(gr, run.x, x.x), fmaf(gr, run.y, x.y), fmaf(gr, run.z, x.z),
                          fmaf(gr, run.w, x.w));
    }
    if (totals) reinterpret_cast<float4 *>(totals + (size_t)bh * E)[e4] = run;
}

}  // namespace

bool tc_supported(const FwdShape &s, int cc_major, int cc_minor) {
    return s.dtype == 1 && cc_major == 10 && cc_minor == 3 && s.d == 32 && s.dv == 64 &&
           encoder() != nullptr;
}

std::atomic<int> g_stall_next{0};   // test hook: stall the next segment-state launch

namespace {
// The shape the output kernel sees: nsub sub-heads per head, of width d / nsub,
// or d / 2 when they pair the two halves crosswise (KATA-Sigma_2, nsub = 4).
FwdShape sub_shape(const FwdShape &s, int nsub, bool cross = false) {
    FwdShape ss = s;
    ss.B = s.B * nsub;
    ss.d = cross ? s.d / 2 : s.d / nsub;
    return ss;
}
// Sub-head partials (N and D, fp32) come first in the workspace, rounded to 256
// bytes: with several sub-heads, or with a map's eps terms still to add.
size_t sub_part_floats(const FwdShape &ss, bool partials) {
    return partials ? (((size_t)ss.BH() * ss.T * 65 + 63) & ~(size_t)63) : 0;
}
// The shapes a map's eps terms are added to: Sigma_2 at d = 64 as four crosswise
// sub-heads, Sigma_1 at d = 32 as the full map.
bool sigma_shape_ok(const FwdShape &s0, int nsub, const MapSpec *sigma) {
    return sigma == nullptr || (nsub == 4 && s0.d == 64 && sigma->g == 2) ||
           (nsub == 1 && s0.d == 32 && sigma->g == 1);
}
}  // namespace

namespace {
// Segmentation: G segments of Lc chunks per head, each taken by `span` CTAs of
// the output kernel (one, or a CTA pair) so that span G BH CTAs fill the SMs
// once when BH is small.  The segment sums come from m pieces of each segment,
// one state-kernel CTA per piece, so that the state kernel fills the SMs as
// well.  Records: [BH][NR][E]: nsum m piece sums, plus (without the final
// state) one record past them that receives the last segment's prefix; the
// exclusive scan over them leaves segment g's prefix at record g m.
struct Plan {
    int NCt, G, Lc, m, nsum, NR;
};

Plan plan(const FwdShape &s, int num_sms, bool with_state, int span) {
    Plan p;
    p.NCt = (s.T + kTile - 1) / kTile;
    int G = num_sms / (span * s.BH());
    if (G < 1) G = 1;
    if (G > p.NCt) G = p.NCt;
    p.Lc = (p.NCt + G - 1) / G;
    p.G = (p.NCt + p.Lc - 1) / p.Lc;
    p.nsum = with_state ? p.G : p.G - 1;
    p.m = p.nsum > 0 ? num_sms / (p.nsum * s.BH()) : 1;
    if (p.m < 1) p.m = 1;
    if (p.m > p.Lc) p.m = p.Lc;
    p.NR = p.nsum > 0 ? p.nsum * p.m + (with_state ? 0 : 1) : 0;
    return p;
}

// The CTA-pair output kernel (kata_tc_pair.cu) splits the feature blocks of a
// segment over two SMs.  It is exact, but slower than the one-CTA kernel on
// every measured shape, so it runs only when KATA_TC_OUTPUT=pair is set (and
// without a state export, which the one-CTA kernel writes).
bool use_pair(int nsub, const MapSpec *sigma, bool with_state) {
    if (nsub != 1 || sigma != nullptr || with_state) return false;
    const char *e = getenv("KATA_TC_OUTPUT");
    return e != nullptr && strcmp(e, "pair") == 0;
}
}  // namespace

size_t tc_workspace_bytes(const FwdShape &s0, int num_sms, bool with_state, int nsub,
                          const MapSpec *sigma) {
    const bool cross = sigma != nullptr && nsub == 4;
    const FwdShape s = sub_shape(s0, nsub, cross);
    // piece records (of the key sub-heads: 2 per head when crosswise), plus the
    // final states when the state is exported
    const Plan p = plan(s, num_sms, false, use_pair(nsub, sigma, with_state) ? 2 : 1);
    const size_t recs = (size_t)p.NR + (with_state ? 1 : 0);
    const size_t heads = cross ? (size_t)s0.BH() * 2 : (size_t)s.BH();
    return sizeof(float) * (sub_part_floats(s, nsub > 1 || sigma) + heads * recs * Cfg<32, 64>::E) +
           (sigma ? sigma_workspace_bytes(s0) : 0);
}

int tc_segments(const FwdShape &s, int num_sms, int *seg_tokens) {
    const Plan p = plan(s, num_sms, false, use_pair(1, nullptr, false) ? 2 : 1);
    if (seg_tokens) *seg_tokens = p.Lc * kTile;
    return p.G;
}

cudaError_t tc_forward(const FwdShape &s0, const void *q, const void *k, const void *v,
                       void *out, void *workspace, int num_sms, cudaStream_t stream,
                       const StateOut &so, int nsub, const MapSpec *sigma) {
    using C = Cfg<32, 64>;
    if (!sigma_shape_ok(s0, nsub, sigma)) return cudaErrorInvalidValue;
    const bool cross = sigma != nullptr && nsub == 4, partials = nsub > 1 || sigma;
    const FwdShape s = sub_shape(s0, nsub, cross);
    const bool with_state = so.state != nullptr, pair = use_pair(nsub, sigma, with_state);
    // the state after the last token comes from the output kernel's last segment,
    // so the segmentation is the one without it
    const Plan p = plan(s, num_sms, false, pair ? 2 : 1);
    CUtensorMap mq, mk, mv;
    // q, k: rows of s0.d columns, read s.d at a time; v: one head's rows, shared by its sub-heads
    if (!make_map(mq, q, s0.d, s.T, s0.BH(), s.d) || !make_map(mk, k, s0.d, s.T, s0.BH(), s.d) ||
        !make_map(mv, v, s.dv, s.T, s0.BH()))
        return cudaErrorInvalidValue;
    float *part = partials ? static_cast<float *>(workspace) : nullptr;
    float *seg = static_cast<float *>(workspace) + sub_part_floats(s, partials);
    // crosswise, the segment sums depend on the key half only: 2 per head
    const int state_heads = cross ? s0.BH() * 2 : s.BH(), state_nsub = cross ? 2 : nsub;
    // Segment sums: of every segment but the last (the output kernel carries the
    // last one on chip).  fin: the final states, [state_heads][E] after the records.
    float *fin = with_state ? seg + (size_t)state_heads * p.NR * C::E : nullptr;
    if (p.nsum > 0) {
        cudaFuncSetAttribute(seg_state_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemState);
        {
            TraceScope tr("tc_segment_state", stream);
            seg_state_kernel<32, 64><<<dim3(p.nsum * p.m, state_heads), 352, kSmemState, stream>>>(
                mk, mv, seg, p.NCt, p.Lc, p.m, p.NR, state_nsub, g_stall_next.exchange(0));
        }
        cudaError_t e = scan_exclusive_launch(seg, state_heads, p.NR, C::E, "tc_segment_scan", stream);
        if (e != cudaSuccess) return e;
    }
    if (pair) {
        cudaError_t e = pair_output_launch(mq, mk, mv, out, seg, s.BH(), s.T, p.NCt, p.Lc, p.G, p.m,
                                           p.NR, stream);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    {
        TraceScope tr("tc_segment_output", stream);
        const dim3 grid(p.G, s.BH());
        const OutGate none{nullptr, nullptr, 1};
        if (part == nullptr && fin == nullptr) {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, false, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutput);
            seg_output_kernel<32, 64, false, false><<<grid, 608, kSmemOutput, stream>>>(
                mq, mk, mv, mk, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.m, p.NR, nsub, cross, part, none,
                nullptr);
        } else if (part == nullptr) {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutput);
            seg_output_kernel<32, 64, false, false, true><<<grid, 608, kSmemOutput, stream>>>(
                mq, mk, mv, mk, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.m, p.NR, nsub, cross, part, none,
                fin);
        } else if (fin == nullptr) {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutput);
            seg_output_kernel<32, 64, true, false><<<grid, 608, kSmemOutput, stream>>>(
                mq, mk, mv, mk, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.m, p.NR, nsub, cross, part, none,
                nullptr);
        } else {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, true, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutput);
            seg_output_kernel<32, 64, true, false, true><<<grid, 608, kSmemOutput, stream>>>(
                mq, mk, mv, mk, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.m, p.NR, nsub, cross, part, none,
                fin);
        }
    }
    if (with_state) {   // the full-map state of every key sub-head, in the decode layout
        TraceScope tr("tc_state_export", stream);
        state_export_kernel<32, 64><<<dim3(C::NBLK + 1, state_heads), 128, 0, stream>>>(fin, so.state,
                                                                                          so.z);
    }
    if (sigma) {   // its scratch follows the records (and the final states)
        const size_t off = sub_part_floats(s, partials) +
                           (size_t)state_heads * (p.NR + (with_state ? 1 : 0)) * C::E;
        return sigma_finalize_launch(s0, cross ? SigmaParts::Sub4 : SigmaParts::Sub1, part,
                                     static_cast<float *>(workspace) + off, q, k, v, out, *sigma,
                                     stream, so.eps_totals);
    }
    if (part != nullptr) {
        TraceScope tr("tc_sub_finalize", stream);
        const int64_t rows = (int64_t)s0.BH() * s0.T;
        const int blocks = (int)std::min<int64_t>((rows * 16 + 255) / 256, 152 * 16);
        sub_finalize_kernel<<<blocks, 256, 0, stream>>>(part, (bf16 *)out, rows, s0.T, nsub);
    }
    return cudaGetLastError();
}

namespace {
// GatedKATA workspace: K' and K'' (bf16 [BH][T][32]), then the piece records
// (plus the totals with a state), the cumulative log2 gates [BH][T], the chunk
// gate products [BH][NC] and the piece gate products [BH][NR].
struct GatedWs {
    bf16 *kc, *kpc;
    float *rec, *lam2, *gch, *pgate;
    size_t bytes;
};
GatedWs gated_ws(const FwdShape &s, const Plan &p, bool with_state, void *base) {
    GatedWs w;
    uint8_t *b = static_cast<uint8_t *>(base);
    const size_t nk = (size_t)s.BH() * s.T * 32 * sizeof(bf16);
    const size_t nrec = (size_t)s.BH() * ((size_t)p.NR + (with_state ? 1 : 0)) * Cfg<32, 64>::E;
    w.kc = reinterpret_cast<bf16 *>(b);
    w.kpc = reinterpret_cast<bf16 *>(b + nk);
    w.rec = reinterpret_cast<float *>(b + 2 * nk);
    w.lam2 = w.rec + nrec;
    w.gch = w.lam2 + (size_t)s.BH() * s.T;
    w.pgate = w.gch + (size_t)s.BH() * p.NCt;
    w.bytes = 2 * nk + sizeof(float) * (nrec + (size_t)s.BH() * s.T + (size_t)s.BH() * p.NCt +
                                        (size_t)s.BH() * p.NR);
    return w;
}
}  // namespace

// The final state comes from the output kernel's last segment, so the plan is the
// one without it; the records gain one final record per head.
size_t tc_gated_workspace_bytes(const FwdShape &s, int num_sms, bool with_state) {
    return gated_ws(s, plan(s, num_sms, false, 1), with_state, nullptr).bytes;
}

cudaError_t tc_forward_gated(const FwdShape &s, const void *q, const void *k, const void *v,
                             const float *gamma, void *out, void *workspace, int num_sms,
                             cudaStream_t stream, const StateOut &so, int normalize) {
    using C = Cfg<32, 64>;
    const bool with_state = so.state != nullptr;
    const Plan p = plan(s, num_sms, false, 1);
    const GatedWs w = gated_ws(s, p, with_state, workspace);
    float *fin = with_state ? w.rec + (size_t)s.BH() * p.NR * C::E : nullptr;   // the final records
    CUtensorMap mq, mk, mv, mkc, mkpc;
    if (!make_map(mq, q, s.d, s.T, s.BH()) || !make_map(mk, k, s.d, s.T, s.BH()) ||
        !make_map(mv, v, s.dv, s.T, s.BH()) || !make_map(mkc, w.kc, s.d, s.T, s.BH()) ||
        !make_map(mkpc, w.kpc, s.d, s.T, s.BH()))
        return cudaErrorInvalidValue;
    cudaError_t e = gate_prep_launch(k, gamma, w.kc, w.lam2, w.gch, s.BH(), s.T, s.d, stream);
    if (e != cudaSuccess) return e;
    if (p.nsum > 0) {
        const int summed = std::min(p.NCt, p.nsum * p.Lc);
        {
            TraceScope tr("tc_gated_piece_prep", stream);
            gated_piece_prep_kernel<<<dim3(summed, s.BH()), 128, 0, stream>>>(
                w.kc, w.gch, w.kpc, w.pgate, s.T, p.NCt, p.Lc, p.m, p.nsum * p.m, p.NR);
        }
        cudaFuncSetAttribute(seg_state_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemState);
        {
            TraceScope tr("tc_segment_state", stream);
            seg_state_kernel<32, 64><<<dim3(p.nsum * p.m, s.BH()), 352, kSmemState, stream>>>(
                mkpc, mv, w.rec, p.NCt, p.Lc, p.m, p.NR, 1, g_stall_next.exchange(0));
        }
        {
            TraceScope tr("tc_gated_scan", stream);
            gated_record_scan_kernel<<<dim3((unsigned)((C::E / 4 + 255) / 256), s.BH()), 256, 0, stream>>>(
                w.rec, w.pgate, p.NR, C::E, nullptr);
        }
    }
    {
        TraceScope tr("tc_segment_output_gated", stream);
        const dim3 grid(p.G, s.BH());
        const OutGate ga{w.lam2, w.gch, normalize};
        if (fin == nullptr) {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutputGated);
            seg_output_kernel<32, 64, false, true><<<grid, 608, kSmemOutputGated, stream>>>(
                mq, mk, mv, mkc, (bf16 *)out, w.rec, s.T, p.NCt, p.Lc, p.m, p.NR, 1, 0, nullptr, ga,
                nullptr);
        } else {
            cudaFuncSetAttribute(seg_output_kernel<32, 64, false, true, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutputGated);
            seg_output_kernel<32, 64, false, true, true><<<grid, 608, kSmemOutputGated, stream>>>(
                mq, mk, mv, mkc, (bf16 *)out, w.rec, s.T, p.NCt, p.Lc, p.m, p.NR, 1, 0, nullptr, ga,
                fin);
        }
    }
    if (with_state) {
        TraceScope tr("tc_state_export", stream);
        state_export_kernel<32, 64><<<dim3(C::NBLK + 1, s.BH()), 128, 0, stream>>>(fin, so.state, so.z);
    }
    return cudaGetLastError();
}

namespace {
// KATA-M_4 at d = 64: each 16-wide block u_a of a q or k row becomes a 32-wide
// row [u_a | 0]; psi of the padded row holds psi(u_a) and zeros, so the four
// padded blocks run as full-map d = 32 sub-heads whose N and D add (Sec. 4.1,
// KATA-M_g: <psi(q), psi(k)> = sum_a (q_a . k_a)^2).  One thread per 16-wide block.
__global__ void __launch_bounds__(256)
pad_blocks16_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ xp, int64_t rows) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (row, block)
    if (e >= rows * 4) return;
    const uint4 *src = x + e * 2;   // 16 bf16 = 2 x 16 bytes
    uint4 *dst = xp + e * 4;        // 32 bf16 = 4 x 16 bytes
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    dst[0] = src[0];
    dst[1] = src[1];
    dst[2] = z;
    dst[3] = z;
}
FwdShape padded_m4(const FwdShape &s) {
    FwdShape sp = s;
    sp.d = 128;   // four 32-wide padded blocks per row
    return sp;
}
}  // namespace

size_t tc_m4_workspace_bytes(const FwdShape &s, int num_sms, bool with_state) {
    const size_t np = (size_t)s.BH() * s.T * 128 * sizeof(bf16);
    return 2 * np + tc_workspace_bytes(padded_m4(s), num_sms, with_state, 4);
}

cudaError_t tc_forward_m4(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                          void *workspace, int num_sms, cudaStream_t stream, const StateOut &so) {
    if (s.d != 64) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)s.BH() * s.T;
    const size_t np = (size_t)rows * 128;
    bf16 *qp = static_cast<bf16 *>(workspace), *kp = qp + np;
    {
        TraceScope tr("tc_m4_pad", stream);
        const unsigned blocks = (unsigned)((rows * 4 + 255) / 256);
        pad_blocks16_kernel<<<blocks, 256, 0, stream>>>((const uint4 *)q, (uint4 *)qp, rows);
        pad_blocks16_kernel<<<blocks, 256, 0, stream>>>((const uint4 *)k, (uint4 *)kp, rows);
    }
    return tc_forward(padded_m4(s), qp, kp, v, out, kp + np, num_sms, stream, so, 4);
}

void tc_arm_stall() { g_stall_next.store(1); }

int tc_take_error() {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (h) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    }
    return h;
}

}  // namespace kata
