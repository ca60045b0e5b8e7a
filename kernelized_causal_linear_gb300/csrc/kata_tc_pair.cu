// Output kernel of the d = 32 tensor-core forward, one segment per CTA pair.
//
// The method (KATA paper, Sec. 4.1 Eq. 17-20, App. D.2 Algorithm 1) walks the
// chunks of a segment carrying the running state S = sum psi(k) v^T in fp32.
// For d = 32 that state is 544 features (five 128-feature blocks, the grouped
// layout of kata_tc_common.cuh) x 64 value columns = 320 TMEM columns, which
// leaves one SM no room to keep the lifted queries in TMEM or to double-buffer
// the output accumulator.  Here the two CTAs of a cluster split the features of
// one (segment, head):
//
//   rank 0: state blocks 0-1, and the intra-chunk term P = (Q K^T)^2 .* M,
//           N += P V with its row sums (the intra part of the denominator);
//   rank 1: state blocks 2-4, and the key Gram G = K^T K with the inter part of
//           the denominator q^T G_pre q (psi(q).z = <q q^T, G>_F, Sec. 3.1).
//
// Each rank accumulates a partial numerator sum_b psi_q,b(Q) S_pre,b over its
// blocks (Eq. 18) with the lifted queries as the A operand in TMEM, and its part
// of the denominator.  Numerator and denominator are sums over the two ranks;
// rank 0 finishes query rows 0-63 of every chunk and rank 1 rows 64-127
// (Eq. 20), after each has sent the other's rows of its partial (fp32, 17 KB per
// chunk) into the peer's shared memory with one bulk copy per warp.
//
// Roles (19 warps per CTA):
//   warp 0       TMA: Q, K tiles (one stage), V tiles (two stages)
//   warp 1       output MMAs: rank 0 Q K^T (N = 128), psi_q S_pre, P V;
//                rank 1 Q G_pre, psi_q S_pre
//   warp 2       state MMAs: rank 1 G += K^T K; psi_k^T V into each own block
//   warps 3-6    S_run block -> bf16 S_pre (shared memory), lane quarter w % 4
//   warps 7-10   rank 0: P from Q K^T in TMEM (bf16, written over Q K^T) and
//                its row sums; rank 1: G -> bf16 G_pre and q^T G_pre q; both:
//                the epilogue and the exchange with the peer
//   warps 11-14  psi_q lift into TMEM (token = TMEM lane)
//   warps 15-18  psi_k lift into a shared-memory ring (the state MMA's A)
//
// TMEM (512 columns):
//   rank 0: S_run [0,128) | R [128,256): Q K^T, then P in R[128,192) |
//           Xo0 [256,320) Xo1 [320,384) | psi_q slots [384,448) [448,512)
//   rank 1: S_run [0,192) | G [192,224) | Q G_pre [224,256) | Xo0, Xo1 | psi_q slots
//
// Every wait is bounded (kata_sm100.cuh); an expired wait sets the CTA's abort
// flag, later waits return at once, and the kernel drains its copies and MMAs
// before it frees TMEM and leaves.
#include "kata_tc_common.cuh"

namespace kata {

__device__ int g_pair_error = 0;   // sticky: bounded waits that expired

namespace {

using C32 = Cfg<32, 64>;
constexpr int kKRing = 2;                       // psi_k ring slots (32 KB each)
constexpr int kXRow = 68;                       // floats per exchanged row: 64 numerators, D part, pad
constexpr int kXHalf = 64 * kXRow * 4;          // one 64-row half, 17408 bytes

// Shared-memory layout (offsets from the 1024-aligned base).  Q/K stage s is
// [Q 8 KB | K 8 KB] at s * 16 KB.
constexpr int kQKStage = 2 * C32::QK_TILE;                  // 16 KB
constexpr int kOffQK = 0;                                   // [2][Q | K]
constexpr int kOffV = kOffQK + 2 * kQKStage;                // 32 KB: [2][16 KB]
constexpr int kOffKR = kOffV + 2 * C32::V_TILE;             // 64 KB: [kKRing][32 KB]
constexpr int kOffSP = kOffKR + kKRing * 32768;             // [2][16 KB]
constexpr int kOffG = kOffSP + 2 * 16384;                   // 2 KB
constexpr int kOffXB = kOffG + 2048;                        // receive [2][17 KB]
constexpr int kSmemPair = kOffXB + 2 * kXHalf + 1024;       // + alignment slack

__device__ __forceinline__ void flag_pair_error(int code) { atomicOr(&g_pair_error, code); }

// psi_q of block b for one token into its TMEM lane: 64 columns (16 for block
// 4), four columns (one chunk position, 8 features) at a time.
__device__ __forceinline__ void lift_q_tmem(int b, const PackedRow<32> &r, uint32_t taddr) {
    const int npos = b == 4 ? 4 : 16;
#pragma unroll 1
    for (int pos = 0; pos < npos; ++pos) tmem_st4(taddr + 4 * pos, chunk_words_rt(b, pos, r, kOne2));
}

// psi_q lift role: token t (a lane of this warp's TMEM quarter) lifts its query
// row into the psi_q slot of every own block, chunk after chunk.  Out of line so
// that its registers are allocated apart from the other roles.
__device__ __noinline__ void psi_q_role(const uint8_t *qk, uint32_t slots, int t, int b0, int NB,
                                        int nch, uint64_t *qk_full, uint64_t *qk_empty,
                                        uint64_t *qslot_full, uint64_t *qslot_empty,
                                        volatile int *abort) {
    const Sync sy{abort};
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
        const int qs = i & 1;
        ok = __all_sync(0xffffffffu, sy.wait(&qk_full[qs], i >> 1));
        if (!ok) break;
        PackedRow<32> r;
        tile_row_packed<32>(qk + qs * kQKStage, t, r);
        __syncwarp();
        if (elect_lane0()) mbar_arrive(&qk_empty[qs]);
        for (int lb = 0; lb < NB && ok; ++lb) {
            const int gb = i * NB + lb, sl = gb & 1, use = gb >> 1;
            if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&qslot_empty[sl], use - 1));
            if (!ok) break;
            tc_fence_after();
            lift_q_tmem(b0 + lb, r, slots + sl * 64);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&qslot_full[sl]);
        }
    }
}

// psi_k lift role: token t lifts its key row into the shared-memory ring slot
// of every own block (the state MMA's MN-major A operand).
__device__ __noinline__ void psi_k_role(const uint8_t *qk, uint8_t *kring, int t, int b0, int NB,
                                        int nch, uint64_t *qk_full, uint64_t *qk_empty,
                                        uint64_t *kslot_full, uint64_t *kslot_empty, int kring_n,
                                        volatile int *abort) {
    const Sync sy{abort};
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
        const int qs = i & 1;
        ok = __all_sync(0xffffffffu, sy.wait(&qk_full[qs], i >> 1));
        if (!ok) break;
        PackedRow<32> r;
        tile_row_packed<32>(qk + qs * kQKStage + C32::QK_TILE, t, r);
        __syncwarp();
        if (elect_lane0()) mbar_arrive(&qk_empty[qs]);
        for (int lb = 0; lb < NB && ok; ++lb) {
            const int gb = i * NB + lb, sl = gb % kring_n, use = gb / kring_n;
            if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&kslot_empty[sl], use - 1));
            if (!ok) break;
            lift_block_rt(b0 + lb, r, kTwo2, block_row_rt(kring + sl * 32768, t));
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&kslot_full[sl]);
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(608, 1)
pair_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, bf16 *__restrict__ out,
                   const float *__restrict__ seg, int T, int NCt, int Lc, int m_pieces, int NR) {
    constexpr int D = 32, DV = 64;
    constexpr int kLiftWarps = 4, kTmemWarps = 4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *qk = sm + kOffQK, *tv = sm + kOffV, *kring = sm + kOffKR;
    uint8_t *spre = sm + kOffSP, *gram = sm + kOffG;
    float *xbuf = reinterpret_cast<float *>(sm + kOffXB);   // [2][64][kXRow]

    __shared__ __align__(8) uint64_t qk_full[2], qk_empty[2], v_full[2], v_empty[2], kslot_full[kKRing],
        kslot_empty[kKRing], qslot_full[2], qslot_empty[2], sp_full[2], sp_empty[2], sread[3],
        sdone[3], xs_full, p_full, pv_done, xo_full[2], xo_empty[2], gram_done, gread, gpre_full,
        qg_done, qg_empty, xfull[2], xempty[2], fin[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int g = blockIdx.x >> 1, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;
    const int NB = rank == 0 ? 2 : 3;            // own state blocks
    const int b0 = rank == 0 ? 0 : 2;            // first own block
    const Sync sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qk_full[i], 1);
            // readers of the Q/K tiles: the output MMA thread and both lifts; on rank 1
            // also the state MMA thread (Gram) and the P warps (q rows)
            mbar_init(&qk_empty[i], rank == 0 ? 1 + 2 * kLiftWarps : 2 + 2 * kLiftWarps + kTmemWarps);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 2);
            mbar_init(&qslot_full[i], kLiftWarps);
            mbar_init(&qslot_empty[i], 1);
            mbar_init(&sp_full[i], kTmemWarps);
            mbar_init(&sp_empty[i], 1);
            mbar_init(&xo_full[i], 1);
            mbar_init(&xo_empty[i], kTmemWarps);
            mbar_init(&xfull[i], 64);       // the peer's 64 sending threads
            mbar_init(&xempty[i], 64);      // the peer's 64 receiving threads
            mbar_init(&fin[i], 1);
        }
        for (int i = 0; i < kKRing; ++i) {
            mbar_init(&kslot_full[i], kLiftWarps);
            mbar_init(&kslot_empty[i], 1);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(&sread[b], kTmemWarps);
            mbar_init(&sdone[b], 1);
        }
        mbar_init(&xs_full, 1);
        mbar_init(&p_full, kTmemWarps);
        mbar_init(&pv_done, 1);
        mbar_init(&gram_done, 1);
        mbar_init(&gread, kTmemWarps);
        mbar_init(&gpre_full, kTmemWarps);
        mbar_init(&qg_done, 1);
        mbar_init(&qg_empty, kTmemWarps);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the peer's barriers exist before any remote arrive or copy
    tc_fence_after();
    const uint32_t tS = tmem_base;
    const uint32_t tR = tmem_base + 128;                          // rank 0
    const uint32_t tG = tmem_base + 192, tQG = tmem_base + 224;   // rank 1
    const uint32_t tXo = tmem_base + 256, tPsi = tmem_base + 384;
    // the segment's exclusive prefix: the scan's record at its first piece (none for g == 0)
    const float *rec = g > 0 ? seg + ((size_t)bh * NR + (size_t)g * m_pieces) * C32::E : nullptr;

    int n_qk0 = 0, n_qk1 = 0, n_v0 = 0, n_v1 = 0;   // TMA loads issued (teardown drain)

    if (warp == 0) {
        // ================= TMA producer
        if (elect_lane0()) {
            for (int i = 0; i < nch; ++i) {
                const int t0 = (c0 + i) * kTile;
                const int st = i & 1, use = i >> 1;
                if (use >= 1 && !sy.wait(&qk_empty[st], use - 1)) break;
                mbar_arrive_expect_tx(&qk_full[st], kQKStage);
                tma_load_3d(qk + st * kQKStage, &tm_q, 0, t0, bh, &qk_full[st]);
                tma_load_3d(qk + st * kQKStage + C32::QK_TILE, &tm_k, 0, t0, bh, &qk_full[st]);
                if (st == 0) ++n_qk0; else ++n_qk1;
                if (use >= 1 && !sy.wait(&v_empty[st], use - 1)) break;
                mbar_arrive_expect_tx(&v_full[st], C32::V_TILE);
                tma_load_3d(tv + st * C32::V_TILE, &tm_v, 0, t0, bh, &v_full[st]);
                if (st == 0) ++n_v0; else ++n_v1;
                if (i + 1 < nch) {   // warm L2 with the next chunk's tiles
                    tma_prefetch_3d(&tm_q, 0, t0 + kTile, bh);
                    tma_prefetch_3d(&tm_k, 0, t0 + kTile, bh);
                    tma_prefetch_3d(&tm_v, 0, t0 + kTile, bh);
                }
            }
        }
    } else if (warp == 1) {
        // ================= output MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
            constexpr uint32_t kIdQG = idesc_bf16(128, D, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
            const uint64_t dQ0 = smem_desc(smem_u32(qk), 16, 512, kSw64);                 // K-major A
            const uint64_t dKb0 = smem_desc(smem_u32(qk + C32::QK_TILE), 16, 512, kSw64); // K-major B
            const uint64_t dGr = smem_desc(smem_u32(gram), 16, 512, kSw64);     // K-major B
            const uint64_t dSp = smem_desc(smem_u32(spre), 16384, 1024, kSw128); // MN-major B
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);  // MN-major B
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int xs = i & 1;
                ok = sy.wait(&qk_full[xs], i >> 1);
                if (!ok) break;
                const uint64_t dQ = desc_add(dQ0, xs * kQKStage), dKb = desc_add(dKb0, xs * kQKStage);
                if (rank == 0) {
                    // R is free once P V of the previous chunk has read P
                    ok = i == 0 || sy.wait(&pv_done, i - 1);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tR, desc_add(dQ, ks * 32), desc_add(dKb, ks * 32), kIdQK, ks > 0);
                    mma_commit(&xs_full);
                } else {
                    ok = sy.wait(&gpre_full, i) && (i == 0 || sy.wait(&qg_empty, i - 1));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tQG, desc_add(dQ, ks * 32), desc_add(dGr, ks * 32), kIdQG, ks > 0);
                    mma_commit(&qg_done);
                }
                mma_commit(&qk_empty[xs]);
                ok = i < 2 || sy.wait(&xo_empty[xs], (i >> 1) - 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t xo = tXo + xs * 64;
#pragma unroll 1
                for (int lb = 0; lb < NB; ++lb) {
                    const int gb = i * NB + lb, sl = gb & 1;
                    ok = sy.wait(&qslot_full[sl], gb >> 1) && sy.wait(&sp_full[sl], gb >> 1);
                    if (!ok) break;
                    tc_fence_after();
                    // Xo (+)= psi_q S_pre for this block; A = the lifted queries in TMEM
                    const uint32_t a0 = tPsi + sl * 64;
                    const uint64_t bs = desc_add(dSp, sl * 16384);
                    if (b0 + lb == 4) {   // block 4: 32 features, 2 K steps
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma_ts(xo, a0 + ks * 8, desc_add(bs, ks * 2048), kIdPV, 1u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ts(xo, a0 + ks * 8, desc_add(bs, ks * 2048), kIdPV,
                                   (lb > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&qslot_empty[sl]);
                    mma_commit(&sp_empty[sl]);
                }
                if (!ok) break;
                if (rank == 0) {   // Xo += P V (A = P in TMEM)
                    ok = sy.wait(&p_full, i) && sy.wait(&v_full[xs], i >> 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t bv = desc_add(dV0, xs * C32::V_TILE);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ts(xo, tR + ks * 8, desc_add(bv, ks * 2048), kIdPV, 1u);
                    mma_commit(&pv_done);
                }
                mma_commit(&xo_full[xs]);
                mma_commit(&v_empty[xs]);
            }
            mma_commit(&fin[0]);
            mbar_wait(&fin[0], 0);   // every MMA of this thread has completed
        }
    } else if (warp == 2) {
        // ================= state MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            const uint64_t dKg0 = smem_desc(smem_u32(qk + C32::QK_TILE), 8192, 512, kSw64); // MN-major (Gram)
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);   // MN-major B
            const uint64_t dLk = smem_desc(smem_u32(kring), 16384, 1024, kSw128); // MN-major A
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                if (rank == 1) {   // G += K^T K once G_pre of this chunk has been read out
                    ok = sy.wait(&qk_full[st], i >> 1) && sy.wait(&gread, i);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        const uint64_t a = desc_add(dKg0, st * kQKStage + ks * 1024);
                        mma_ss(tG, a, a, kIdGram, 1u);
                    }
                    mma_commit(&gram_done);
                    mma_commit(&qk_empty[st]);
                }
                ok = sy.wait(&v_full[st], i >> 1);
                if (!ok) break;
#pragma unroll 1
                for (int lb = 0; lb < NB; ++lb) {
                    const int gb = i * NB + lb, ks_ = gb % kKRing;
                    // S_run block += psi_k^T V once the convert warps have read it
                    ok = sy.wait(&kslot_full[ks_], gb / kKRing) && sy.wait(&sread[lb], i);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = desc_add(dLk, ks_ * 32768), bv = desc_add(dV0, st * C32::V_TILE);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + lb * DV, desc_add(a0, ks * 2048), desc_add(bv, ks * 2048), kIdState, 1u);
                    mma_commit(&kslot_empty[ks_]);
                    mma_commit(&sdone[lb]);
                }
                if (!ok) break;
                mma_commit(&v_empty[st]);
            }
            mma_commit(&fin[1]);
            mbar_wait(&fin[1], 0);
        }
    } else if (warp < 7) {
        // ================= convert warps: S_run block -> bf16 S_pre slot
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        // initial state: the segment's exclusive prefix of the own blocks (zero for g == 0)
        for (int lb = 0; lb < NB; ++lb) {
            const int b = b0 + lb;
#pragma unroll
            for (int c = 0; c < DV; c += 8) {
                uint32_t v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = rec ? __float_as_uint(rec[(size_t)(b * 128 + row) * DV + c + e]) : 0u;
                tmem_st8(tS + lsel + lb * DV + c, v);
            }
        }
        tmem_st_wait();
        tc_fence_before();
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
#pragma unroll 1
            for (int lb = 0; lb < NB; ++lb) {
                const int gb = i * NB + lb, sl = gb & 1, use = gb >> 1;
                bool w = (use == 0 || sy.wait(&sp_empty[sl], use - 1)) &&
                         (i == 0 || sy.wait(&sdone[lb], i - 1));
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                tc_fence_after();
                const bool live = quarter * 32 < C32::NF - (b0 + lb) * 128;   // real feature rows
                uint32_t va[32], vb[32];
                if (live) {
                    tmem_ld32(tS + lsel + lb * DV, va);
                    tmem_ld32(tS + lsel + lb * DV + 32, vb);
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&sread[lb]);   // S_run block may now be updated
                if (live) {
                    const uint32_t srow = smem_u32(spre + sl * 16384 + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
                    for (int ch = 0; ch < DV / 8; ++ch) {
                        const uint32_t *x = ch < 4 ? va + 8 * ch : vb + 8 * (ch - 4);
                        st_shared_v4(srow + ((ch ^ (row & 7)) << 4),
                                     pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                     pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                     pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                     pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&sp_full[sl]);
            }
        }
    } else if (warp < 11) {
        // ================= P / Gram / epilogue warps (lane quarter w % 4)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        const bool own_rows = (quarter >> 1) == (int)rank;   // rank 0 finishes rows 0-63
        const int hrow = row & 63;                           // row within the 64-row half

        // G_pre -> bf16 [D][D] K-major, 64-byte swizzle (quarter 0: G rows i = lane)
        auto gram_store = [&](const float (&gv)[D]) {
#pragma unroll
            for (int ch = 0; ch < D / 8; ++ch) {
                uint4 u;
                u.x = pack_bf16(gv[8 * ch + 0], gv[8 * ch + 1]);
                u.y = pack_bf16(gv[8 * ch + 2], gv[8 * ch + 3]);
                u.z = pack_bf16(gv[8 * ch + 4], gv[8 * ch + 5]);
                u.w = pack_bf16(gv[8 * ch + 6], gv[8 * ch + 7]);
                *reinterpret_cast<uint4 *>(gram + (lane >> 3) * 512 + (lane & 7) * 64 +
                                           ((ch ^ ((lane >> 1) & 3)) << 4)) = u;
            }
        };

        // rank 0: P of chunk i from Q K^T (R), written over its first 64 columns
        // 16 keys at a time: keys 16j .. 16j + 15 (columns 16j ..) give P words
        // 8j .. 8j + 7, stored at columns 8j .., which have been read by then;
        // returns this row's intra denominator in dsum
        auto build_p = [&](int i, float &dsum) -> bool {
            bool w = __all_sync(0xffffffffu, sy.wait(&xs_full, i));
            if (!w) return false;
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                uint32_t v[16], pw[8];
                tmem_ld16(tR + lsel + 16 * j, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s = 16 * j + 2 * e;
                    const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                    const float w0 = s <= row ? x0 * x0 : 0.f;
                    const float w1 = s + 1 <= row ? x1 * x1 : 0.f;
                    dsum += w0;
                    dsum += w1;
                    pw[e] = pack_bf16(w0, w1);
                }
                tmem_st8(tR + lsel + 8 * j, pw);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&p_full);
            return true;
        };

        // rank 1: G_pre of chunk i (G after chunk i - 1) into shared memory, then
        // this row's inter denominator q^T G_pre q from Q G_pre
        auto gram_and_dinter = [&](int i, float &dsum) -> bool {
            if (i > 0) {
                bool w = __all_sync(0xffffffffu, sy.wait(&gram_done, i - 1) && sy.wait(&qg_done, i - 1));
                if (!w) return false;
                tc_fence_after();
                float gv[D];
                if (quarter == 0) {
#pragma unroll
                    for (int c = 0; c < D; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tG + lsel + c, v);
#pragma unroll
                        for (int e = 0; e < 16; ++e) gv[c + e] = __uint_as_float(v[e]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&gread);   // G may take chunk i's update
                if (quarter == 0) gram_store(gv);
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&gpre_full);
            }
            // Q G_pre of this chunk is done (so its Q tile has landed); the q row
            // is read and used before the tile is released
            bool w = __all_sync(0xffffffffu, sy.wait(&qk_full[i & 1], i >> 1) && sy.wait(&qg_done, i));
            if (!w) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tQG + lsel, v);
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&qg_empty);
            PackedRow<D> r;
            tile_row_packed<D>(qk + (i & 1) * kQKStage, row, r);
#pragma unroll
            for (int m = 0; m < D / 2; ++m) {
                dsum = fmaf(__uint_as_float(v[2 * m]), __uint_as_float(r.w[m] << 16), dsum);
                dsum = fmaf(__uint_as_float(v[2 * m + 1]), __uint_as_float(r.w[m] & 0xFFFF0000u), dsum);
            }
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&qk_empty[i & 1]);
            return true;
        };

        // chunk i's numerator rows: own rows get the peer's partial and are
        // written out; the peer's rows are sent with this rank's denominator part
        auto epilogue = [&](int i, float dpart) -> bool {
            const int xs = i & 1, use = i >> 1;
            bool w = __all_sync(0xffffffffu, sy.wait(&xo_full[xs], use));
            if (!w) return false;
            tc_fence_after();
            const uint32_t xo = tXo + xs * 64 + lsel;
            float *myrow = xbuf + ((size_t)xs * 64 + hrow) * kXRow;
            if (!own_rows) {
                // the peer's rows: [numerators | D part] straight into the peer's
                // receive slot, then one release arrive per thread on its barrier
                w = __all_sync(0xffffffffu, use == 0 || mbar_wait_cluster(&xempty[xs], (use - 1) & 1));
                if (!w) {
                    abort_flag = 1;
                    return false;
                }
                const uint32_t dst = mapa(smem_u32(myrow), peer);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tmem_ld32(xo + 32 * h, v);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_cluster_v4(dst + 128 * h + 16 * c, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&xo_empty[xs]);
                st_cluster_v4(dst + 4 * DV, __float_as_uint(dpart), 0u, 0u, 0u);
                mbar_arrive_cluster(mapa(smem_u32(&xfull[xs]), peer));
                return true;
            }
            // own rows: the peer's partial arrives in xbuf
            w = __all_sync(0xffffffffu, mbar_wait_cluster(&xfull[xs], use & 1));
            if (!w) {
                abort_flag = 1;
                return false;
            }
            const float den = dpart + myrow[DV];
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const int t = (c0 + i) * kTile + row;
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * T + (t < T ? t : 0)) * DV);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
                tmem_ld32(xo + 32 * h, v);
#pragma unroll
                for (int c = 0; c < 4; ++c) {   // 8 output columns at a time
                    const float4 p0 = *reinterpret_cast<const float4 *>(myrow + 32 * h + 8 * c);
                    const float4 p1 = *reinterpret_cast<const float4 *>(myrow + 32 * h + 8 * c + 4);
                    const uint32_t *x = v + 8 * c;
                    const uint4 o = make_uint4(
                        pack_bf16((__uint_as_float(x[0]) + p0.x) * inv, (__uint_as_float(x[1]) + p0.y) * inv),
                        pack_bf16((__uint_as_float(x[2]) + p0.z) * inv, (__uint_as_float(x[3]) + p0.w) * inv),
                        pack_bf16((__uint_as_float(x[4]) + p1.x) * inv, (__uint_as_float(x[5]) + p1.y) * inv),
                        pack_bf16((__uint_as_float(x[6]) + p1.z) * inv, (__uint_as_float(x[7]) + p1.w) * inv));
                    if (t < T) dst[4 * h + c] = o;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&xo_empty[xs]);
            mbar_arrive_cluster(mapa(smem_u32(&xempty[xs]), peer));   // the slot may take the peer's next rows
            return true;
        };

        if (rank == 1) {   // G and G_pre of chunk 0: the segment prefix's Gram (zero for g == 0)
            float gv[D];
            const float *gp = rec ? rec + (size_t)C32::NBLK * 128 * DV + (size_t)lane * D : nullptr;
#pragma unroll
            for (int e = 0; e < D; ++e) gv[e] = gp ? gp[e] : 0.f;
            if (quarter == 0) {
#pragma unroll
                for (int c = 0; c < D; c += 8) {
                    uint32_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(gv[c + e]);
                    tmem_st8(tG + lsel + c, v);
                }
                tmem_st_wait();
                gram_store(gv);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) {
                mbar_arrive(&gread);
                mbar_arrive(&gpre_full);
            }
        }

        bool ok = true;
        float dprev = 0.f;
        for (int i = 0; i <= nch && ok; ++i) {   // chunk i's denominator part, chunk i-1's output
            float dsum = 0.f;
            if (i < nch) {
                if (rank == 0) {
                    ok = build_p(i, dsum);
                } else {
                    ok = gram_and_dinter(i, dsum);
                }
                if (!ok) break;
            }
            if (i > 0) ok = epilogue(i - 1, dprev);
            dprev = dsum;
        }
        if (!ok) abort_flag = 1;
    } else if (warp < 15) {
        // ================= psi_q lift into TMEM: token = lane of this warp's quarter
        const int quarter = warp & 3;
        psi_q_role(qk, tPsi + ((uint32_t)(quarter * 32) << 16), quarter * 32 + lane, b0, NB, nch,
                   qk_full, qk_empty, qslot_full, qslot_empty, &abort_flag);
    } else {
        // ================= psi_k lift into the shared-memory ring: token t
        psi_k_role(qk, kring, (warp - 15) * 32 + lane, b0, NB, nch, qk_full, qk_empty, kslot_full,
                   kslot_empty, kKRing, &abort_flag);
    }

    // ================= teardown
    // TMA loads still in flight after an abort land before the CTA leaves;
    // remote stores and arrives are complete once every thread of both CTAs
    // has passed the cluster barrier.
    if (warp == 0 && elect_lane0()) {
        if (n_qk0 > 0) mbar_wait(&qk_full[0], (n_qk0 - 1) & 1);
        if (n_qk1 > 0) mbar_wait(&qk_full[1], (n_qk1 - 1) & 1);
        if (n_v0 > 0) mbar_wait(&v_full[0], (n_v0 - 1) & 1);
        if (n_v1 > 0) mbar_wait(&v_full[1], (n_v1 - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (threadIdx.x == 0 && abort_flag) flag_pair_error(4);
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace

size_t pair_smem_bytes() { return kSmemPair; }

cudaError_t pair_output_launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               void *out, const float *seg, int BH, int T, int NCt, int Lc, int G,
                               int m_pieces, int NR, cudaStream_t stream) {
    cudaFuncSetAttribute(pair_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPair);
    TraceScope tr("tc_pair_output", stream);
    pair_output_kernel<<<dim3(2 * G, BH), 608, kSmemPair, stream>>>(
        mq, mk, mv, (bf16 *)out, seg, T, NCt, Lc, m_pieces, NR);
    return cudaGetLastError();
}

int pair_take_error() {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_pair_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (h) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_pair_error, &zero, sizeof(int));
    }
    return h;
}

}  // namespace kata
