// tcgen05 tensor-core path of the KATA chunked forward at d = 64 (bf16, sm_103a).
//
// At d = 64 the lift has n = 2080 coordinates: 17 blocks of 128 features in the
// grouped layout below, whose fp32 state (17 x 64 TMEM columns) does not fit in
// the 512 TMEM columns of one SM.  The state is therefore split by feature
// blocks over four CTAs per head ("feature groups"):
//   group 0: blocks 0-1, plus the intra-chunk term P = (Q K^T)^2 .* M, P V, and
//            the normaliser (Gram G = K^T K; q^T G_pre q)      [Eq. 18, 19]
//   groups 1-3: blocks 2-6, 7-11, 12-16
// Every group walks all chunks of its head with its blocks' running state in
// TMEM ([KATA] Sec. 4.1 Eq. 17), adds psi_q(Q) S_pre over its blocks into an
// output accumulator (Eq. 18), and writes that partial numerator per token in
// fp32; group 0 also writes the denominator.  finalize_kernel then forms
// O = (N_0 + N_1 + N_2 + N_3) / D (Eq. 20), in that fixed order.
//
// The kernel keeps one segment per head: it is used when the four groups of all
// heads fill the GPU (4 * B * H >= SM count).  Structure per CTA as in the d = 32
// output kernel: warp 0 TMA, warps 1-2 MMA issue (output / state), warps 3-6
// convert S_run -> bf16 S_pre, warps 7-10 P and the epilogue, warps 11-18 lift
// the group's blocks.
#include "kata_tc_common.cuh"

namespace kata {

__device__ int g_tc64_error = 0;   // sticky: bounded waits that expired

namespace {

__device__ __forceinline__ void flag_error64(int code) { atomicOr(&g_tc64_error, code); }

// Bounded barrier wait as Sync, with the slow path out of line: one copy of the
// spin serves every wait site, which keeps this kernel's code 15% smaller (its
// warps fetch from eight roles' code at once).
__device__ __noinline__ bool wait_slow64(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (*abort) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort = 1;
    return false;
}
struct Sync64 {
    volatile int *abort;
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t n) const {
        const uint32_t parity = n & 1u;
        if (mbar_try_wait(bar, parity)) return true;   // fast path: a completed phase
        return wait_slow64(bar, parity, abort);
    }
};

// ---- grouped feature layout at d = 64 (17 blocks of 128 slots, 2080 real)
// Eight groups of eight coordinates.  Blocks 0-13 hold the 28 cross-group
// 8 x 8 rectangles (X, Y), X < Y, in lexicographic order, one per 64-feature
// atom column (rectangle 2b and 2b + 1 in block b); blocks 14-16 hold the eight
// within-group triangles as one run of 40 chunks (5 per group): chunks 0-15,
// 16-31 and 32-39, the last block using its first atom column only.  Rows,
// triangles and the key factor 2 are as at d = 32.
constexpr int kBlocks64 = 17;

// Rectangle r (0..27) -> groups (X, Y), X < Y, lexicographic.
__device__ __forceinline__ void rect_pair64(int r, int &X, int &Y) {
    X = 0;
    int n = 7;   // rectangles whose first group is X: 7 - X
    while (r >= n) {
        r -= n;
        ++X;
        --n;
    }
    Y = X + 1 + r;
}

// Lift block b (0..16) of the d = 64 layout for one token whose row (bf16
// pairs, group g = columns 4g .. 4g + 3) sits in TMEM at trow.  The groups a
// block needs are chosen at run time, so one copy of the code serves every
// block and every feature group (per-group compile-time copies were slower,
// through instruction fetch); fetching a group from TMEM at a warp-uniform
// column costs one load, where selecting it from registers took 28 ALU selects.
__device__ __forceinline__ void lift_block64(int b, uint32_t trow, uint32_t f, const BlockRowRt &br) {
    if (b < 14) {
#pragma unroll 1
        for (int rr = 0; rr < 2; ++rr) {
            int X, Y;
            rect_pair64(2 * b + rr, X, Y);
            Group8 gx, gy;
            tmem_ld4x2(trow + 4 * X, trow + 4 * Y, gx.w, gy.w);
            lift_rect_rt(gx, gy, f, br, 8 * rr);
        }
    } else {
        const int c0 = 16 * (b - 14), c1 = min(40, c0 + 16);
#pragma unroll 1
        for (int g = c0 / 5; g * 5 < c1; ++g) {
            Group8 gg;
            tmem_ld4(trow + 4 * g, gg.w);
            lift_tri_rt(gg, f, br, max(0, c0 - 5 * g), min(5, c1 - 5 * g), 5 * g - c0);
        }
    }
}

// Blocks of feature group grp: [first, first + count).
__device__ __forceinline__ int group_first(int grp) { return grp == 0 ? 0 : 2 + 5 * (grp - 1); }
__device__ __forceinline__ int group_count(int grp) { return grp == 0 ? 2 : 5; }
// Real features of block b (the last block holds 64).
__device__ __forceinline__ int block_feats(int b) { return b == kBlocks64 - 1 ? 64 : 128; }

// Final-state record of one head (state export): S in the grouped layout
// [17 blocks][128 features][64] fp32, then G = sum k k^T [64][64] fp32.
constexpr int kRec64 = kBlocks64 * 128 * 64 + 64 * 64;

// Coordinates (i, j), i <= j, of feature p (0..127) of block b of the d = 64
// grouped layout; false for a pad slot.
__device__ __forceinline__ bool grouped_slot_pair64(int b, int p, int &i, int &j) {
    const int pos = p >> 3, k = (p & 7) >> 1, hf = p & 1;
    if (b < 14) {   // rectangle 2b + pos / 8, row pos % 8
        int X, Y;
        rect_pair64(2 * b + (pos >> 3), X, Y);
        i = 8 * X + (pos & 7);
        j = 8 * Y + 2 * k + hf;
        return true;
    }
    const int c = 16 * (b - 14) + pos;   // chunk of the run of 40 triangle chunks
    if (c >= 40) return false;
    const int g = c / 5;
    int I = 0, w = 4 * (c % 5) + k;   // pair w of the triangle: row I has (9 - I) / 2 pairs
    while (w >= (9 - I) / 2) {
        w -= (9 - I) / 2;
        ++I;
    }
    const int J = I + 2 * w + hf;
    if (J >= 8) return false;
    i = 8 * g + I;
    j = 8 * g + J;
    return true;
}

// Lift role (out of line: its registers are allocated apart from the other
// roles).  Token t = 32 * (warp % 4) + lane: its row is parked in TMEM lane t
// (the warp's lane quarter), columns trow .. trow + 31, once per chunk.
__device__ __noinline__ void wide_lift_role(const uint8_t *tile, uint8_t *ring, int t, bool key,
                                            uint32_t trow, int b_first, int nb, int nch,
                                            uint64_t *chunk_full,
                                            uint64_t *qk_empty, uint64_t *block_ready,
                                            uint64_t *block_empty, volatile int *abort) {
    const Sync64 sy{abort};
    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
        ok = __all_sync(0xffffffffu, sy.wait(&chunk_full[i & 1], i >> 1));
        if (!ok) break;
        {
            PackedRow<64> r;
            tile_row_packed<64>(tile, t, r);
            tmem_st32(trow, r.w);   // the previous chunk's loads of these columns have completed
            tmem_st_wait();
        }
        __syncwarp();
        if (elect_lane0()) mbar_arrive(qk_empty);
        for (int b = 0; b < nb && ok; ++b) {
            const int gb = i * nb + b, ls = gb & 1, use = gb >> 1;
            if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&block_empty[ls], use - 1));
            if (!ok) break;
            lift_block64(b_first + b, trow, key ? kTwo2 : kOne2, block_row_rt(ring + ls * 65536, t));
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&block_ready[ls]);
        }
    }
}

// ================================================================= output kernel
// Grid (4 feature groups, B*H), 608 threads.  TMEM: S_run [0, 64 * nb) | (group 0:
// G [128,192) | Q G_pre [192,256) | Q K^T [256,384), P of key quarter q written
// over the first 16 columns of its 32) | output accumulator [384,448) | the lift
// warps' q and k rows [448,480) [480,512).  Shared memory: Q, K tiles (16 KB
// each, 128-byte swizzle), V tiles [2][16 KB], lift ring [2][psi_q 32 KB |
// psi_k 32 KB], and [2][16 KB] for S_pre: two blocks in groups 1-3 (the convert
// of block b + 1 overlaps the MMAs of block b); in group 0 one block, G_pre bf16
// [64][64] (8 KB) and the epilogue staging (8 KB).
//
// Group 0 computes Q K^T of a chunk with one N = 128 MMA; the P warps turn
// each 32-key quarter into P in place and release it (p_full[q]) for its P V
// MMA, so no quarter waits on a Q K^T round trip.
//
// Epilogue.  In groups 1-3 only the lift warps read the Q and K tiles, once per
// chunk, so from then until the next chunk's TMA load the 32 KB of the two
// tiles stage the partial numerators: fp32 [128][64] as four warp quarters of
// two 128-byte-swizzled [32 x 32] boxes, written to memory by TMA stores (whole
// lines, and no load/store-unit work while the lift runs).  The TMA load of
// chunk i + 2 waits for the stores of chunk i to have read the staging
// (stage_free).  In group 0, whose tiles feed its MMAs through the chunk, the
// convert warps (two blocks a chunk leave them idle most of the time) store the
// rows through an 8 KB staging area as [32 x 16] boxes, 64-byte swizzled.
constexpr int kSmemWide = 2 * 16384 + 2 * 16384 + 2 * 65536 + 2 * 16384 + 1024;

__global__ void __launch_bounds__(608, 1)
wide_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_part,
                   const __grid_constant__ CUtensorMap tm_part16, float *__restrict__ dden,
                   float *__restrict__ srec, int T, int NCt) {
    constexpr int D = 64, DV = 64;
    constexpr int kQK = kTile * D * 2, kV = kTile * DV * 2;
    constexpr int kLiftWarps = 8, kTmemWarps = 4;
    constexpr int kWarpP = 7, kWarpLift = 11;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tq = sm;
    uint8_t *tk = sm + kQK;
    uint8_t *tv = sm + 2 * kQK;                         // [2][16 KB]
    uint8_t *lring = tv + 2 * kV;                       // [2][psi_q 32 KB | psi_k 32 KB]
    uint8_t *spre = lring + 2 * 65536;                  // S_pre blocks [2][16 KB]
    uint8_t *gram = spre + 16384;                       // group 0: G_pre bf16, K-major, 8 KB
    uint8_t *stage = tq;                                // groups 1-3: epilogue staging (Q, K tiles)
    uint8_t *gstage = gram + 8192;                      // group 0: epilogue staging, 4 x 2 KB
    __shared__ __align__(8) uint64_t chunk_full[2], qk_empty, v_empty[2], xs_full, p_full[4],
        pv_done, block_ready[2], block_empty[2], spre_empty[2], state_done[5], o_full, o_empty,
        gram_done, qg_done, fin_bar[2], stage_free;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int grp = blockIdx.x, bh = blockIdx.y;
    const bool intra = grp == 0;
    const int b_first = group_first(grp), nb = group_count(grp);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = NCt;
    const Sync64 sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // Q/K tiles: read by the lift warps, and in group 0 by both MMA threads
        // and the P warps
        mbar_init(&qk_empty, kLiftWarps + (intra ? 2 + kTmemWarps : 0));
        for (int i = 0; i < 2; ++i) {
            mbar_init(&chunk_full[i], 1 + (intra ? kTmemWarps : 0));   // TMA (+ G_pre in group 0)
            mbar_init(&v_empty[i], intra ? 2 : 1);
            mbar_init(&block_ready[i], kLiftWarps + kTmemWarps);
            mbar_init(&block_empty[i], 2);
            mbar_init(&fin_bar[i], 1);
            mbar_init(&spre_empty[i], 1);
        }
        mbar_init(&xs_full, 1);
        for (int q = 0; q < 4; ++q) mbar_init(&p_full[q], kTmemWarps);
        mbar_init(&pv_done, 1);
        mbar_init(&stage_free, kTmemWarps);
        for (int b = 0; b < 5; ++b) mbar_init(&state_done[b], 1);
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
    const uint32_t tS = tmem_base, tG = tmem_base + 128, tQG = tmem_base + 192;
    const uint32_t tXs = tmem_base + 256, tXo = tmem_base + 384;

    if (warp == 0) {
        // ================= TMA producer
        if (elect_lane0()) {
            for (int i = 0; i < nch; ++i) {
                const int t0 = i * kTile, st = i & 1, use = i >> 1;
                if (i >= 1 && !sy.wait(&qk_empty, i - 1)) break;
                if (use >= 1 && !sy.wait(&v_empty[st], use - 1)) break;
                // groups 1-3: the staging (these tiles) of chunk i - 2 has been stored
                if (!intra && i >= 2 && !sy.wait(&stage_free, i - 2)) break;
                mbar_arrive_expect_tx(&chunk_full[st], 2 * kQK + kV);
                tma_load_3d(tq, &tm_q, 0, t0, bh, &chunk_full[st]);
                tma_load_3d(tk, &tm_k, 0, t0, bh, &chunk_full[st]);
                tma_load_3d(tv + st * kV, &tm_v, 0, t0, bh, &chunk_full[st]);
                if (i + 1 < nch) {
                    tma_prefetch_3d(&tm_q, 0, t0 + kTile, bh);
                    tma_prefetch_3d(&tm_k, 0, t0 + kTile, bh);
                    tma_prefetch_3d(&tm_v, 0, t0 + kTile, bh);
                }
            }
        }
    } else if (warp == 1) {
        // ================= output MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdQK = idesc_bf16(128, kTile, false, false);
            constexpr uint32_t kIdQG = idesc_bf16(128, D, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
            const uint64_t dQ = smem_desc(smem_u32(tq), 16, 1024, kSw128);       // K-major A
            const uint64_t dKb = smem_desc(smem_u32(tk), 16, 1024, kSw128);      // K-major B
            const uint64_t dGr = smem_desc(smem_u32(gram), 16, 1024, kSw128);    // K-major B
            const uint64_t dSp = smem_desc(smem_u32(spre), 16384, 1024, kSw128); // MN-major B
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);   // MN-major B
            const uint64_t dLq = smem_desc(smem_u32(lring), 16, 1024, kSw128);   // K-major A
            // P of key quarter q is ready: Xo += P_q V[32q .. 32q + 31]
            auto pv_quarter = [&](int i, int q, uint32_t vo) -> bool {
                if (!sy.wait(&p_full[q], i)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_ts(tXo, tXs + 32 * q + ks * 8, desc_add(dV0, vo + (2 * q + ks) * 2048), kIdPV, 1u);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t vo = st * kV;
                if (intra) {
                    ok = sy.wait(&chunk_full[st], i >> 1);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tQG, desc_add(dQ, ks * 32), desc_add(dGr, ks * 32), kIdQG, ks > 0);
                    mma_commit(&qg_done);
                    // Xs = Q K^T over the whole chunk, once the previous chunk's P V
                    // MMAs (which read P from these columns) have completed
                    if (i > 0 && !sy.wait(&pv_done, i - 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_ss(tXs, desc_add(dQ, ks * 32), desc_add(dKb, ks * 32), kIdQK, ks > 0);
                    mma_commit(&xs_full);
                    mma_commit(&qk_empty);
                }
#pragma unroll 1
                for (int b = 0; b < nb && ok; ++b) {
                    const int gb = i * nb + b, ls = gb & 1;
                    ok = sy.wait(&block_ready[ls], gb >> 1) &&
                         (b != 0 || i == 0 || sy.wait(&o_empty, i - 1));
                    if (!ok) break;
                    tc_fence_after();
                    const int sp = intra ? 0 : ls;   // S_pre slot
                    const uint64_t a0 = desc_add(dLq, ls * 65536), b0 = desc_add(dSp, sp * 16384);
                    if (block_feats(b_first + b) == 128) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ss(tXo, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32),
                                   desc_add(b0, ks * 2048), kIdPV, (b > 0 || ks > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tXo, desc_add(a0, ks * 32), desc_add(b0, ks * 2048), kIdPV,
                                   (b > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&spre_empty[sp]);
                    mma_commit(&block_empty[ls]);
                    if (intra) ok = pv_quarter(i, b, vo);
                }
                for (int q = nb; intra && q < 4 && ok; ++q) ok = pv_quarter(i, q, vo);
                if (!ok) break;
                if (intra) mma_commit(&pv_done);
                mma_commit(&o_full);
                if (intra) mma_commit(&v_empty[st]);
            }
            mma_commit(&fin_bar[0]);
            sy.wait(&fin_bar[0], 0);
        }
    } else if (warp == 2) {
        // ================= state MMAs
        if (elect_lane0()) {
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            const uint64_t dKg = smem_desc(smem_u32(tk), 16384, 1024, kSw128);  // MN-major (Gram)
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);  // MN-major B
            const uint64_t dLk = smem_desc(smem_u32(lring + 32768), 16384, 1024, kSw128); // MN-major A
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t vo = st * kV;
                ok = sy.wait(&chunk_full[st], i >> 1);
                if (!ok) break;
                tc_fence_after();
                if (intra) {   // G += K^T K, after the P warps have read G_pre for this chunk
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        const uint64_t a = desc_add(dKg, ks * 2048);
                        mma_ss(tG, a, a, kIdGram, (i > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&gram_done);
                    mma_commit(&qk_empty);
                }
#pragma unroll 1
                for (int b = 0; b < nb && ok; ++b) {
                    const int gb = i * nb + b, ls = gb & 1;
                    ok = sy.wait(&block_ready[ls], gb >> 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = desc_add(dLk, ls * 65536), b0 = desc_add(dV0, vo);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + b * DV, desc_add(a0, ks * 2048), desc_add(b0, ks * 2048), kIdState,
                               (i > 0 || ks > 0) ? 1u : 0u);
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
        // ================= convert warps: S_run block -> bf16 S_pre (and, in
        // group 0, the epilogue)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        // Group 0: numerator rows of chunk i -> the warp's 2 KB staging slot, 16
        // columns at a time -> TMA stores of [32 rows x 16 floats]
        uint8_t *slot = gstage + quarter * 2048;
        auto epilogue0 = [&](int i) -> bool {
            bool w = __all_sync(0xffffffffu, sy.wait(&o_full, i));
            if (!w) return false;
            tc_fence_after();
            uint32_t v[DV];
            tmem_ld64(tXo + lsel, v);
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&o_empty);
            const int t0 = i * kTile + quarter * 32;
#pragma unroll
            for (int r = 0; r < DV / 16; ++r) {
                if (elect_lane0()) bulk_wait_read_all();   // the slot's previous store has read it
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 4; ++c)   // 64-byte swizzle: chunk c of row l at c ^ ((l / 2) % 4)
                    st_shared_v4(smem_u32(slot + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)),
                                 v[16 * r + 4 * c], v[16 * r + 4 * c + 1], v[16 * r + 4 * c + 2],
                                 v[16 * r + 4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_lane0() && t0 < T) {   // rows past T are clipped by the store
                    tma_store_3d(&tm_part16, 16 * r, t0, bh, slot);
                    bulk_commit();
                }
            }
            return true;
        };
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
#pragma unroll 1
            for (int b = 0; b < nb && ok; ++b) {
                // group 0: the previous chunk's output goes out between this chunk's
                // two blocks (its OUT MMAs of block 0 wait for the accumulator)
                if (intra && b == 1 && i > 0 && !(ok = epilogue0(i - 1))) break;
                const int gb = i * nb + b, ss = gb & 1;
                const int sp = intra ? 0 : ss, suse = intra ? gb : gb >> 1;   // S_pre slot, use
                // S_pre of the first chunk is zero (one segment per head); the
                // state MMAs start their accumulators from zero
                bool w = (suse == 0 || sy.wait(&spre_empty[sp], suse - 1)) &&
                         (i == 0 || sy.wait(&state_done[b], i - 1));
                ok = __all_sync(0xffffffffu, w);
                if (!ok) break;
                tc_fence_after();
                if (quarter * 32 < block_feats(b_first + b)) {
                    const uint32_t srow =
                        smem_u32(spre + sp * 16384 + (row >> 3) * 1024 + (row & 7) * 128);
#pragma unroll
                    for (int c32 = 0; c32 < DV; c32 += 32) {
                        uint32_t v[32];
                        if (i > 0) tmem_ld32(tS + lsel + b * DV + c32, v);
                        else
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = 0u;
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
                }
                tc_fence_before();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&block_ready[ss]);
            }
        }
        if (intra && ok && nch > 0) ok = epilogue0(nch - 1);
        if (srec != nullptr && ok && nch > 0) {   // state export: S after the last chunk
#pragma unroll 1
            for (int b = 0; b < nb && ok; ++b) {
                ok = __all_sync(0xffffffffu, sy.wait(&state_done[b], nch - 1));
                if (!ok) break;
                tc_fence_after();
                if (quarter * 32 < block_feats(b_first + b)) {
                    float *dst = srec + (size_t)bh * kRec64 + ((size_t)(b_first + b) * 128 + row) * DV;
#pragma unroll
                    for (int c32 = 0; c32 < DV; c32 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tS + lsel + b * DV + c32, v);
#pragma unroll
                        for (int e = 0; e < 4; ++e) st_global_v8(dst + c32 + 8 * e, v + 8 * e);
                    }
                }
            }
        }
        if (elect_lane0()) bulk_wait_all();
    } else if (warp < kWarpLift) {
        // ================= P warps: lane quarter q owns query rows 32q..32q+31
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        // P of key quarter q of the chunk (Q K^T ready in TMEM), written over the
        // first 16 columns of the quarter; adds this row's weights to dsum
        auto build_p = [&](int q, float &dsum) {
            uint32_t v[32];
            tmem_ld32(tXs + lsel + 32 * q, v);
            uint32_t pw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int s = 32 * q + 2 * j;
                const float x0 = __uint_as_float(v[2 * j]), x1 = __uint_as_float(v[2 * j + 1]);
                const float w0 = s <= row ? x0 * x0 : 0.f;
                const float w1 = s + 1 <= row ? x1 * x1 : 0.f;
                dsum += w0;
                dsum += w1;
                pw[j] = pack_bf16(w0, w1);
            }
            tmem_st16(tXs + lsel + 32 * q, pw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&p_full[q]);
        };
        // Groups 1-3: this group's numerator rows of chunk i.  The accumulator
        // is read into registers and released at once.
        uint8_t *sq = stage + quarter * 8192;
        auto epilogue = [&](int i) -> bool {
            bool w = __all_sync(0xffffffffu, sy.wait(&o_full, i));
            if (!w) return false;
            tc_fence_after();
            const int t0 = i * kTile + quarter * 32;
            uint32_t v[DV];
            tmem_ld64(tXo + lsel, v);
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&o_empty);
            // the tiles hold chunk i + 1 until the lift warps have read it
            w = __all_sync(0xffffffffu, sy.wait(&qk_empty, min(i + 1, nch - 1)));
            if (!w) return false;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(smem_u32(sq + h * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)),
                                 v[32 * h + 4 * c], v[32 * h + 4 * c + 1], v[32 * h + 4 * c + 2],
                                 v[32 * h + 4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (elect_lane0()) {
                if (t0 < T) {   // rows past T are clipped by the store
                    const int z = grp * (int)gridDim.y + bh;
                    tma_store_3d(&tm_part, 0, t0, z, sq);
                    tma_store_3d(&tm_part, 32, t0, z, sq + 4096);
                    bulk_commit();
                }
                bulk_wait_read_all();
                mbar_arrive(&stage_free);
            }
            return true;
        };
        // G rows r = 32 * quarter + lane (quarters 0-1) -> bf16 [64][64] K-major,
        // 128-byte swizzle; from_tmem false: zero (G_pre of the first chunk; the
        // first Gram MMA overwrites the accumulator)
        auto gram_to_smem = [&](bool from_tmem) {
            if (quarter >= 2) return;
#pragma unroll
            for (int c32 = 0; c32 < D; c32 += 32) {
                uint32_t v[32];
                if (from_tmem) tmem_ld32(tG + lsel + c32, v);
                else
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = (c32 >> 3) + cc;
                    *reinterpret_cast<uint4 *>(gram + row * 128 + ((chunk ^ (row & 7)) << 4)) =
                        make_uint4(pack_bf16(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1])),
                                   pack_bf16(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3])),
                                   pack_bf16(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5])),
                                   pack_bf16(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7])));
                }
            }
        };
        // q^T G_pre q (Q G_pre from TMEM, q from the Q tile), then G -> bf16 for chunk i + 1
        auto d_inter = [&](int i, float &dsum) -> bool {
            bool w = __all_sync(0xffffffffu, sy.wait(&chunk_full[i & 1], i >> 1) &&
                                                 sy.wait(&qg_done, i) && sy.wait(&gram_done, i));
            if (!w) return false;
            tc_fence_after();
            PackedRow<D> r;
            tile_row_packed<D>(tq, row, r);
#pragma unroll
            for (int c32 = 0; c32 < D; c32 += 32) {
                uint32_t v[32];
                tmem_ld32(tQG + lsel + c32, v);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const uint32_t pr = r.w[c32 / 2 + m];
                    dsum = fmaf(__uint_as_float(v[2 * m]), __uint_as_float(pr << 16), dsum);
                    dsum = fmaf(__uint_as_float(v[2 * m + 1]), __uint_as_float(pr & 0xFFFF0000u), dsum);
                }
            }
            gram_to_smem(true);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) {
                mbar_arrive(&chunk_full[(i + 1) & 1]);   // G_pre of chunk i + 1
                mbar_arrive(&qk_empty);
            }
            return true;
        };

        bool ok = true;
        if (intra) {
            gram_to_smem(false);   // G_pre of the first chunk: zero
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&chunk_full[0]);
        }
        if (intra) {   // chunk i's P quarters and denominators
            for (int i = 0; i < nch && ok; ++i) {
                ok = __all_sync(0xffffffffu, sy.wait(&xs_full, i));
                if (!ok) break;
                tc_fence_after();
                float dsum = 0.f;
                build_p(0, dsum);
                if (!(ok = d_inter(i, dsum))) break;
#pragma unroll 1
                for (int q = 1; q < 4; ++q) build_p(q, dsum);
                const int t = i * kTile + row;
                if (t < T) dden[(size_t)bh * T + t] = dsum;
            }
            // state export: G after the last chunk (its rows are TMEM lanes 0-63;
            // the P warps waited for the last Gram MMA in d_inter)
            if (srec != nullptr && ok && nch > 0 && quarter < 2) {
                tc_fence_after();
                float *dst = srec + (size_t)bh * kRec64 + (size_t)kBlocks64 * 128 * DV + (size_t)row * D;
#pragma unroll
                for (int c32 = 0; c32 < D; c32 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tG + lsel + c32, v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) st_global_v8(dst + c32 + 8 * e, v + 8 * e);
                }
            }
        } else {
            for (int i = 0; i < nch && ok; ++i) ok = epilogue(i);
        }
        if (elect_lane0()) bulk_wait_all();
    } else {
        // ================= lift warps: token t, side (0 query, 1 key)
        const int side = (warp - kWarpLift) >> 2;
        const int quarter = warp & 3;   // TMEM lane quarter of this warp
        wide_lift_role(side ? tk : tq, lring + side * 32768, quarter * 32 + lane, side != 0,
                       tmem_base + 448 + 32 * side + ((uint32_t)(quarter * 32) << 16), b_first, nb,
                       nch, chunk_full, &qk_empty, block_ready, block_empty, &abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) flag_error64(4);
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// O = (N_0 + N_1 + N_2 + N_3) / D in bf16 (zero where D = 0); one thread per
// four output values.
__global__ void __launch_bounds__(256)
wide_finalize_kernel(const float *__restrict__ part, const float *__restrict__ dden,
                     __nv_bfloat16 *__restrict__ out, int64_t rows, int64_t stride) {
    const int64_t n4 = rows * 16;   // 64 values per row
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e >> 4;
        const float4 *p = reinterpret_cast<const float4 *>(part) + e;
        float4 s = p[0];
#pragma unroll
        for (int g = 1; g < 4; ++g) {
            const float4 x = p[g * stride / 4];
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
        const float dd = dden[row];
        const float inv = dd > 0.f ? 1.f / dd : 0.f;
        __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(out) + 2 * e;
        o[0] = __floats2bfloat162_rn(s.x * inv, s.y * inv);
        o[1] = __floats2bfloat162_rn(s.z * inv, s.w * inv);
    }
}

// The final state of a head in the decode layout (as the d = 32 export):
// state[f][c] and z[f] for the row-major upper-triangle feature f of (i, j),
// sqrt(2) on the off-diagonal entries.  The grouped layout carries a factor 2 on
// the key side off the diagonal, so those rows are scaled by 1/sqrt(2); z_f is
// G_ij (sqrt(2) G_ij for i < j).  Grid (kBlocks64 + 1, BH), 128 threads: CTA
// b < kBlocks64 moves feature block b (one thread per feature slot), the last
// one the Gram into z.
__global__ void __launch_bounds__(128)
state_export64_kernel(const float *__restrict__ srec, float *__restrict__ state,
                      float *__restrict__ z) {
    constexpr int D = 64, DV = 64, kN = D * (D + 1) / 2;
    const int b = blockIdx.x, bh = blockIdx.y, p = threadIdx.x;
    const float *rec = srec + (size_t)bh * kRec64;
    float *st = state + (size_t)bh * kN * DV;
    if (b < kBlocks64) {
        int i = 0, j = 0;
        if (!grouped_slot_pair64(b, p, i, j)) return;
        const int f = i * D - i * (i - 1) / 2 + (j - i);
        const float sc = i == j ? 1.f : 0.70710678118654752f;
        const float4 *src = reinterpret_cast<const float4 *>(rec + ((size_t)b * 128 + p) * DV);
        float4 *dst = reinterpret_cast<float4 *>(st + (size_t)f * DV);
#pragma unroll 4
        for (int e = 0; e < DV / 4; ++e) {
            const float4 x = src[e];
            dst[e] = make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc);
        }
        return;
    }
    const float *gram = rec + (size_t)kBlocks64 * 128 * DV;
    for (int e = p; e < D * D; e += blockDim.x) {
        const int i = e / D, j = e % D;
        if (j < i) continue;
        z[(size_t)bh * kN + i * D - i * (i - 1) / 2 + (j - i)] = i == j ? gram[e] : kSqrt2 * gram[e];
    }
}

}  // namespace

// ================================================================= host side
// The partial numerators part[4 * BH][T][64] fp32 as a 3-D tensor for TMA
// stores; box = [32 rows x `cols` floats], swizzled over its row of cols * 4
// bytes (32 columns: 128-byte swizzle; 16 columns: 64-byte swizzle).
bool make_part_map(CUtensorMap &m, void *base, int T, int Z, int cols) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)Z};
    const cuuint64_t strides[2] = {64 * 4, (cuuint64_t)T * 64 * 4};
    const cuuint32_t box[3] = {(cuuint32_t)cols, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Any head count: with fewer than 38 heads the four CTAs per head leave SMs idle,
// and each head's chunks run in order, but the kernels still outpace the CUDA
// cores from two heads on (measured on GB300 at T = 2048 .. 65536: 2x to 25x; one
// head at T = 65536 runs ~10 % slower than there, and the quadratic form is 5x
// faster than both).
bool tc64_supported(const FwdShape &s, int cc_major, int cc_minor, int num_sms) {
    (void)num_sms;
    return s.dtype == 1 && cc_major == 10 && cc_minor == 3 && s.d == 64 && s.dv == 64 &&
           s.BH() <= 65535 && encoder() != nullptr;
}

// Workspace: partial numerators [4][rows][64] fp32, D [rows] fp32, then (state
// export) the final-state records [BH][kRec64] fp32 from a 256-byte boundary
// (their 32-byte stores need it), then (eps terms) the finalize's scratch from
// the next 256-byte boundary.
size_t srec_offset_floats(size_t rows) { return (rows * 64 * 4 + rows + 63) & ~(size_t)63; }
size_t sigma_offset_floats(const FwdShape &s, bool with_state) {
    const size_t o = srec_offset_floats((size_t)s.BH() * s.T);
    return with_state ? (o + (size_t)s.BH() * kRec64 + 63) & ~(size_t)63 : o;
}

size_t tc64_workspace_bytes(const FwdShape &s, bool with_state, const MapSpec *sigma) {
    const size_t rows = (size_t)s.BH() * s.T;
    if (sigma != nullptr)
        return sizeof(float) * sigma_offset_floats(s, with_state) + sigma_workspace_bytes(s);
    return sizeof(float) * (with_state ? srec_offset_floats(rows) + (size_t)s.BH() * kRec64
                                       : rows * 64 * 4 + rows);
}

cudaError_t tc64_forward(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                         void *workspace, cudaStream_t stream, const StateOut &so,
                         const MapSpec *sigma) {
    const int NCt = (s.T + kTile - 1) / kTile;
    const size_t rows = (size_t)s.BH() * s.T;
    if (rows == 0) return cudaSuccess;
    float *part = static_cast<float *>(workspace);
    float *dden = part + rows * 64 * 4;
    float *srec = so.state != nullptr ? part + srec_offset_floats(rows) : nullptr;   // final-state records
    CUtensorMap mq, mk, mv, mp, mp16;
    if (!make_map(mq, q, s.d, s.T, s.BH()) || !make_map(mk, k, s.d, s.T, s.BH()) ||
        !make_map(mv, v, s.dv, s.T, s.BH()) || !make_part_map(mp, part, s.T, 4 * s.BH(), 32) ||
        !make_part_map(mp16, part, s.T, 4 * s.BH(), 16))
        return cudaErrorInvalidValue;
    cudaFuncSetAttribute(wide_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemWide);
    {
        TraceScope tr("tc64_output", stream);
        wide_output_kernel<<<dim3(4, s.BH()), 608, kSmemWide, stream>>>(mq, mk, mv, mp, mp16, dden,
                                                                        srec, s.T, NCt);
    }
    if (sigma != nullptr) {
        cudaError_t e = sigma_finalize_launch(s, SigmaParts::Wide, part,
                                              part + sigma_offset_floats(s, srec != nullptr), q, k, v,
                                              out, *sigma, stream, so.eps_totals);
        if (e != cudaSuccess) return e;
    } else {
        TraceScope tr("tc64_finalize", stream);
        const int64_t n4 = (int64_t)rows * 16;
        const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, 152 * 16);
        wide_finalize_kernel<<<blocks, 256, 0, stream>>>(part, dden, (__nv_bfloat16 *)out,
                                                          (int64_t)rows, (int64_t)rows * 64);
    }
    if (srec != nullptr) {
        TraceScope tr("tc64_state_export", stream);
        state_export64_kernel<<<dim3(kBlocks64 + 1, s.BH()), 128, 0, stream>>>(srec, so.state, so.z);
    }
    return cudaGetLastError();
}

int tc64_take_error() {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc64_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (h) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_tc64_error, &zero, sizeof(int));
    }
    return h;
}

}  // namespace kata
