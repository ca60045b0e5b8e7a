// tcgen05 tensor-core path of the KATA chunked forward (bf16 inputs, sm_103a).
//
// The method (KATA paper, Sec. 4.1 Eq. 17-20, App. D.2 Algorithm 1) walks the
// chunks of a head in order, carrying the state (S, Z).  To fill 152 SMs at
// small batch (B*H = 16 heads for T = 131072), each head is cut into G
// segments of whole 128-token chunks, and the exclusive scan over chunks of
// Eq. 17 (Sec. 4.2) is done at two levels:
//
//   1. seg_state_kernel   per (segment, head): the segment's state sum
//                         Psi(K)^T V over all its chunks (tcgen05, fp32
//                         accumulators in TMEM) and its key Gram matrix K^T K.
//                                                                      [Eq. 17]
//   2. exclusive scan     of the segment states over segments (CUDA cores).
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
// packing of psi: row i of the upper triangle (j = i..d-1) is padded to an even
// length and consecutive (j, j+1) share one 32-bit bf16 pair; the sqrt(2) of
// the off-diagonal entries is applied as a factor 2 on the key side only
// (psi_q = q_i q_j, psi_k = 2 k_i k_j for i < j, k_i^2 on the diagonal), which
// keeps psi(q).psi(k) = (q.k)^2 and makes every lifted entry an exactly
// rounded bf16 product.  Padded entries are zero.
//
// Chunk.  The tensor path uses 128-token chunks (the MMA tile height) for
// every requested C; Eq. 17-20 give the same function for any chunk size, so
// C only changes rounding.
#include <cuda.h>

#include <mutex>
#include <utility>

#include "kata_internal.cuh"
#include "kata_sm100.cuh"

namespace kata {

__device__ int g_tc_error = 0;   // sticky: bounded waits that expired

namespace {

using namespace sm100;
using bf16 = __nv_bfloat16;

constexpr int kTile = 128;   // tokens per chunk = MMA M

// ---------------------------------------------------------------- feature order
template <int D>
struct Words {
    static constexpr int rowlen(int i) { return (D - i + 1) / 2; }
    static constexpr int count() {
        int s = 0;
        for (int i = 0; i < D; ++i) s += rowlen(i);
        return s;
    }
    static constexpr int row_of(int w) {
        int i = 0;
        while (w >= rowlen(i)) {
            w -= rowlen(i);
            ++i;
        }
        return i;
    }
    static constexpr int col_of(int w) {
        int i = 0;
        while (w >= rowlen(i)) {
            w -= rowlen(i);
            ++i;
        }
        return i + 2 * w;
    }
};

template <int D, int DV>
struct Cfg {
    static constexpr int NW = Words<D>::count();       // bf16 pairs per lifted row
    static constexpr int NF = 2 * NW;                  // padded feature count
    static constexpr int NBLK = (NF + 127) / 128;      // 128-feature state blocks
    static constexpr int QK_ROW = D * 2;               // bytes per q/k row
    static constexpr int V_ROW = DV * 2;
    static constexpr int QK_TILE = kTile * QK_ROW;
    static constexpr int V_TILE = kTile * V_ROW;
    static constexpr int E = NBLK * 128 * DV + D * D;  // floats per segment record
};

// ---- packed bf16x2 lift: one mul.rn.bf16x2 per lifted pair.  A product of two
// bf16 values is exact in fp32, so this rounds exactly like the fp32 lift above.
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// A row as bf16 pairs: w[m] = (x_2m, x_2m+1); so[m] = (x_2m+1, x_2m+2) with x_D = 0.
template <int D>
struct PackedRow {
    uint32_t w[D / 2];
    uint32_t so[D / 2];
};

template <int D>
__device__ __forceinline__ void load_packed(const bf16 *__restrict__ p, int bh, int T, int tok,
                                            PackedRow<D> &r) {
    if (tok < T) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p + ((size_t)bh * T + tok) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 u = __ldg(src + c);
            r.w[4 * c + 0] = u.x;
            r.w[4 * c + 1] = u.y;
            r.w[4 * c + 2] = u.z;
            r.w[4 * c + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int m = 0; m < D / 2; ++m) r.w[m] = 0u;
    }
#pragma unroll
    for (int m = 0; m < D / 2; ++m)
        r.so[m] = __byte_perm(r.w[m], m + 1 < D / 2 ? r.w[m + 1] : 0u, 0x5432);
}

template <int D, bool KEY, int W>
__device__ __forceinline__ uint32_t lift_word2(const PackedRow<D> &r) {
    if constexpr (W >= Words<D>::count()) {
        return 0u;
    } else {
        constexpr int I = Words<D>::row_of(W);
        constexpr int J = Words<D>::col_of(W);
        uint32_t pair;
        if constexpr (J % 2 == 0) pair = r.w[J / 2];
        else pair = r.so[(J - 1) / 2];
        uint32_t bc = __byte_perm(r.w[I / 2], 0u, (I % 2 == 0) ? 0x1010 : 0x3232);   // (x_I, x_I)
        if constexpr (KEY) {
            const uint32_t bc2 = bmul2(bc, 0x40004000u);                             // (2x_I, 2x_I)
            if constexpr (J == I) bc = __byte_perm(bc, bc2, 0x7610);                 // (x_I, 2x_I)
            else bc = bc2;
        }
        return bmul2(bc, pair);
    }
}

template <int D, bool KEY, int W0>
__device__ __forceinline__ void lift_chunk2(const PackedRow<D> &r, uint8_t *dst) {
    uint4 v;
    v.x = lift_word2<D, KEY, W0 + 0>(r);
    v.y = lift_word2<D, KEY, W0 + 1>(r);
    v.z = lift_word2<D, KEY, W0 + 2>(r);
    v.w = lift_word2<D, KEY, W0 + 3>(r);
    *reinterpret_cast<uint4 *>(dst) = v;
}

// ---- lift with per-row broadcasts computed once per token: bc[i] holds
// (x_i, x_i) for queries and (2 x_i, 2 x_i) for keys, so each lifted pair is a
// single mul.bf16x2 (keys: the diagonal pair of row i uses (x_i, 2 x_i)).
template <int D>
struct LiftRow {
    uint32_t w[D / 2];    // (x_2m, x_2m+1)
    uint32_t so[D / 2];   // (x_2m+1, x_2m+2), x_D = 0
    uint32_t bc[D];       // row broadcasts
};

template <int D, bool KEY>
__device__ __forceinline__ void make_lift_row(const PackedRow<D> &p, LiftRow<D> &r) {
#pragma unroll
    for (int m = 0; m < D / 2; ++m) {
        r.w[m] = p.w[m];
        r.so[m] = p.so[m];
    }
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const uint32_t b = __byte_perm(p.w[i / 2], 0u, (i % 2 == 0) ? 0x1010 : 0x3232);
        r.bc[i] = KEY ? bmul2(b, 0x40004000u) : b;
    }
}

template <int D, bool KEY, int W>
__device__ __forceinline__ uint32_t lift_word3(const LiftRow<D> &r) {
    if constexpr (W >= Words<D>::count()) {
        return 0u;
    } else {
        constexpr int I = Words<D>::row_of(W);
        constexpr int J = Words<D>::col_of(W);
        uint32_t pair;
        if constexpr (J % 2 == 0) pair = r.w[J / 2];
        else pair = r.so[(J - 1) / 2];
        uint32_t bc = r.bc[I];
        if constexpr (KEY && J == I)   // (x_I, 2 x_I): low half from the raw row
            bc = __byte_perm(r.w[I / 2], bc, (I % 2 == 0) ? 0x7610 : 0x7632);
        return bmul2(bc, pair);
    }
}

template <int D, bool KEY, int W0>
__device__ __forceinline__ void lift_chunk3(const LiftRow<D> &r, uint8_t *dst) {
    uint4 v;
    v.x = lift_word3<D, KEY, W0 + 0>(r);
    v.y = lift_word3<D, KEY, W0 + 1>(r);
    v.z = lift_word3<D, KEY, W0 + 2>(r);
    v.w = lift_word3<D, KEY, W0 + 3>(r);
    *reinterpret_cast<uint4 *>(dst) = v;
}

// Destinations of the 8 16-byte chunks of token row t in a [128 x 64] atom
// column with the 128-byte swizzle (chunk c stored at chunk c ^ (t % 8)).
struct ChunkPtrs {
    uint8_t *p[8];
};
__device__ __forceinline__ ChunkPtrs chunk_ptrs(uint8_t *tile_col, int t) {
    ChunkPtrs c;
    uint8_t *row = tile_col + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) c.p[ch] = row + ((ch ^ (t & 7)) << 4);
    return c;
}

template <int D, bool KEY, int AC, int... CH>
__device__ __forceinline__ void lift_col2_impl(const PackedRow<D> &r, const ChunkPtrs &cp,
                                               std::integer_sequence<int, CH...>) {
    (lift_chunk2<D, KEY, 32 * AC + 4 * CH>(r, cp.p[CH]), ...);
}

// Lift words 32*AC .. 32*AC + 4*NCH - 1 (NCH chunks) of one token row.
template <int D, bool KEY, int AC, int NCH = 8>
__device__ __forceinline__ void lift_col2(const PackedRow<D> &r, const ChunkPtrs &cp) {
    lift_col2_impl<D, KEY, AC>(r, cp, std::make_integer_sequence<int, NCH>{});
}

// Runtime atom-column dispatch.  Atom columns holding only padding (every word
// >= Words<D>::count()) are skipped, and a partly padded column stops at its
// last real chunk: no MMA reads past the real features of a column's block.
template <int D, bool KEY>
__device__ __forceinline__ void lift_col2_rt(int ac, const PackedRow<D> &r, const ChunkPtrs &cp) {
    constexpr int NW = Words<D>::count();
    switch (ac) {
#define KATA_LIFT_CASE(A)                                                                  \
    case A:                                                                                \
        if constexpr (32 * (A) < NW) {                                                     \
            constexpr int nch = (NW - 32 * (A)) >= 32 ? 8 : ((NW - 32 * (A)) + 3) / 4;    \
            lift_col2<D, KEY, A, nch>(r, cp);                                              \
        }                                                                                  \
        break;
        KATA_LIFT_CASE(0) KATA_LIFT_CASE(1) KATA_LIFT_CASE(2) KATA_LIFT_CASE(3)
        KATA_LIFT_CASE(4) KATA_LIFT_CASE(5) KATA_LIFT_CASE(6) KATA_LIFT_CASE(7)
        KATA_LIFT_CASE(8) KATA_LIFT_CASE(9)
#undef KATA_LIFT_CASE
        default: break;
    }
}

template <int D, bool KEY, int AC, int... CH>
__device__ __forceinline__ void lift_col3_impl(const LiftRow<D> &r, const ChunkPtrs &cp,
                                               std::integer_sequence<int, CH...>) {
    (lift_chunk3<D, KEY, 32 * AC + 4 * CH>(r, cp.p[CH]), ...);
}

template <int D, bool KEY>
__device__ __forceinline__ void lift_col3_rt(int ac, const LiftRow<D> &r, const ChunkPtrs &cp) {
    constexpr int NW = Words<D>::count();
    switch (ac) {
#define KATA_LIFT3_CASE(A)                                                                     \
    case A:                                                                                    \
        if constexpr (32 * (A) < NW) {                                                         \
            constexpr int nch = (NW - 32 * (A)) >= 32 ? 8 : ((NW - 32 * (A)) + 3) / 4;        \
            lift_col3_impl<D, KEY, A>(r, cp, std::make_integer_sequence<int, nch>{});          \
        }                                                                                      \
        break;
        KATA_LIFT3_CASE(0) KATA_LIFT3_CASE(1) KATA_LIFT3_CASE(2) KATA_LIFT3_CASE(3)
        KATA_LIFT3_CASE(4) KATA_LIFT3_CASE(5) KATA_LIFT3_CASE(6) KATA_LIFT3_CASE(7)
        KATA_LIFT3_CASE(8) KATA_LIFT3_CASE(9)
#undef KATA_LIFT3_CASE
        default: break;
    }
}

// Row t of a [128 x D] bf16 tile written by TMA with the swizzle matching its
// row width (32/64/128 bytes): the 16-byte chunk c of row t sits at chunk
// c ^ ((t * row_bytes >> 7) & (chunks_per_row - 1)).
template <int D>
__device__ __forceinline__ void tile_row_packed(const uint8_t *tile, int t, PackedRow<D> &r) {
    constexpr int RB = D * 2, CPR = RB / 16;
    const uint8_t *row = tile + t * RB;
    const int x = (t * RB >> 7) & (CPR - 1);
#pragma unroll
    for (int c = 0; c < CPR; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + ((c ^ x) << 4));
        r.w[4 * c + 0] = u.x;
        r.w[4 * c + 1] = u.y;
        r.w[4 * c + 2] = u.z;
        r.w[4 * c + 3] = u.w;
    }
#pragma unroll
    for (int m = 0; m < D / 2; ++m)
        r.so[m] = __byte_perm(r.w[m], m + 1 < D / 2 ? r.w[m + 1] : 0u, 0x5432);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void flag_error(int code) { atomicOr(&g_tc_error, code); }

// Shared abort flag: any role whose bounded wait expires sets it; every later
// wait then returns at once, so all roles drain to the final barrier.
struct Sync {
    volatile int *abort;
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t n) const {
        if (*abort) return false;
        if (mbar_wait(bar, n & 1u)) return true;
        *abort = 1;
        return false;
    }
};

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

// ================================================================= kernel 1
// Segment state of one (segment, head): S_seg = sum over the segment's tokens of
// psi_k(k) v^T (all feature blocks, fp32 in TMEM) and G_seg = K^T K.
//   warp 0: TMA (K and V tiles, 2 stages)      warp 1: MMA issue
//   warps 2-9: key lift into a 3-stage ring (two warps per 32 tokens, one
//   64-feature atom column each), then the epilogue (warps 2-5)
template <int D, int DV>
__global__ void __launch_bounds__(320, 1)
seg_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 float *__restrict__ seg, int NCt, int Lc, int G) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32, "layouts below are written for d = 32, dv = 64");
    constexpr int kStage = C::QK_TILE + C::V_TILE;
    constexpr int kRing = 3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *ring = sm + 2 * kStage;                     // [kRing][32 KB]: psi_k block
    __shared__ __align__(8) uint64_t tile_full[2], tile_empty[2], lift_full[kRing],
        lift_empty[kRing], done_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int g = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;
    const Sync sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tile_full[i], 1);
            mbar_init(&tile_empty[i], 1 + 8);        // MMA commit + 8 lift warps
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&lift_full[i], 8);
            mbar_init(&lift_empty[i], 1);
        }
        mbar_init(&done_bar, 1);
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
            for (int i = 0; i < nch; ++i) {
                const int st = i & 1, use = i >> 1;
                if (use >= 1 && !sy.wait(&tile_empty[st], use - 1)) break;
                uint8_t *tk = sm + st * kStage;
                const int t0 = (c0 + i) * kTile;
                mbar_arrive_expect_tx(&tile_full[st], kStage);
                tma_load_3d(tk, &tm_k, 0, t0, bh, &tile_full[st]);
                tma_load_3d(tk + C::QK_TILE, &tm_v, 0, t0, bh, &tile_full[st]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issue
        if (elect_lane0()) {
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            // base descriptors: K tile as MN-major A/B of the Gram, lifted keys as
            // MN-major A and V as MN-major B of the state update
            const uint64_t dK = smem_desc(smem_u32(sm), 8192, 512, kSw64);
            const uint64_t dV = smem_desc(smem_u32(sm + C::QK_TILE), 16384, 1024, kSw128);
            const uint64_t dR = smem_desc(smem_u32(ring), 16384, 1024, kSw128);
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                ok = sy.wait(&tile_full[st], i >> 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    const uint64_t a = desc_add(dK, st * kStage + ks * 1024);
                    mma_ss(tG, a, a, kIdGram, (i > 0 || ks > 0) ? 1u : 0u);
                }
                for (int b = 0; b < C::NBLK && ok; ++b) {
                    const int gb = i * C::NBLK + b, rs = gb % kRing;
                    ok = sy.wait(&lift_full[rs], gb / kRing);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + b * DV, desc_add(dR, rs * 32768 + ks * 2048),
                               desc_add(dV, st * kStage + ks * 2048), kIdState, (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&lift_empty[rs]);
                }
                mma_commit(&tile_empty[st]);
            }
            mma_commit(&done_bar);
        }
    } else {
        // ---------------- lift warps (2..9): token t, atom column half h
        const int t = ((warp - 2) & 3) * 32 + lane, h = (warp - 2) >> 2;
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
                lift_col2_rt<D, true>(2 * b + h, r, chunk_ptrs(ring + rs * 32768 + h * 16384, t));
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&lift_full[rs]);
            }
        }
        // ---------------- epilogue (warps 2-5): state and Gram rows to the segment record
        ok = __all_sync(0xffffffffu, sy.wait(&done_bar, 0));
        tc_fence_after();
        if (ok && h == 0) {
            const int quarter = warp & 3;
            const int lrow = quarter * 32 + lane;
            const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
            float *rec = seg + ((size_t)bh * G + g) * C::E;
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

// ================================================================= kernel 3
// Segment output: walk the segment's chunks with the running state in TMEM.
//   warp 0: TMA (Q, K tiles: 1 stage; V tile: 2 stages)     warp 1: MMA issue
//   warps 2-5 ("TMEM warps", lane quarter = warp % 4): P = (QK^T)^2 masked,
//     denominators, S_run -> S_pre conversion, output epilogue, Gram -> bf16
//   warps 6-13: query/key lift into a 2-stage ring; each thread lifts one
//     token's row of one side (query or key) into both atom columns of a block
// TMEM: S_run [0,320) | G [320,352) | Q G_pre [352,384) | QK^T half [384,448) |
//       output accumulator [448,512)
template <int D, int DV>
__global__ void __launch_bounds__(448, 1)
seg_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, bf16 *__restrict__ out,
                  const float *__restrict__ seg, int T, int NCt, int Lc, int G) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32 && C::NBLK == 5, "layouts below are written for d = 32, dv = 64");
    constexpr int NB = C::NBLK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tq = sm;                                   // Q tile, 8 KB (64-byte swizzle)
    uint8_t *tk = sm + C::QK_TILE;                      // K tile, 8 KB
    uint8_t *tv = sm + 2 * C::QK_TILE;                  // V tiles [2][16 KB]
    uint8_t *lring = tv + 2 * C::V_TILE;                // [2][psi_q 32 KB | psi_k 32 KB]
    uint8_t *pbuf = lring + 2 * 65536;                  // P half, 16 KB
    uint8_t *spre = pbuf + 16384;                       // S_pre block, 16 KB
    uint8_t *gram = spre + 16384;                       // G_pre bf16, 2 KB
    __shared__ __align__(8) uint64_t qk_full, qk_empty, v_full[2], v_empty[2], xs_full, xs_empty,
        p_full, p_empty, lift_full[2], lift_empty[2], spre_full, spre_empty, state_done[NB],
        o_full, o_empty, gram_done, gram_ready, fin_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int g = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;
    const Sync sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&qk_full, 1);
        mbar_init(&qk_empty, 1 + 8 + 4);   // MMA commit, 8 lift warps, 4 TMEM warps
        for (int i = 0; i < 2; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&lift_full[i], 8);
            mbar_init(&lift_empty[i], 1);
        }
        mbar_init(&xs_full, 1);
        mbar_init(&xs_empty, 4);
        mbar_init(&p_full, 4);
        mbar_init(&p_empty, 1);
        mbar_init(&spre_full, 4);
        mbar_init(&spre_empty, 1);
        for (int b = 0; b < NB; ++b) mbar_init(&state_done[b], 1);
        mbar_init(&o_full, 1);
        mbar_init(&o_empty, 4);
        mbar_init(&gram_done, 1);
        mbar_init(&gram_ready, 4);
        mbar_init(&fin_bar, 1);
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
    const uint32_t tXs = tmem_base + 384, tXo = tmem_base + 448;

    if (warp == 0) {
        // ================= TMA producer
        if (elect_lane0()) {
            for (int i = 0; i < nch; ++i) {
                const int t0 = (c0 + i) * kTile;
                if (i >= 1 && !sy.wait(&qk_empty, i - 1)) break;
                mbar_arrive_expect_tx(&qk_full, 2 * C::QK_TILE);
                tma_load_3d(tq, &tm_q, 0, t0, bh, &qk_full);
                tma_load_3d(tk, &tm_k, 0, t0, bh, &qk_full);
                const int st = i & 1, use = i >> 1;
                if (use >= 1 && !sy.wait(&v_empty[st], use - 1)) break;
                mbar_arrive_expect_tx(&v_full[st], C::V_TILE);
                tma_load_3d(tv + st * C::V_TILE, &tm_v, 0, t0, bh, &v_full[st]);
            }
        }
    } else if (warp == 1) {
        // ================= MMA issue
        if (elect_lane0()) {
            constexpr uint32_t kIdQK = idesc_bf16(128, 64, false, false);
            constexpr uint32_t kIdQG = idesc_bf16(128, D, false, false);
            constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
            constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
            constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
            // base descriptors, built once; each MMA only offsets the start address
            const uint64_t dQ = smem_desc(smem_u32(tq), 16, 512, kSw64);        // K-major A
            const uint64_t dKb = smem_desc(smem_u32(tk), 16, 512, kSw64);       // K-major B
            const uint64_t dKg = smem_desc(smem_u32(tk), 8192, 512, kSw64);     // MN-major (Gram)
            const uint64_t dGr = smem_desc(smem_u32(gram), 16, 512, kSw64);     // K-major B
            const uint64_t dP = smem_desc(smem_u32(pbuf), 16, 1024, kSw128);    // K-major A
            const uint64_t dSp = smem_desc(smem_u32(spre), 16384, 1024, kSw128); // MN-major B
            const uint64_t dV0 = smem_desc(smem_u32(tv), 16384, 1024, kSw128);  // MN-major B
            const uint64_t dLq = smem_desc(smem_u32(lring), 16, 1024, kSw128);  // K-major A
            const uint64_t dLk = smem_desc(smem_u32(lring + 32768), 16384, 1024, kSw128); // MN-major A
            auto qk_half = [&](int h) {   // Xs = Q K[64h .. 64h+63]^T
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tXs, desc_add(dQ, ks * 32), desc_add(dKb, h * 64 * 64 + ks * 32), kIdQK,
                           ks > 0);
                mma_commit(&xs_full);
            };
            auto pv_half = [&](int h, uint32_t vo) {   // Xo += P[:, 64h..] V[64h..]
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tXo, desc_add(dP, ks * 32), desc_add(dV0, vo + (h * 4 + ks) * 2048), kIdPV, 1u);
                mma_commit(&p_empty);
            };
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t vo = st * C::V_TILE;     // byte offset of this chunk's V tile
                // S/G pieces that need only the Q, K tiles
                ok = sy.wait(&qk_full, i) && sy.wait(&gram_ready, i) &&
                     (i == 0 || sy.wait(&xs_empty, 2 * i - 1));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tQG, desc_add(dQ, ks * 32), desc_add(dGr, ks * 32), kIdQG, ks > 0);
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    const uint64_t a = desc_add(dKg, ks * 1024);
                    mma_ss(tG, a, a, kIdGram, 1u);
                }
                mma_commit(&gram_done);
                qk_half(0);
                ok = sy.wait(&v_full[st], i >> 1);
                for (int b = 0; b < NB && ok; ++b) {
                    const int gb = i * NB + b, ls = gb & 1;
                    ok = sy.wait(&lift_full[ls], gb >> 1) && sy.wait(&spre_full, gb) &&
                         (b != 0 || i == 0 || sy.wait(&o_empty, i - 1));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t lo = ls * 65536;
                    const int fleft = C::NF - b * 128;
                    const int ksteps = fleft >= 128 ? 8 : (fleft + 15) / 16;
                    for (int ks = 0; ks < ksteps; ++ks)
                        mma_ss(tXo, desc_add(dLq, lo + (ks >> 2) * 16384 + (ks & 3) * 32),
                               desc_add(dSp, ks * 2048), kIdPV, (b > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&spre_empty);
                    if (b == NB - 1) mma_commit(&o_full);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(tS + b * DV, desc_add(dLk, lo + ks * 2048), desc_add(dV0, vo + ks * 2048),
                               kIdState, 1u);
                    mma_commit(&lift_empty[ls]);
                    mma_commit(&state_done[b]);
                    if (b == 0) {
                        // second half of Q K^T once the first has been read, then P V for it
                        ok = sy.wait(&xs_empty, 2 * i);
                        if (!ok) break;
                        tc_fence_after();
                        qk_half(1);
                        mma_commit(&qk_empty);
                        ok = sy.wait(&p_full, 2 * i);
                        if (!ok) break;
                        tc_fence_after();
                        pv_half(0, vo);
                    }
                    if (b == 2) {
                        ok = sy.wait(&p_full, 2 * i + 1);
                        if (!ok) break;
                        tc_fence_after();
                        pv_half(1, vo);
                    }
                }
                mma_commit(&v_empty[st]);
            }
            mma_commit(&fin_bar);
            sy.wait(&fin_bar, 0);
        }
    } else if (warp < 6) {
        // ================= TMEM warps: lane quarter q owns rows / features 32q..32q+31
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        auto convert_spre = [&](int i, int b) -> bool {   // S_run block b -> spre (bf16)
            const int gb = i * NB + b;
            bool w = (gb == 0 || sy.wait(&spre_empty, gb - 1)) && (i == 0 || sy.wait(&state_done[b], i - 1));
            w = __all_sync(0xffffffffu, w);
            if (!w) return false;
            tc_fence_after();
            uint8_t *srow = spre + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c32 = 0; c32 < DV; c32 += 32) {
                uint32_t v[32];
                tmem_ld32(tS + lsel + b * DV + c32, v);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = (c32 >> 3) + cc;
                    uint4 u;
                    u.x = pack_bf16(__uint_as_float(v[8 * cc + 0]), __uint_as_float(v[8 * cc + 1]));
                    u.y = pack_bf16(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3]));
                    u.z = pack_bf16(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5]));
                    u.w = pack_bf16(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7]));
                    *reinterpret_cast<uint4 *>(srow + ((chunk ^ (row & 7)) << 4)) = u;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&spre_full);
            return true;
        };
        // P for key half h from the Xs accumulator; returns this row's sum of weights
        auto build_p = [&](int i, int h, float &dsum) -> bool {
            bool w = sy.wait(&xs_full, 2 * i + h) && (2 * i + h == 0 || sy.wait(&p_empty, 2 * i + h - 1));
            w = __all_sync(0xffffffffu, w);
            if (!w) return false;
            tc_fence_after();
            uint8_t *prow = pbuf + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c32 = 0; c32 < 64; c32 += 32) {
            uint32_t v[32];
            tmem_ld32(tXs + lsel + c32, v);           // warp-collective: always executed
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int chunk = (c32 >> 3) + cc;
                const int s0 = h * 64 + chunk * 8;
                float wv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = __uint_as_float(v[8 * cc + e]);
                    wv[e] = (s0 + e <= row) ? x * x : 0.f;
                    dsum += wv[e];
                }
                uint4 u;
                u.x = pack_bf16(wv[0], wv[1]);
                u.y = pack_bf16(wv[2], wv[3]);
                u.z = pack_bf16(wv[4], wv[5]);
                u.w = pack_bf16(wv[6], wv[7]);
                *reinterpret_cast<uint4 *>(prow + ((chunk ^ (row & 7)) << 4)) = u;
            }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) {
                mbar_arrive(&xs_empty);
                mbar_arrive(&p_full);
            }
            return true;
        };
        auto epilogue = [&](int i, float dsum) -> bool {   // O = N / D for chunk i
            bool w = __all_sync(0xffffffffu, sy.wait(&o_full, i));
            if (!w) return false;
            tc_fence_after();
            const int t0 = (c0 + i) * kTile;
            const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
            const bool valid = t0 + row < T;
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * T + t0 + row) * DV);
#pragma unroll
            for (int c32 = 0; c32 < DV; c32 += 32) {
                uint32_t v[32];
                tmem_ld32(tXo + lsel + c32, v);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint4 u;
                    u.x = pack_bf16(__uint_as_float(v[8 * cc + 0]) * inv, __uint_as_float(v[8 * cc + 1]) * inv);
                    u.y = pack_bf16(__uint_as_float(v[8 * cc + 2]) * inv, __uint_as_float(v[8 * cc + 3]) * inv);
                    u.z = pack_bf16(__uint_as_float(v[8 * cc + 4]) * inv, __uint_as_float(v[8 * cc + 5]) * inv);
                    u.w = pack_bf16(__uint_as_float(v[8 * cc + 6]) * inv, __uint_as_float(v[8 * cc + 7]) * inv);
                    if (valid) dst[(c32 >> 3) + cc] = u;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&o_empty);
            return true;
        };
        auto gram_to_smem = [&](bool from_tmem, const float *pre) {
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
            if (!from_tmem) {
#pragma unroll
                for (int c = 0; c < D; c += 8) {
                    uint32_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(gv[c + e]);
                    tmem_st8(tG + lsel + c, v);
                }
            }
        };

        // ---- initial state: the segment's exclusive prefix (zero for g == 0)
        {
            const float *pre = g > 0 ? seg + ((size_t)bh * G + g) * C::E : nullptr;
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
            gram_to_smem(false, pre ? pre + (size_t)NB * 128 * DV : nullptr);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&gram_ready);
        }
        float dprev = 0.f;
        for (int i = 0; i < nch && ok; ++i) {
            ok = convert_spre(i, 0);
            if (ok && i > 0) ok = epilogue(i - 1, dprev);
            float dsum = 0.f;
            if (ok) ok = build_p(i, 0, dsum);
            if (ok) {   // inter-chunk denominator q^T G_pre q, with q from the Q tile
                PackedRow<D> r;
                tile_row_packed<D>(tq, row, r);
                float qv[D];
#pragma unroll
                for (int m = 0; m < D / 2; ++m) {
                    qv[2 * m] = __uint_as_float(r.w[m] << 16);
                    qv[2 * m + 1] = __uint_as_float(r.w[m] & 0xFFFF0000u);
                }
                {
                    uint32_t v[32];
                    tmem_ld32(tQG + lsel, v);
#pragma unroll
                    for (int e = 0; e < D; ++e) dsum = fmaf(__uint_as_float(v[e]), qv[e], dsum);
                }
                // Gram of this chunk -> bf16 for the next chunk's Q G MMA
                ok = __all_sync(0xffffffffu, sy.wait(&gram_done, i));
                if (ok) {
                    tc_fence_after();
                    gram_to_smem(true, nullptr);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (elect_lane0()) {
                        mbar_arrive(&gram_ready);
                        mbar_arrive(&qk_empty);
                    }
                }
            }
            if (ok) ok = convert_spre(i, 1);
            if (ok) ok = build_p(i, 1, dsum);
            for (int b = 2; b < NB && ok; ++b) ok = convert_spre(i, b);
            dprev = dsum;
        }
        if (ok && nch > 0) epilogue(nch - 1, dprev);
    } else {
        // ================= lift warps 6..13: token t, side (0 query, 1 key)
        const int lw = warp - 6;
        const int t = (lw & 3) * 32 + lane, side = lw >> 2;
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            ok = __all_sync(0xffffffffu, sy.wait(&qk_full, i));
            if (!ok) break;
            PackedRow<D> r;
            tile_row_packed<D>(side ? tk : tq, t, r);
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&qk_empty);
            for (int b = 0; b < NB && ok; ++b) {
                const int gb = i * NB + b, ls = gb & 1, use = gb >> 1;
                if (use >= 1) ok = __all_sync(0xffffffffu, sy.wait(&lift_empty[ls], use - 1));
                if (!ok) break;
                uint8_t *col = lring + ls * 65536 + side * 32768;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const ChunkPtrs cp = chunk_ptrs(col + h * 16384, t);
                    if (side) lift_col2_rt<D, true>(2 * b + h, r, cp);
                    else lift_col2_rt<D, false>(2 * b + h, r, cp);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (elect_lane0()) mbar_arrive(&lift_full[ls]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) flag_error(2);
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ================================================================= host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// [BH][T][inner] bf16 viewed as a 3-D tensor; box = one 128-row tile of one head.
bool make_map(CUtensorMap &m, const void *base, int inner, int T, int BH) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)T * inner * 2};
    const cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)kTile, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const int rb = inner * 2;
    const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int NCt, G, Lc;
};

Plan plan(const FwdShape &s, int num_sms) {
    Plan p;
    p.NCt = (s.T + kTile - 1) / kTile;
    int G = num_sms / s.BH();
    if (G < 1) G = 1;
    if (G > p.NCt) G = p.NCt;
    p.Lc = (p.NCt + G - 1) / G;
    p.G = (p.NCt + p.Lc - 1) / p.Lc;
    return p;
}

constexpr int kSmemState = 2 * (Cfg<32, 64>::QK_TILE + Cfg<32, 64>::V_TILE) + 3 * 32768 + 2048;
constexpr int kSmemOutput = 2 * Cfg<32, 64>::QK_TILE + 2 * Cfg<32, 64>::V_TILE + 2 * 65536 +
                            16384 + 16384 + 2048 + 2048;

}  // namespace

bool tc_supported(const FwdShape &s, int cc_major, int cc_minor) {
    return s.dtype == 1 && cc_major == 10 && cc_minor == 3 && s.d == 32 && s.dv == 64 &&
           encoder() != nullptr;
}

size_t tc_workspace_bytes(const FwdShape &s, int num_sms) {
    const Plan p = plan(s, num_sms);
    if (p.G <= 1) return 0;
    return sizeof(float) * (size_t)s.BH() * p.G * Cfg<32, 64>::E;
}

cudaError_t tc_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                       void *out, void *workspace, int num_sms, cudaStream_t stream) {
    using C = Cfg<32, 64>;
    const Plan p = plan(s, num_sms);
    CUtensorMap mq, mk, mv;
    if (!make_map(mq, q, s.d, s.T, s.BH()) || !make_map(mk, k, s.d, s.T, s.BH()) ||
        !make_map(mv, v, s.dv, s.T, s.BH()))
        return cudaErrorInvalidValue;
    float *seg = static_cast<float *>(workspace);
    if (p.G > 1) {
        cudaFuncSetAttribute(seg_state_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemState);
        {
            TraceScope tr("tc_segment_state", stream);
            seg_state_kernel<32, 64><<<dim3(p.G - 1, s.BH()), 320, kSmemState, stream>>>(
                mk, mv, seg, p.NCt, p.Lc, p.G);
        }
        cudaError_t e = scan_exclusive_launch(seg, s.BH(), p.G, C::E, "tc_segment_scan", stream);
        if (e != cudaSuccess) return e;
    }
    cudaFuncSetAttribute(seg_output_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemOutput);
    {
        TraceScope tr("tc_segment_output", stream);
        seg_output_kernel<32, 64><<<dim3(p.G, s.BH()), 448, kSmemOutput, stream>>>(
            mq, mk, mv, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.G);
    }
    return cudaGetLastError();
}

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
