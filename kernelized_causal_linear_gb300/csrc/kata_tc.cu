// tcgen05 tensor-core path of the KATA chunked forward (bf16 inputs, sm_103a).
//
// The method (KATA paper, Sec. 4.1 Eq. 17-20, App. D.2 Algorithm 1) walks the
// chunks of a head in order, carrying the state (S, Z).  To fill 152 SMs at
// small batch (B*H = 16 heads for T = 131072), each head is cut into G
// segments of whole 128-token chunks, and the exclusive scan over chunks of
// Eq. 17 (Sec. 4.2) is done at two levels:
//
//   1. seg_state_kernel   per (feature block, segment, head): the segment's
//                         state sum Psi(K)^T V over all its chunks (tcgen05,
//                         fp32 accumulator in TMEM) and its key Gram matrix
//                         K^T K.                                       [Eq. 17]
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
    static constexpr int NAC = 2 * NBLK;               // 64-feature atom columns
    static constexpr int QK_ROW = D * 2;               // bytes per q/k row
    static constexpr int V_ROW = DV * 2;
    static constexpr int QK_TILE = kTile * QK_ROW;
    static constexpr int V_TILE = kTile * V_ROW;
    static constexpr int E = NBLK * 128 * DV + D * D;  // floats per segment record
    static constexpr uint32_t QK_SW = QK_ROW == 128 ? kSw128 : QK_ROW == 64 ? kSw64 : kSw32;
};

// One lifted bf16 pair (features 2W, 2W+1) of one row x.
template <int D, bool KEY, int W>
__device__ __forceinline__ uint32_t lift_word(const float (&x)[D]) {
    if constexpr (W >= Words<D>::count()) {
        return 0u;
    } else {
        constexpr int I = Words<D>::row_of(W);
        constexpr int J = Words<D>::col_of(W);
        float lo = x[I] * x[J];
        float hi = 0.f;
        if constexpr (J + 1 < D) hi = x[I] * x[J + 1];
        if constexpr (KEY) {
            if constexpr (J != I) lo *= 2.f;
            hi *= 2.f;
        }
        return pack_bf16(lo, hi);
    }
}

template <int D, bool KEY, int W0>
__device__ __forceinline__ void lift_chunk(const float (&x)[D], uint8_t *dst) {
    uint4 v;
    v.x = lift_word<D, KEY, W0 + 0>(x);
    v.y = lift_word<D, KEY, W0 + 1>(x);
    v.z = lift_word<D, KEY, W0 + 2>(x);
    v.w = lift_word<D, KEY, W0 + 3>(x);
    *reinterpret_cast<uint4 *>(dst) = v;
}

// Lift one token row into one 64-feature atom column AC of a [128 x 64] SW128
// tile: row t, 8 chunks of 8 features, chunk c stored at chunk (c ^ (t % 8)).
template <int D, bool KEY, int AC, int... CH>
__device__ __forceinline__ void lift_col_impl(const float (&x)[D], uint8_t *row, int t7,
                                              std::integer_sequence<int, CH...>) {
    (lift_chunk<D, KEY, 32 * AC + 4 * CH>(x, row + ((CH ^ t7) << 4)), ...);
}

template <int D, bool KEY, int AC>
__device__ __forceinline__ void lift_col(const float (&x)[D], uint8_t *tile_col, int t) {
    lift_col_impl<D, KEY, AC>(x, tile_col + (t >> 3) * 1024 + (t & 7) * 128, t & 7,
                              std::make_integer_sequence<int, 8>{});
}

// Runtime atom-column dispatch (ac < 2 * NBLK).
template <int D, bool KEY>
__device__ __forceinline__ void lift_col_rt(int ac, const float (&x)[D], uint8_t *tile_col,
                                            int t) {
    switch (ac) {
        case 0: lift_col<D, KEY, 0>(x, tile_col, t); break;
        case 1: lift_col<D, KEY, 1>(x, tile_col, t); break;
        case 2: lift_col<D, KEY, 2>(x, tile_col, t); break;
        case 3: lift_col<D, KEY, 3>(x, tile_col, t); break;
        case 4: lift_col<D, KEY, 4>(x, tile_col, t); break;
        case 5: lift_col<D, KEY, 5>(x, tile_col, t); break;
        case 6: lift_col<D, KEY, 6>(x, tile_col, t); break;
        case 7: lift_col<D, KEY, 7>(x, tile_col, t); break;
        case 8: lift_col<D, KEY, 8>(x, tile_col, t); break;
        case 9: lift_col<D, KEY, 9>(x, tile_col, t); break;
        default: break;
    }
}

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

template <int D, bool KEY, int AC, int... CH>
__device__ __forceinline__ void lift_col2_impl(const PackedRow<D> &r, uint8_t *row, int t7,
                                               std::integer_sequence<int, CH...>) {
    (lift_chunk2<D, KEY, 32 * AC + 4 * CH>(r, row + ((CH ^ t7) << 4)), ...);
}

template <int D, bool KEY, int AC>
__device__ __forceinline__ void lift_col2(const PackedRow<D> &r, uint8_t *tile_col, int t) {
    lift_col2_impl<D, KEY, AC>(r, tile_col + (t >> 3) * 1024 + (t & 7) * 128, t & 7,
                               std::make_integer_sequence<int, 8>{});
}

template <int D, bool KEY>
__device__ __forceinline__ void lift_col2_rt(int ac, const PackedRow<D> &r, uint8_t *tile_col,
                                             int t) {
    switch (ac) {
        case 0: lift_col2<D, KEY, 0>(r, tile_col, t); break;
        case 1: lift_col2<D, KEY, 1>(r, tile_col, t); break;
        case 2: lift_col2<D, KEY, 2>(r, tile_col, t); break;
        case 3: lift_col2<D, KEY, 3>(r, tile_col, t); break;
        case 4: lift_col2<D, KEY, 4>(r, tile_col, t); break;
        case 5: lift_col2<D, KEY, 5>(r, tile_col, t); break;
        case 6: lift_col2<D, KEY, 6>(r, tile_col, t); break;
        case 7: lift_col2<D, KEY, 7>(r, tile_col, t); break;
        case 8: lift_col2<D, KEY, 8>(r, tile_col, t); break;
        case 9: lift_col2<D, KEY, 9>(r, tile_col, t); break;
        default: break;
    }
}

// Row `tok` of a [BH][T][D] bf16 tensor as fp32 (zeros past T).
template <int D>
__device__ __forceinline__ void load_row(const bf16 *__restrict__ p, int bh, int T, int tok,
                                         float (&x)[D]) {
    if (tok < T) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p + ((size_t)bh * T + tok) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 u = __ldg(src + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * c + 2 * e] = __uint_as_float(w[e] << 16);
                x[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < D; ++i) x[i] = 0.f;
    }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void flag_error(int code) { atomicOr(&g_tc_error, code); }

// ================================================================= kernel 1
// Segment state: S_seg[blk] = sum over the segment's tokens of psi_k(k)[blk] v^T
// (128 features x DV, fp32 in TMEM), and for blk 0 also G_seg = K^T K.
template <int D, int DV>
__global__ void __launch_bounds__(128, 2)
seg_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const bf16 *__restrict__ k, float *__restrict__ seg, int T, int NCt, int Lc,
                 int G) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32, "layouts below are written for d = 32, dv = 64");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    constexpr int kStage = C::QK_TILE + C::V_TILE;
    uint8_t *phiK = sm + 2 * kStage;
    __shared__ __align__(8) uint64_t bar_tile[2];
    __shared__ __align__(8) uint64_t bar_mma;
    __shared__ uint32_t tmem_base;

    const int blk = blockIdx.x, g = blockIdx.y, bh = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;

    if (tid == 0) {
        mbar_init(&bar_tile[0], 1);
        mbar_init(&bar_tile[1], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base, tG = tmem_base + 64;
    constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);
    constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);

    auto issue_tile = [&](int i) {
        const int st = i & 1;
        uint8_t *tk = sm + st * kStage, *tv = tk + C::QK_TILE;
        const int t0 = (c0 + i) * kTile;
        mbar_arrive_expect_tx(&bar_tile[st], C::V_TILE + (blk == 0 ? C::QK_TILE : 0));
        if (blk == 0) tma_load_3d(tk, &tm_k, 0, t0, bh, &bar_tile[st]);
        tma_load_3d(tv, &tm_v, 0, t0, bh, &bar_tile[st]);
    };
    if (tid == 0) {
        issue_tile(0);
        if (nch > 1) issue_tile(1);
    }

    bool ok = true;
    int issued = 0;
#pragma unroll 1
    for (int i = 0; i < nch; ++i) {
        const int st = i & 1;
        if (i >= 1) {
            ok = ok && mbar_wait(&bar_mma, (i - 1) & 1);     // chunk i-1's MMAs done
            if (tid == 0 && ok && i + 1 < nch) issue_tile(i + 1);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float x[D];
            load_row<D>(k, bh, T, (c0 + i) * kTile + tid, x);
            lift_col_rt<D, true>(2 * blk + h, x, phiK + h * 16384, tid);
            asm volatile("" ::: "memory");
        }
        fence_proxy_async_smem();
        ok = ok && mbar_wait(&bar_tile[st], (i >> 1) & 1);
        tc_fence_before();
        ok = __syncthreads_and(ok);
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) {
            const uint32_t tv = smem_u32(sm + st * kStage + C::QK_TILE);
            const uint32_t pk = smem_u32(phiK);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks) {
                const uint64_t a = smem_desc(pk + ks * 2048, 16384, 1024, kSw128);
                const uint64_t b = smem_desc(tv + ks * 2048, 16384, 1024, kSw128);
                mma_ss(tS, a, b, kIdState, (i > 0 || ks > 0) ? 1u : 0u);
            }
            if (blk == 0) {
                const uint32_t tk = smem_u32(sm + st * kStage);
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    const uint64_t a = smem_desc(tk + ks * 1024, 8192, 512, kSw64);
                    mma_ss(tG, a, a, kIdGram, (i > 0 || ks > 0) ? 1u : 0u);
                }
            }
            mma_commit(&bar_mma);
        }
        ++issued;
    }
    if (issued > 0) ok = mbar_wait(&bar_mma, (issued - 1) & 1) && ok;
    tc_fence_after();
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == 0) flag_error(1);
    } else {
        // state rows: TMEM lane = feature (blk*128 + lane), 64 fp32 columns
        float *dst = seg + ((size_t)bh * G + g) * C::E + (size_t)(blk * 128 + warp * 32 + lane) * DV;
        const uint32_t lrow = (uint32_t)(warp * 32) << 16;
#pragma unroll
        for (int c = 0; c < DV; c += 16) {
            uint32_t r[16];
            tmem_ld16(tS + lrow + c, r);
            float4 *d4 = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                d4[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                    __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
        }
        if (blk == 0 && warp == 0) {   // Gram rows 0..D-1 live in lanes 0..D-1
            float *gd = seg + ((size_t)bh * G + g) * C::E + (size_t)C::NBLK * 128 * DV +
                        (size_t)lane * D;
#pragma unroll
            for (int c = 0; c < D; c += 16) {
                uint32_t r[16];
                tmem_ld16(tG + c, r);
                float4 *d4 = reinterpret_cast<float4 *>(gd + c);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    d4[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                        __uint_as_float(r[4 * e + 2]),
                                        __uint_as_float(r[4 * e + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 128);
}

// ================================================================= kernel 3
// Segment output: walk the segment's chunks with the running state in TMEM.
template <int D, int DV>
__global__ void __launch_bounds__(256, 1)
seg_output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const bf16 *__restrict__ q,
                  const bf16 *__restrict__ k, bf16 *__restrict__ out,
                  const float *__restrict__ seg, int T, int NCt, int Lc, int G) {
    using C = Cfg<D, DV>;
    static_assert(DV == 64 && D == 32, "layouts below are written for d = 32, dv = 64");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    constexpr int kStage = 2 * C::QK_TILE + C::V_TILE;     // Q, K, V tiles of one chunk
    uint8_t *phiQ = sm + 2 * kStage;                         // [2][32 KB]; phiQ[1] also holds P
    uint8_t *phiK = phiQ + 2 * 32768;                        // [2][32 KB]
    uint8_t *spre = phiK + 2 * 32768;                        // 16 KB: S_pre block, bf16
    uint8_t *gram = spre + 16384;                            // 2 KB: G_pre, bf16, SW64
    __shared__ __align__(8) uint64_t bar_tile[2];
    __shared__ __align__(8) uint64_t bar_qk, bar_pv;
    __shared__ __align__(8) uint64_t bar_blk[2];
    __shared__ uint32_t tmem_base;
    __shared__ float dpart[2][kTile];

    const int g = blockIdx.x, bh = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;          // TMEM lane / tile row owned by this thread
    const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
    const int c0 = g * Lc;
    const int nch = min(NCt, c0 + Lc) - c0;

    if (tid == 0) {
        mbar_init(&bar_tile[0], 1);
        mbar_init(&bar_tile[1], 1);
        mbar_init(&bar_qk, 1);
        mbar_init(&bar_pv, 1);
        mbar_init(&bar_blk[0], 1);
        mbar_init(&bar_blk[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;          // [NBLK][DV] fp32 running state
    const uint32_t tG = tmem_base + 320;    // D cols: running Gram (lanes 0..D-1)
    const uint32_t tQG = tmem_base + 352;   // D cols: Q G_pre
    const uint32_t tX = tmem_base + 384;    // 128 cols: Q K^T, then the output accumulator

    // ---- initial state: exclusive prefix of the segment states (zero for g == 0)
    {
        const float *pre = seg + ((size_t)bh * G + g) * C::E;
        for (int blk = 0; blk < C::NBLK; ++blk) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint32_t r[8];
                if (g > 0) {
                    const float4 *s4 = reinterpret_cast<const float4 *>(
                        pre + (size_t)(blk * 128 + row) * DV + half * 32 + c);
                    const float4 a = s4[0], b = s4[1];
                    r[0] = __float_as_uint(a.x); r[1] = __float_as_uint(a.y);
                    r[2] = __float_as_uint(a.z); r[3] = __float_as_uint(a.w);
                    r[4] = __float_as_uint(b.x); r[5] = __float_as_uint(b.y);
                    r[6] = __float_as_uint(b.z); r[7] = __float_as_uint(b.w);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = 0u;
                }
                tmem_st8(tS + lrow + blk * DV + half * 32 + c, r);
            }
        }
        if (quarter == 0) {   // Gram rows i = lane, columns 16*half .. 16*half+15
            float gv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                gv[e] = g > 0 ? pre[(size_t)C::NBLK * 128 * DV + lane * D + half * 16 + e] : 0.f;
#pragma unroll
            for (int c = 0; c < 16; c += 8) {
                uint32_t r[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(gv[c + e]);
                tmem_st8(tG + lrow + half * 16 + c, r);
            }
            // bf16 copy for the Q G MMA: [D rows][D] K-major, 64-byte swizzle
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int chunk = 2 * half + cc;
                uint4 v;
                v.x = pack_bf16(gv[8 * cc + 0], gv[8 * cc + 1]);
                v.y = pack_bf16(gv[8 * cc + 2], gv[8 * cc + 3]);
                v.z = pack_bf16(gv[8 * cc + 4], gv[8 * cc + 5]);
                v.w = pack_bf16(gv[8 * cc + 6], gv[8 * cc + 7]);
                *reinterpret_cast<uint4 *>(gram + (lane >> 3) * 512 + (lane & 7) * 64 +
                                           ((chunk ^ ((lane >> 1) & 3)) << 4)) = v;
            }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    auto issue_tile = [&](int i) {
        const int st = i & 1;
        uint8_t *tq = sm + st * kStage;
        const int t0 = (c0 + i) * kTile;
        mbar_arrive_expect_tx(&bar_tile[st], kStage);
        tma_load_3d(tq, &tm_q, 0, t0, bh, &bar_tile[st]);
        tma_load_3d(tq + C::QK_TILE, &tm_k, 0, t0, bh, &bar_tile[st]);
        tma_load_3d(tq + 2 * C::QK_TILE, &tm_v, 0, t0, bh, &bar_tile[st]);
    };
    if (tid == 0) {
        issue_tile(0);
        if (nch > 1) issue_tile(1);
    }

    constexpr int kEvenBlocks = (C::NBLK + 1) / 2, kOddBlocks = C::NBLK / 2;
    constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
    constexpr uint32_t kIdQG = idesc_bf16(128, D, false, false);
    constexpr uint32_t kIdGram = idesc_bf16(128, D, true, true);
    constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
    constexpr uint32_t kIdState = idesc_bf16(128, DV, true, true);

    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < nch && ok; ++i) {
        const int st = i & 1;
        const int t0 = (c0 + i) * kTile;
        uint8_t *tq = sm + st * kStage;
        uint8_t *tk = tq + C::QK_TILE;
        uint8_t *tv = tk + C::QK_TILE;
        ok = mbar_wait(&bar_tile[st], (i >> 1) & 1);
        if (tid == 0 && ok) {
            const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), ag = smem_u32(gram);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                mma_ss(tX, smem_desc(aq + ks * 32, 16, 512, kSw64),
                       smem_desc(ak + ks * 32, 16, 512, kSw64), kIdQK, ks > 0);
                mma_ss(tQG, smem_desc(aq + ks * 32, 16, 512, kSw64),
                       smem_desc(ag + ks * 32, 16, 512, kSw64), kIdQG, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks) {
                const uint64_t a = smem_desc(ak + ks * 1024, 8192, 512, kSw64);
                mma_ss(tG, a, a, kIdGram, 1u);
            }
            mma_commit(&bar_qk);
        }
        ok = mbar_wait(&bar_qk, i & 1) && ok;
        tc_fence_after();

        // ---- intra-chunk weights: P = (Q K^T)^2 on s <= t, bf16, into phiQ[1]
        float dacc = 0.f;
        {
            uint8_t *prow = phiQ + 32768 + half * 16384 + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c = 0; c < 64; c += 16) {
                uint32_t r[16];
                tmem_ld16(tX + lrow + half * 64 + c, r);
                float w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int s = half * 64 + c + e;
                    const float xv = __uint_as_float(r[e]);
                    w[e] = (s <= row) ? xv * xv : 0.f;
                    dacc += w[e];
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int chunk = (c >> 3) + h2;
                    uint4 v;
                    v.x = pack_bf16(w[8 * h2 + 0], w[8 * h2 + 1]);
                    v.y = pack_bf16(w[8 * h2 + 2], w[8 * h2 + 3]);
                    v.z = pack_bf16(w[8 * h2 + 4], w[8 * h2 + 5]);
                    v.w = pack_bf16(w[8 * h2 + 6], w[8 * h2 + 7]);
                    *reinterpret_cast<uint4 *>(prow + ((chunk ^ (row & 7)) << 4)) = v;
                }
            }
            // inter-chunk denominator: q^T G_pre q, columns 16*half.. of Q G_pre
            float xq[D];
            load_row<D>(q, bh, T, t0 + row, xq);
            uint32_t r[16];
            tmem_ld16(tQG + lrow + half * 16, r);
#pragma unroll
            for (int e = 0; e < 16; ++e) dacc = fmaf(__uint_as_float(r[e]), xq[half * 16 + e], dacc);
            dpart[half][row] = dacc;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        tc_fence_after();
        if (tid == 0 && ok) {
            const uint32_t ap = smem_u32(phiQ + 32768), bv = smem_u32(tv);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
                mma_ss(tX, smem_desc(ap + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSw128),
                       smem_desc(bv + ks * 2048, 16384, 1024, kSw128), kIdPV, ks > 0);
            mma_commit(&bar_pv);
        }

        // ---- feature blocks: O += Psi(Q)[blk] S_pre[blk];  S[blk] += Psi(K)[blk]^T V
#pragma unroll 1
        for (int blk = 0; blk < C::NBLK && ok; ++blk) {
            const int sb = blk & 1;
            // bar_blk[0] completes for even blocks, bar_blk[1] for odd ones
            auto parity = [&](int b) {
                return (uint32_t)(((b & 1) ? kOddBlocks * i + (b >> 1) : kEvenBlocks * i + (b >> 1)) & 1);
            };
            if (blk == 1) ok = mbar_wait(&bar_pv, i & 1) && ok;             // P consumed
            if (blk >= 2) ok = mbar_wait(&bar_blk[sb], parity(blk - 2)) && ok;
            {   // one row at a time; the barriers keep the two lifts from interleaving
                float x[D];
                load_row<D>(q, bh, T, t0 + row, x);
                lift_col_rt<D, false>(2 * blk + half, x, phiQ + sb * 32768 + half * 16384, row);
            }
            asm volatile("" ::: "memory");
            {
                float x[D];
                load_row<D>(k, bh, T, t0 + row, x);
                lift_col_rt<D, true>(2 * blk + half, x, phiK + sb * 32768 + half * 16384, row);
            }
            asm volatile("" ::: "memory");
            if (blk >= 1) ok = mbar_wait(&bar_blk[(blk - 1) & 1], parity(blk - 1)) && ok;
            tc_fence_after();
            {   // S_run[blk] -> S_pre (bf16, [128 features][DV], 128-byte swizzle)
                uint8_t *srow = spre + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                for (int c = 0; c < 32; c += 16) {
                    uint32_t r[16];
                    tmem_ld16(tS + lrow + blk * DV + half * 32 + c, r);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int chunk = half * 4 + (c >> 3) + h2;
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(r[8 * h2 + 0]), __uint_as_float(r[8 * h2 + 1]));
                        v.y = pack_bf16(__uint_as_float(r[8 * h2 + 2]), __uint_as_float(r[8 * h2 + 3]));
                        v.z = pack_bf16(__uint_as_float(r[8 * h2 + 4]), __uint_as_float(r[8 * h2 + 5]));
                        v.w = pack_bf16(__uint_as_float(r[8 * h2 + 6]), __uint_as_float(r[8 * h2 + 7]));
                        *reinterpret_cast<uint4 *>(srow + ((chunk ^ (row & 7)) << 4)) = v;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            ok = __syncthreads_and(ok);
            tc_fence_after();
            if (tid == 0 && ok) {
                const uint32_t aq = smem_u32(phiQ + sb * 32768), ak = smem_u32(phiK + sb * 32768);
                const uint32_t bs = smem_u32(spre), bv = smem_u32(tv);
                const int fleft = C::NF - blk * 128;
                const int ksteps = fleft >= 128 ? 8 : (fleft + 15) / 16;
                for (int ks = 0; ks < ksteps; ++ks)
                    mma_ss(tX, smem_desc(aq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSw128),
                           smem_desc(bs + ks * 2048, 16384, 1024, kSw128), kIdPV, 1u);
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ss(tS + blk * DV, smem_desc(ak + ks * 2048, 16384, 1024, kSw128),
                           smem_desc(bv + ks * 2048, 16384, 1024, kSw128), kIdState, 1u);
                mma_commit(&bar_blk[sb]);
            }
        }
        {
            constexpr int kLast = C::NBLK - 1;
            const uint32_t par = (uint32_t)((((kLast & 1) ? kOddBlocks : kEvenBlocks) * i + (kLast >> 1)) & 1);
            ok = mbar_wait(&bar_blk[kLast & 1], par) && ok;
        }
        tc_fence_after();
        ok = __syncthreads_and(ok);
        if (!ok) break;

        // ---- epilogue: O = N / D for valid rows; refresh the bf16 Gram copy
        {
            const float den = dpart[0][row] + dpart[1][row];
            const float inv = den > 0.f ? 1.f / den : 0.f;
            // tcgen05.ld is warp-collective: every lane loads, only valid rows store
            const bool valid = t0 + row < T;
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * T + t0 + row) * DV + half * 32);
#pragma unroll
            for (int c16 = 0; c16 < 2; ++c16) {
                uint32_t r[16];
                tmem_ld16(tX + lrow + half * 32 + c16 * 16, r);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(r[8 * c + 0]) * inv, __uint_as_float(r[8 * c + 1]) * inv);
                    v.y = pack_bf16(__uint_as_float(r[8 * c + 2]) * inv, __uint_as_float(r[8 * c + 3]) * inv);
                    v.z = pack_bf16(__uint_as_float(r[8 * c + 4]) * inv, __uint_as_float(r[8 * c + 5]) * inv);
                    v.w = pack_bf16(__uint_as_float(r[8 * c + 6]) * inv, __uint_as_float(r[8 * c + 7]) * inv);
                    if (valid) dst[2 * c16 + c] = v;
                }
            }
            if (quarter == 0) {
                uint32_t gr[16];
                tmem_ld16(tG + lrow + half * 16, gr);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int chunk = 2 * half + cc;
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(gr[8 * cc + 0]), __uint_as_float(gr[8 * cc + 1]));
                    v.y = pack_bf16(__uint_as_float(gr[8 * cc + 2]), __uint_as_float(gr[8 * cc + 3]));
                    v.z = pack_bf16(__uint_as_float(gr[8 * cc + 4]), __uint_as_float(gr[8 * cc + 5]));
                    v.w = pack_bf16(__uint_as_float(gr[8 * cc + 6]), __uint_as_float(gr[8 * cc + 7]));
                    *reinterpret_cast<uint4 *>(gram + (lane >> 3) * 512 + (lane & 7) * 64 +
                                               ((chunk ^ ((lane >> 1) & 3)) << 4)) = v;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0 && i + 2 < nch) issue_tile(i + 2);
    }
    if (!ok && tid == 0) flag_error(2);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 512);
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

constexpr int kSmemState = 2 * (Cfg<32, 64>::QK_TILE + Cfg<32, 64>::V_TILE) + 32768 + 1024;
constexpr int kSmemOutput =
    2 * (2 * Cfg<32, 64>::QK_TILE + Cfg<32, 64>::V_TILE) + 4 * 32768 + 16384 + 2048 + 1024;

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
            seg_state_kernel<32, 64><<<dim3(C::NBLK, p.G - 1, s.BH()), 128, kSmemState, stream>>>(
                mk, mv, (const bf16 *)k, seg, s.T, p.NCt, p.Lc, p.G);
        }
        cudaError_t e = scan_exclusive_launch(seg, s.BH(), p.G, C::E, "tc_segment_scan", stream);
        if (e != cudaSuccess) return e;
    }
    cudaFuncSetAttribute(seg_output_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemOutput);
    {
        TraceScope tr("tc_segment_output", stream);
        seg_output_kernel<32, 64><<<dim3(p.G, s.BH()), 256, kSmemOutput, stream>>>(
            mq, mk, mv, (const bf16 *)q, (const bf16 *)k, (bf16 *)out, seg, s.T, p.NCt, p.Lc, p.G);
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
