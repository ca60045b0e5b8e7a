// Device and host helpers shared by the tensor-core kernels (kata_tc.cu for
// d = 32, kata_tc64.cu for d = 64): the grouped feature layout and its lift,
// TMA-tile row reads, the bounded barrier wait with an abort flag, and the
// tensor-map encoder.
#pragma once

#include <cuda.h>

#include <mutex>
#include <utility>

#include "kata_internal.cuh"
#include "kata_sm100.cuh"

namespace kata {
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

// ---- lift arithmetic: one mul.rn.bf16x2 per pair of features.  A product of
// two bf16 values is exact in fp32, so every lifted entry is the correctly
// rounded bf16 of x_i x_j (times the key factor 2, which is exact).
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

constexpr uint32_t kOne2 = 0x3F803F80u;   // bf16 pair (1, 1): query factor
constexpr uint32_t kTwo2 = 0x40004000u;   // bf16 pair (2, 2): key factor off the diagonal

// A row as bf16 pairs: w[m] = (x_2m, x_2m+1).
template <int D>
struct PackedRow {
    uint32_t w[D / 2];
};

// ---- grouped feature layout (d = 32, 544 slots = 5 blocks of 128, 528 real)
// The coordinates form four groups of eight (group g = coordinates 8g..8g+7).
// Blocks 0-2 hold the 384 cross-group products as six 8 x 8 rectangles, one
// per 64-feature atom column: block 0 = (0,1) | (2,3), block 1 = (0,2) | (1,3),
// block 2 = (0,3) | (1,2).  Row a of rectangle (X,Y) is one 16-byte chunk:
// x_{8X+a} * (x_{8Y}, ..., x_{8Y+7}).  Blocks 3-4 hold the four within-group
// triangles, each packed like the full upper triangle of an 8-vector (row a:
// pairs (x_a x_J, x_a x_{J+1}) for J = a, a+2, ...; odd rows end with a zero
// pad), 20 pairs = 5 chunks per group, groups back to back: block 3 = groups
// 0, 1, 2 and chunk 0 of group 3, block 4 = chunks 1-4 of group 3.  The state
// kernel lifts every block with its own compile-time code (fewest instructions);
// the output kernel lifts every block with one rectangle and one triangle
// routine whose groups are chosen at run time (least code, since its other
// roles already fill most of the instruction cache).

// Token t's row in one 128-feature block ([128 tokens x 128 features], two
// 64-feature atom columns 16 KB apart, 128-byte swizzle): chunk position pos
// (0..15) is atom column pos / 8, chunk pos % 8, stored at chunk (pos % 8) ^ (t % 8).
struct BlockRow {
    uint32_t row;      // shared address of the row in atom column 0
    uint32_t off[8];   // byte offset of chunk c within an atom-column row: (c ^ (t % 8)) * 16
    template <int POS>
    __device__ __forceinline__ uint32_t at() const {
        return row + (POS >> 3) * 16384 + off[POS & 7];
    }
};
__device__ __forceinline__ BlockRow block_row(uint8_t *block, int t) {
    BlockRow br;
    br.row = smem_u32(block) + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) br.off[c] = (uint32_t)((c ^ (t & 7)) << 4);
    return br;
}

// Rectangle (X,Y) into chunk positions POS0 .. POS0+7; f is the side factor.
template <int X, int Y, int POS0>
__device__ __forceinline__ void lift_rect(const PackedRow<32> &r, uint32_t f, const BlockRow &br) {
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const uint32_t bc = bmul2(__byte_perm(r.w[4 * X + (a >> 1)], 0u, (a & 1) ? 0x3232 : 0x1010), f);
        const uint32_t addr = br.row + (POS0 >> 3) * 16384 + br.off[a];
        st_shared_v4(addr, bmul2(bc, r.w[4 * Y + 0]), bmul2(bc, r.w[4 * Y + 1]),
                     bmul2(bc, r.w[4 * Y + 2]), bmul2(bc, r.w[4 * Y + 3]));
    }
}

// Pair W (0..19) of group G's triangle; so[k] = (x_{2k+1}, x_{2k+2}) within the group.
template <int G, int W>
__device__ __forceinline__ uint32_t tri_word(const PackedRow<32> &r, const uint32_t (&so)[4],
                                             uint32_t f) {
    constexpr int I = Words<8>::row_of(W), J = Words<8>::col_of(W);
    const uint32_t pair = (J % 2 == 0) ? r.w[4 * G + J / 2] : so[(J - 1) / 2];
    const uint32_t bc = __byte_perm(r.w[4 * G + I / 2], 0u, (I % 2 == 0) ? 0x1010 : 0x3232);
    uint32_t bk = bmul2(bc, f);
    if constexpr (J == I) bk = __byte_perm(bc, bk, 0x7610);   // the square keeps factor 1
    return bmul2(bk, pair);
}

// Chunks CLO .. CHI-1 of group G's triangle, chunk c at position POS0 + c.
template <int G, int CLO, int CHI, int POS0, int... C>
__device__ __forceinline__ void lift_tri_impl(const PackedRow<32> &r, uint32_t f, const BlockRow &br,
                                              std::integer_sequence<int, C...>) {
    uint32_t so[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        so[k] = __byte_perm(r.w[4 * G + k], k < 3 ? r.w[4 * G + k + 1] : 0u, 0x5432);
    (st_shared_v4(br.at<POS0 + CLO + C>(), tri_word<G, 4 * (CLO + C) + 0>(r, so, f),
                  tri_word<G, 4 * (CLO + C) + 1>(r, so, f), tri_word<G, 4 * (CLO + C) + 2>(r, so, f),
                  tri_word<G, 4 * (CLO + C) + 3>(r, so, f)),
     ...);
}
template <int G, int CLO, int CHI, int POS0>
__device__ __forceinline__ void lift_tri(const PackedRow<32> &r, uint32_t f, const BlockRow &br) {
    lift_tri_impl<G, CLO, CHI, POS0>(r, f, br, std::make_integer_sequence<int, CHI - CLO>{});
}

// Lift part PART of NPARTS of block B for one token: NPARTS = 1 lifts the whole
// block; NPARTS = 2 splits the blocks so that, over the five blocks, each half
// holds 34 of the 68 16-byte chunks of a token row.
template <int B, int PART, int NPARTS>
__device__ __forceinline__ void lift_block_ct(const PackedRow<32> &r, uint32_t f, const BlockRow &br) {
    constexpr bool p0 = NPARTS == 1 || PART == 0, p1 = NPARTS == 1 || PART == 1;
    if constexpr (B < 3) {
        constexpr int X2 = B == 0 ? 2 : 1, Y2 = B == 2 ? 2 : 3;
        if constexpr (p0) lift_rect<0, B + 1, 0>(r, f, br);
        if constexpr (p1) lift_rect<X2, Y2, 8>(r, f, br);
    } else if constexpr (B == 3) {
        if constexpr (p0) {
            lift_tri<0, 0, 5, 0>(r, f, br);
            lift_tri<1, 0, 5, 5>(r, f, br);
        }
        if constexpr (p1) {
            lift_tri<2, 0, 5, 10>(r, f, br);
            lift_tri<3, 0, 1, 15>(r, f, br);
        }
    } else {
        if constexpr (p1) lift_tri<3, 1, 5, -1>(r, f, br);
    }
}

// Run-time block (and part) dispatch to the compile-time lifts above.
template <int NPARTS>
__device__ __forceinline__ void lift_block(int b, int part, const PackedRow<32> &r, uint32_t f,
                                           const BlockRow &br) {
    switch (b * 2 + (NPARTS == 1 ? 0 : part)) {
        case 0: lift_block_ct<0, 0, NPARTS>(r, f, br); break;
        case 1: lift_block_ct<0, 1, NPARTS>(r, f, br); break;
        case 2: lift_block_ct<1, 0, NPARTS>(r, f, br); break;
        case 3: lift_block_ct<1, 1, NPARTS>(r, f, br); break;
        case 4: lift_block_ct<2, 0, NPARTS>(r, f, br); break;
        case 5: lift_block_ct<2, 1, NPARTS>(r, f, br); break;
        case 6: lift_block_ct<3, 0, NPARTS>(r, f, br); break;
        case 7: lift_block_ct<3, 1, NPARTS>(r, f, br); break;
        case 8: lift_block_ct<4, 0, NPARTS>(r, f, br); break;
        case 9: lift_block_ct<4, 1, NPARTS>(r, f, br); break;
        default: break;
    }
}

// ---- the same layout lifted into registers, half a block (one 64-feature atom
// column, 32 bf16 pairs) at a time: word 4p + m of half h is the pair m of chunk
// position 8h + p.  The pair kernel stores these words in TMEM as the A operand
// of its output MMAs (token t = TMEM lane t).

// Rectangle (X,Y) into words 0..31 (chunk positions 0..7 of the half).
template <int X, int Y>
__device__ __forceinline__ void rect_regs(const PackedRow<32> &r, uint32_t f, uint32_t (&w)[32]) {
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const uint32_t bc = bmul2(__byte_perm(r.w[4 * X + (a >> 1)], 0u, (a & 1) ? 0x3232 : 0x1010), f);
#pragma unroll
        for (int m = 0; m < 4; ++m) w[4 * a + m] = bmul2(bc, r.w[4 * Y + m]);
    }
}

// Chunks CLO .. CHI-1 of group G's triangle at half positions P0 .. P0+CHI-CLO-1.
template <int G, int CLO, int CHI, int P0, int... C>
__device__ __forceinline__ void tri_regs_impl(const PackedRow<32> &r, uint32_t f, uint32_t (&w)[32],
                                              std::integer_sequence<int, C...>) {
    uint32_t so[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        so[k] = __byte_perm(r.w[4 * G + k], k < 3 ? r.w[4 * G + k + 1] : 0u, 0x5432);
    ((w[4 * (P0 + C) + 0] = tri_word<G, 4 * (CLO + C) + 0>(r, so, f),
      w[4 * (P0 + C) + 1] = tri_word<G, 4 * (CLO + C) + 1>(r, so, f),
      w[4 * (P0 + C) + 2] = tri_word<G, 4 * (CLO + C) + 2>(r, so, f),
      w[4 * (P0 + C) + 3] = tri_word<G, 4 * (CLO + C) + 3>(r, so, f)),
     ...);
}
template <int G, int CLO, int CHI, int P0>
__device__ __forceinline__ void tri_regs(const PackedRow<32> &r, uint32_t f, uint32_t (&w)[32]) {
    tri_regs_impl<G, CLO, CHI, P0>(r, f, w, std::make_integer_sequence<int, CHI - CLO>{});
}

// Half HALF of block B (positions 8 HALF .. 8 HALF + 7); block 4 has only
// positions 0..3 (words 0..15 of half 0; the rest are left unset).
template <int B, int HALF>
__device__ __forceinline__ void lift_half_regs(const PackedRow<32> &r, uint32_t f, uint32_t (&w)[32]) {
    if constexpr (B < 3) {
        constexpr int X2 = B == 0 ? 2 : 1, Y2 = B == 2 ? 2 : 3;
        if constexpr (HALF == 0) rect_regs<0, B + 1>(r, f, w);
        else rect_regs<X2, Y2>(r, f, w);
    } else if constexpr (B == 3) {
        if constexpr (HALF == 0) {
            tri_regs<0, 0, 5, 0>(r, f, w);   // positions 0-4
            tri_regs<1, 0, 3, 5>(r, f, w);   // positions 5-7
        } else {
            tri_regs<1, 3, 5, 0>(r, f, w);   // positions 8-9
            tri_regs<2, 0, 5, 2>(r, f, w);   // positions 10-14
            tri_regs<3, 0, 1, 7>(r, f, w);   // position 15
        }
    } else {
        if constexpr (HALF == 0) tri_regs<3, 1, 5, 0>(r, f, w);   // positions 0-3
    }
}

// The 4 words (8 features) of chunk position POS of block B, f the side factor.
template <int B, int POS>
__device__ __forceinline__ void chunk_words(const PackedRow<32> &r, uint32_t f, uint32_t *w4) {
    if constexpr (B < 3) {
        constexpr int X = POS < 8 ? 0 : (B == 0 ? 2 : 1);
        constexpr int Y = POS < 8 ? B + 1 : (B == 2 ? 2 : 3);
        constexpr int a = POS & 7;
        const uint32_t bc = bmul2(__byte_perm(r.w[4 * X + (a >> 1)], 0u, (a & 1) ? 0x3232 : 0x1010), f);
#pragma unroll
        for (int m = 0; m < 4; ++m) w4[m] = bmul2(bc, r.w[4 * Y + m]);
    } else {
        constexpr int G = B == 4 ? 3 : (POS < 15 ? POS / 5 : 3);
        constexpr int c = B == 4 ? POS + 1 : (POS < 15 ? POS % 5 : 0);
        uint32_t so[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            so[k] = __byte_perm(r.w[4 * G + k], k < 3 ? r.w[4 * G + k + 1] : 0u, 0x5432);
        w4[0] = tri_word<G, 4 * c + 0>(r, so, f);
        w4[1] = tri_word<G, 4 * c + 1>(r, so, f);
        w4[2] = tri_word<G, 4 * c + 2>(r, so, f);
        w4[3] = tri_word<G, 4 * c + 3>(r, so, f);
    }
}

// Words of chunk positions 4Q .. 4Q+3 of block B (16 words).
template <int B, int Q>
__device__ __forceinline__ void lift_quarter_regs(const PackedRow<32> &r, uint32_t f, uint32_t (&w)[16]) {
    chunk_words<B, 4 * Q + 0>(r, f, w + 0);
    chunk_words<B, 4 * Q + 1>(r, f, w + 4);
    chunk_words<B, 4 * Q + 2>(r, f, w + 8);
    chunk_words<B, 4 * Q + 3>(r, f, w + 12);
}

// ---- the same layout lifted with the groups chosen at run time: one copy of
// the rectangle and triangle code serves every block, which keeps the lift of
// the output kernel (whose other roles already fill most of the instruction
// cache) small.

struct Group8 {
    uint32_t w[4];   // (x_{8g+2k}, x_{8g+2k+1}), k = 0..3
};

__device__ __forceinline__ Group8 group8(const PackedRow<32> &r, int g) {
    Group8 o;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        o.w[k] = g == 0 ? r.w[k] : g == 1 ? r.w[4 + k] : g == 2 ? r.w[8 + k] : r.w[12 + k];
    return o;
}

// BlockRow with the chunk position known only at run time.
struct BlockRowRt {
    uint32_t row;   // shared address of the row in atom column 0
    uint32_t x16;   // (t % 8) * 16
    __device__ __forceinline__ uint32_t at(int pos) const {
        return row + (pos >> 3) * 16384 + (((pos & 7) << 4) ^ x16);
    }
};
__device__ __forceinline__ BlockRowRt block_row_rt(uint8_t *block, int t) {
    return BlockRowRt{smem_u32(block) + (t >> 3) * 1024 + (t & 7) * 128, (uint32_t)(t & 7) << 4};
}

// Rectangle (X,Y) into chunk positions pos0 .. pos0+7; f is the side factor.
__device__ __forceinline__ void lift_rect_rt(const Group8 &gx, const Group8 &gy, uint32_t f,
                                          const BlockRowRt &br, int pos0) {
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const uint32_t bc = bmul2(__byte_perm(gx.w[a >> 1], 0u, (a & 1) ? 0x3232 : 0x1010), f);
        st_shared_v4(br.at(pos0 + a), bmul2(bc, gy.w[0]), bmul2(bc, gy.w[1]), bmul2(bc, gy.w[2]),
                     bmul2(bc, gy.w[3]));
    }
}

// Pair W (0..19) of one group's triangle; so[k] = (x_{2k+1}, x_{2k+2}) within the group.
template <int W>
__device__ __forceinline__ uint32_t tri_word_rt(const Group8 &g, const uint32_t (&so)[4], uint32_t f) {
    constexpr int I = Words<8>::row_of(W), J = Words<8>::col_of(W);
    const uint32_t pair = (J % 2 == 0) ? g.w[J / 2] : so[(J - 1) / 2];
    const uint32_t bc = __byte_perm(g.w[I / 2], 0u, (I % 2 == 0) ? 0x1010 : 0x3232);
    uint32_t bk = bmul2(bc, f);
    if constexpr (J == I) bk = __byte_perm(bc, bk, 0x7610);   // the square keeps factor 1
    return bmul2(bk, pair);
}

template <int C>
__device__ __forceinline__ void tri_chunk_rt(const Group8 &g, const uint32_t (&so)[4], uint32_t f,
                                          const BlockRowRt &br, int c_lo, int c_hi, int pos0) {
    if (C >= c_lo && C < c_hi)
        st_shared_v4(br.at(pos0 + C), tri_word_rt<4 * C + 0>(g, so, f), tri_word_rt<4 * C + 1>(g, so, f),
                     tri_word_rt<4 * C + 2>(g, so, f), tri_word_rt<4 * C + 3>(g, so, f));
}

// Chunks c_lo .. c_hi-1 of one group's triangle, chunk c at position pos0 + c.
__device__ __forceinline__ void lift_tri_rt(const Group8 &g, uint32_t f, const BlockRowRt &br, int c_lo,
                                         int c_hi, int pos0) {
    uint32_t so[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) so[k] = __byte_perm(g.w[k], k < 3 ? g.w[k + 1] : 0u, 0x5432);
    tri_chunk_rt<0>(g, so, f, br, c_lo, c_hi, pos0);
    tri_chunk_rt<1>(g, so, f, br, c_lo, c_hi, pos0);
    tri_chunk_rt<2>(g, so, f, br, c_lo, c_hi, pos0);
    tri_chunk_rt<3>(g, so, f, br, c_lo, c_hi, pos0);
    tri_chunk_rt<4>(g, so, f, br, c_lo, c_hi, pos0);
}

// Lift the whole of block b (run time) for one token.
__device__ __forceinline__ void lift_block_rt(int b, const PackedRow<32> &r, uint32_t f,
                                              const BlockRowRt &br) {
    if (b < 3) {
#pragma unroll 1
        for (int rr = 0; rr < 2; ++rr) {
            const int X = rr == 0 ? 0 : (b == 0 ? 2 : 1);
            const int Y = rr == 0 ? b + 1 : (b == 2 ? 2 : 3);
            lift_rect_rt(group8(r, X), group8(r, Y), f, br, 8 * rr);
        }
    } else {
        // block 3: groups 0..3 (group 3 only its chunk 0); block 4: group 3, chunks 1-4
        const int g0 = b == 3 ? 0 : 3;
#pragma unroll 1
        for (int g = g0; g < 4; ++g)
            lift_tri_rt(group8(r, g), f, br, b == 3 ? 0 : 1, (b == 3 && g == 3) ? 1 : 5,
                        b == 3 ? 5 * g : -1);
    }
}

// The 4 words (8 features) of chunk position pos of block b, both chosen at run
// time: called from a rolled loop it is one small copy of code for every block,
// so that a kernel whose roles run many different loops keeps its lift code in
// the instruction cache.
__device__ __forceinline__ uint4 chunk_words_rt(int b, int pos, const PackedRow<32> &r, uint32_t f) {
    uint4 o;
    if (b < 3) {
        const int h = pos >> 3, a = pos & 7;
        const int X = h == 0 ? 0 : (b == 0 ? 2 : 1);
        const int Y = h == 0 ? b + 1 : (b == 2 ? 2 : 3);
        const Group8 gx = group8(r, X), gy = group8(r, Y);
        const uint32_t bc = bmul2(__byte_perm(gx.w[a >> 1], 0u, (a & 1) ? 0x3232 : 0x1010), f);
        o.x = bmul2(bc, gy.w[0]);
        o.y = bmul2(bc, gy.w[1]);
        o.z = bmul2(bc, gy.w[2]);
        o.w = bmul2(bc, gy.w[3]);
        return o;
    }
    const int g = b == 4 ? 3 : (pos < 15 ? pos / 5 : 3);
    const int c = b == 4 ? pos + 1 : (pos < 15 ? pos % 5 : 0);
    const Group8 gg = group8(r, g);
    uint32_t so[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) so[k] = __byte_perm(gg.w[k], k < 3 ? gg.w[k + 1] : 0u, 0x5432);
    switch (c) {
        case 0: o = make_uint4(tri_word_rt<0>(gg, so, f), tri_word_rt<1>(gg, so, f), tri_word_rt<2>(gg, so, f), tri_word_rt<3>(gg, so, f)); break;
        case 1: o = make_uint4(tri_word_rt<4>(gg, so, f), tri_word_rt<5>(gg, so, f), tri_word_rt<6>(gg, so, f), tri_word_rt<7>(gg, so, f)); break;
        case 2: o = make_uint4(tri_word_rt<8>(gg, so, f), tri_word_rt<9>(gg, so, f), tri_word_rt<10>(gg, so, f), tri_word_rt<11>(gg, so, f)); break;
        case 3: o = make_uint4(tri_word_rt<12>(gg, so, f), tri_word_rt<13>(gg, so, f), tri_word_rt<14>(gg, so, f), tri_word_rt<15>(gg, so, f)); break;
        default: o = make_uint4(tri_word_rt<16>(gg, so, f), tri_word_rt<17>(gg, so, f), tri_word_rt<18>(gg, so, f), tri_word_rt<19>(gg, so, f)); break;
    }
    return o;
}

// Coordinates (i, j), i <= j, of feature p (0..127) of block b in the grouped
// layout; false for a pad slot.  Used to export the state in the decode
// layout, whose features are in row-major upper-triangle order.
__device__ __forceinline__ bool grouped_slot_pair(int b, int p, int &i, int &j) {
    const int k = (p & 7) >> 1, hf = p & 1;
    if (b < 3) {
        const int h = p >> 6, a = (p & 63) >> 3;
        const int X = h == 0 ? 0 : (b == 0 ? 2 : 1);
        const int Y = h == 0 ? b + 1 : (b == 2 ? 2 : 3);
        i = 8 * X + a;
        j = 8 * Y + 2 * k + hf;
        return true;
    }
    const int pos = p >> 3;
    int g, c;
    if (b == 3) {
        g = pos < 15 ? pos / 5 : 3;
        c = pos < 15 ? pos % 5 : 0;
    } else {
        if (pos >= 4) return false;
        g = 3;
        c = pos + 1;
    }
    int I = 0, w = 4 * c + k;   // pair w of the triangle: row I has (9 - I) / 2 pairs
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

// Row t of a [128 x D] bf16 tile written by TMA with the swizzle matching its
// row width (32/64/128 bytes): the 16-byte chunk c of row t sits at chunk
// c ^ ((t * row_bytes >> 7) & (chunks_per_row - 1)).
// The loads are volatile: a caller releases the tile (one lane's mbarrier arrive
// after __syncwarp) right after reading its row, and the TMA may then overwrite
// it.  With plain loads, even behind a compiler memory barrier, the CTA-pair
// kernel read rows of the next tile in some runs; volatile loads keep every
// lane's reads ahead of the release.
template <int D>
__device__ __forceinline__ void tile_row_packed(const uint8_t *tile, int t, PackedRow<D> &r) {
    constexpr int RB = D * 2, CPR = RB / 16;
    const uint32_t row = smem_u32(tile + t * RB);
    const int x = (t * RB >> 7) & (CPR - 1);
#pragma unroll
    for (int c = 0; c < CPR; ++c)
        asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r.w[4 * c + 0]), "=r"(r.w[4 * c + 1]), "=r"(r.w[4 * c + 2]), "=r"(r.w[4 * c + 3])
                     : "r"(row + ((c ^ x) << 4))
                     : "memory");
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
}

// Shared abort flag: any role whose bounded wait expires sets it; every later
// wait then returns at once, so all roles drain to the final barrier.
struct Sync {
    volatile int *abort;
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t n) const {
        const uint32_t parity = n & 1u;
        if (mbar_try_wait(bar, parity)) return true;   // fast path: a completed phase
        if (*abort) return false;
        if (mbar_wait(bar, parity)) return true;
        *abort = 1;
        return false;
    }
};

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

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

// [BH][T][inner] bf16 viewed as a 3-D tensor; box = one 128-row tile of one head,
// box_inner columns wide (all of them by default; fewer to read one block of
// the columns), swizzled over its row of box_inner * 2 bytes.
bool make_map(CUtensorMap &m, const void *base, int inner, int T, int BH, int box_inner = 0) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    if (box_inner <= 0) box_inner = inner;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)T * inner * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)kTile, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const int rb = box_inner * 2;
    const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
    return enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// ---- the pair output kernel (kata_tc_pair.cu)
cudaError_t pair_output_launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                               void *out, const float *seg, int BH, int T, int NCt, int Lc, int G,
                               int m_pieces, int NR, cudaStream_t stream);

}  // namespace kata
