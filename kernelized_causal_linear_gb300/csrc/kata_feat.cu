// Explicit-feature tensor-core path of the chunked forward, for lift maps with
// few packed features: KATA-Sigma_g and KATA-M_g (the reduced PSD families of
// [KATA] Sec. 4.1) and the orthant map, whose psi is not a rank-one lift of one
// short vector, so the rank-one kernels (kata_tc.cu) cannot form it.
//
// With n features (n <= 192) the features themselves are small enough to write
// out, and the chunk form of Eq. 17-20 becomes three tcgen05 kernels around the
// chunk scan (Sec. 4.2), every chunk of 128 tokens independent:
//
//   feat_lift_kernel    Phi = psi(x) for every q and k row as two bf16 parts,
//                       Phi_hi = bf16(psi) and Phi_lo = bf16(psi - Phi_hi),
//                       [rows][n8] each (n8 = n rounded up to 8 for 16-byte
//                       rows), from a table of the map's features
//   feat_state_kernel   per chunk: S_loc = Phi_K^T V (MMA, 128-feature blocks)
//                       and z_loc = Phi_K^T 1 (column sums), one fp32 record
//                       [n][65] per chunk                            [Eq. 17]
//   exclusive scan      over the chunks' records (scan_exclusive_launch)
//   feat_output_kernel  per chunk: X = Phi_Q Phi_K^T (MMA, from the hi and lo
//                       parts), P = X masked to s <= t (no square: X already
//                       holds psi(q).psi(k)), N = Phi_Q S_pre + P V (MMA),
//                       D = Phi_Q . z_pre + P 1, O = N / D      [Eq. 18-20]
//
// The record scan moves n * 65 * 4 bytes per chunk three times, i.e. about
// 6 n bytes per token and head: 0.8 KB at n = 136, small against the kernels'
// work, which is why this path needs no segments.  Operands are bf16,
// accumulation fp32 in TMEM, as on the other tensor paths.  The intra-chunk
// weights need more than one bf16 feature part: rounding a feature to bf16 errs
// by 2^-9 of the feature, and the weight psi(q).psi(k) is a sum of signed
// products that can be far smaller than |psi(q)| |psi(k)| (near-orthogonal
// blocks), so bf16 features leave weights with large relative errors where few
// tokens are averaged (3e-2 of the output on the first rows at d = 16).  X is
// therefore Phi_Q,hi Phi_K,hi^T + Phi_Q,hi Phi_K,lo^T + Phi_Q,lo Phi_K,hi^T (error
// ~2^-16 of the features).  The state and the inter-chunk term, sums over many
// tokens, take Phi_hi alone, as the rank-one path rounds its lifted features.
#include "kata_feat.cuh"
#include "kata_map.cuh"
#include "kata_tc_common.cuh"

namespace kata {
namespace {

constexpr int kAtom = 64;                   // features per 128-byte swizzle atom (one TMA box)
constexpr int kAtomBytes = kTile * 128;     // one atom of a 128-row tile: 16 KB
constexpr int kDv = 64;
constexpr int kW = kDv + 1;                 // record row: 64 state columns and z

__device__ int g_feat_error = 0;   // sticky: bounded waits that expired

struct FeatPlan {
    int n, n8, nbox, nb, kst, NC;
};

FeatPlan feat_plan(const FwdShape &s, const MapSpec &map) {
    FeatPlan p;
    p.n = map.n(s.d);
    p.n8 = (p.n + 7) & ~7;
    p.nbox = (p.n + kAtom - 1) / kAtom;   // 64-feature boxes of a tile
    p.nb = (p.n + 127) / 128;             // 128-feature state blocks (MMA M)
    p.kst = (p.n + 15) / 16;              // 16-feature K steps of the Phi_Q products
    p.NC = (s.T + kTile - 1) / kTile;
    return p;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

// ---------------------------------------------------------------- lift
// One packed feature as a table entry (Feat of kata_map.cuh without its term
// count, which the kernel takes as a template argument).
struct FeatEntry {
    int16_t i0, j0, step, pad;
    float cf, add, scl;
};

// TERMS < 0: the orthant map's max(x[i0], 0) + add; else cf (add + scl sum of
// TERMS products x[i0 + a step] x[j0 + a step]).
template <int TERMS>
__device__ __forceinline__ float feat_eval(const FeatEntry &e, const float *x) {
    if constexpr (TERMS < 0) {
        return fmaxf(x[e.i0], 0.f) + e.add;
    } else {
        float s = 0.f;
#pragma unroll
        for (int a = 0; a < TERMS; ++a) s = fmaf(x[e.i0 + a * e.step], x[e.j0 + a * e.step], s);
        return e.cf * fmaf(e.scl, s, e.add);
    }
}

constexpr int kLiftThreads = 256;
constexpr int kLiftRows = 64;   // rows per block step

// psi of every row of x [rows][d] into phi [rows][n8] (entries n .. n8-1 zero).
// Each block builds the map's feature table once, then walks blocks of 64 rows:
// the rows are staged in shared memory as fp32 (stride d + 1), and the block's
// (row, feature pair) items are dealt to threads in output order, so that a
// warp's 4-byte stores are contiguous.
// The bf16 pair (a, b) as hi = bf16(a, b) and lo = bf16(a - hi.a, b - hi.b).
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(a, b);
    lo = pack_bf16(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
}

template <int TERMS>
__global__ void __launch_bounds__(kLiftThreads)
feat_lift_kernel(const bf16 *__restrict__ x, bf16 *__restrict__ phi, bf16 *__restrict__ phi_lo,
                 int64_t rows, int d, int n, int n8, MapSpec mp) {
    __shared__ FeatEntry tab[kFeatMax];
    __shared__ float xs[kLiftRows * 65];
    for (int f = threadIdx.x; f < n8; f += blockDim.x) {
        FeatEntry e{0, 0, 0, 0, 0.f, 0.f, 0.f};
        if (f < n) {
            const Feat ft = map_feature(f, d, mp);
            e = FeatEntry{(int16_t)ft.i0, (int16_t)ft.j0, (int16_t)ft.step, 0, ft.cf, ft.add, ft.scl};
        }
        tab[f] = e;
    }
    const int P = n8 / 2;                          // feature pairs per row
    const int dq = kLiftThreads / P, dr = kLiftThreads % P;   // item stride in (rows, pairs)
    for (int64_t r0 = (int64_t)blockIdx.x * kLiftRows; r0 < rows; r0 += (int64_t)gridDim.x * kLiftRows) {
        const int nr = (int)(rows - r0 < kLiftRows ? rows - r0 : kLiftRows);
        __syncthreads();   // the table is built / the previous rows are used
        for (int e = threadIdx.x; e < nr * d / 2; e += blockDim.x) {
            const __nv_bfloat162 p2 = reinterpret_cast<const __nv_bfloat162 *>(x + r0 * d)[e];
            const int row = (2 * e) / d, col = (2 * e) % d;
            xs[row * (d + 1) + col] = __low2float(p2);
            xs[row * (d + 1) + col + 1] = __high2float(p2);
        }
        __syncthreads();
        uint32_t *dst = reinterpret_cast<uint32_t *>(phi + r0 * n8);
        uint32_t *dlo = reinterpret_cast<uint32_t *>(phi_lo + r0 * n8);
        int row = threadIdx.x / P, p = threadIdx.x % P;
        for (int i = threadIdx.x; i < nr * P; i += kLiftThreads) {
            const float *xr = xs + row * (d + 1);
            split_pair(feat_eval<TERMS>(tab[2 * p], xr), feat_eval<TERMS>(tab[2 * p + 1], xr), dst[i], dlo[i]);
            row += dq;
            p += dr;
            if (p >= P) {
                p -= P;
                ++row;
            }
        }
    }
}

// psi of a row of x with the map fixed at compile time: KIND 1 the rank-one
// lift of each of the G blocks of width D / G, KIND 2 the Sigma_G matrix
// eps I + scl sum_a x_a x_a^T; packed row-major over the upper triangle (block
// by block for KIND 1), sqrt(2) off the diagonal, the features of kata_map.cuh's
// map_feature in the same order.  One thread per row: the row sits in registers
// and every feature's indices are constants, so a feature costs its products
// and nothing else.  Used for Sigma_G, G >= 2, where the products dominate.
// The block's 128 rows of both parts are staged in shared memory ([2][128][n8]
// bf16, dynamic) and copied out in order.
template <int KIND, int D, int G>
__global__ void __launch_bounds__(128)
feat_lift_rows_kernel(const bf16 *__restrict__ x, bf16 *__restrict__ phi, bf16 *__restrict__ phi_lo,
                      int64_t rows, int n8, float eps, float scl) {
    constexpr int M = D / G;
    constexpr int NBLK = KIND == 1 ? G : 1;
    extern __shared__ uint4 stage[];
    const int w8 = n8 / 8;                          // 16-byte words per row
    const int64_t r0 = (int64_t)blockIdx.x * blockDim.x;
    const int nr = (int)(rows - r0 < (int64_t)blockDim.x ? rows - r0 : (int64_t)blockDim.x);
    const int64_t r = r0 + threadIdx.x;
    if (threadIdx.x < nr) {
    float xv[D];
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 u = src[c];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            xv[8 * c + 2 * e] = __uint_as_float(w[e] << 16);
            xv[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
    uint4 *dst = stage + threadIdx.x * w8;
    uint4 *dlo = stage + (blockDim.x + threadIdx.x) * w8;
    uint32_t wb[4] = {0u, 0u, 0u, 0u}, wl[4] = {0u, 0u, 0u, 0u};
    float lo = 0.f;
    int f = 0;
#pragma unroll
    for (int b = 0; b < NBLK; ++b)
#pragma unroll
        for (int i = 0; i < M; ++i)
#pragma unroll
            for (int j = i; j < M; ++j) {
                float v;
                if constexpr (KIND == 2) {
                    float acc = 0.f;
#pragma unroll
                    for (int a = 0; a < G; ++a) acc = fmaf(xv[a * M + i], xv[a * M + j], acc);
                    v = fmaf(scl, acc, i == j ? eps : 0.f);
                } else {
                    v = xv[b * M + i] * xv[b * M + j];
                }
                if (i != j) v *= kSqrt2;
                if ((f & 1) == 0)
                    lo = v;
                else
                    split_pair(lo, v, wb[(f >> 1) & 3], wl[(f >> 1) & 3]);
                if ((f & 7) == 7) {
                    dst[f >> 3] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                    dlo[f >> 3] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
                ++f;
            }
    if ((f & 7) != 0) {   // the last word group, zero past n
        if (f & 1) split_pair(lo, 0.f, wb[(f >> 1) & 3], wl[(f >> 1) & 3]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k >= (((f + 1) >> 1) & 3) && (((f + 1) >> 1) & 3) != 0) wb[k] = wl[k] = 0u;
        dst[f >> 3] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        dlo[f >> 3] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
    }
    __syncthreads();
    uint4 *gh = reinterpret_cast<uint4 *>(phi + r0 * n8), *gl = reinterpret_cast<uint4 *>(phi_lo + r0 * n8);
    for (int i = threadIdx.x; i < nr * w8; i += blockDim.x) {
        gh[i] = stage[i];
        gl[i] = stage[blockDim.x * w8 + i];
    }
}

// Feature f of token row t in a TMA tile of 64-feature atoms, 128-byte swizzle.
__device__ __forceinline__ const uint8_t *tile_elem(const uint8_t *tile, int t, int f) {
    const int a = f / kAtom, col = f % kAtom;
    return tile + a * kAtomBytes + t * 128 + ((((col >> 3) ^ (t & 7))) << 4) + (col & 7) * 2;
}

// ---------------------------------------------------------------- chunk state
// One CTA per (chunk c, head bh), four warps.  Thread 0 loads the chunk's Phi_K
// tile (nbox boxes) and V tile and issues S_blk(b) = Phi_K[:, 128b ..]^T V for
// each block b (A MN-major: features contiguous within an atom, atoms 16 KB
// apart; B MN-major).  The state block's rows are TMEM lanes: warp w writes
// features 128 b + 32 w + lane of the record; z comes from column sums of the
// tile on the CUDA cores.  Atoms of the last block that no box fills are zeroed
// (the MMA reads all 128 rows of M).
__global__ void __launch_bounds__(128, 1)
feat_state_kernel(const __grid_constant__ CUtensorMap tm_pk, const __grid_constant__ CUtensorMap tm_v,
                  float *__restrict__ rec, int NC, int n, int nbox, int nb, uint32_t tcols) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tpk = sm;                              // 2 nb atoms: Phi_K [tokens][features]
    uint8_t *tv = sm + 2 * nb * kAtomBytes;         // V tile [tokens][64]
    __shared__ __align__(8) uint64_t full, done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float zsum[kFeatMax];

    const int c = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Sync sy{&abort_flag};

    for (int e = threadIdx.x; e < (2 * nb - nbox) * kAtomBytes / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(tpk + nbox * kAtomBytes)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&full, 1);
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, tcols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;

    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&full, (uint32_t)(nbox + 1) * kAtomBytes);
        for (int j = 0; j < nbox; ++j)
            tma_load_3d(tpk + j * kAtomBytes, &tm_pk, j * kAtom, c * kTile, bh, &full);
        tma_load_3d(tv, &tm_v, 0, c * kTile, bh, &full);
        if (sy.wait(&full, 0)) {
            tc_fence_after();
            constexpr uint32_t kId = idesc_bf16(128, kDv, true, true);
            const uint64_t dA = smem_desc(smem_u32(tpk), kAtomBytes, 1024, kSw128);
            const uint64_t dB = smem_desc(smem_u32(tv), kAtomBytes, 1024, kSw128);
            for (int b = 0; b < nb; ++b)
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ss(tS + b * kDv, desc_add(dA, b * 2 * kAtomBytes + ks * 2048),
                           desc_add(dB, ks * 2048), kId, ks > 0 ? 1u : 0u);
        }
        mma_commit(&done);
    }
    // z_loc = Phi_K^T 1 (rows past T are zero-filled by the TMA): thread p sums
    // the feature pair (2p, 2p + 1) over the chunk's tokens
    const bool tiles = sy.wait(&full, 0);
    for (int p = threadIdx.x; 2 * p < n; p += blockDim.x) {
        float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};
        if (tiles)
            for (int t = 0; t < kTile; t += 4)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(tile_elem(tpk, t + u, 2 * p));
                    z0[u] += __uint_as_float(w << 16);
                    z1[u] += __uint_as_float(w & 0xFFFF0000u);
                }
        zsum[2 * p] = (z0[0] + z0[1]) + (z0[2] + z0[3]);
        if (2 * p + 1 < n) zsum[2 * p + 1] = (z1[0] + z1[1]) + (z1[2] + z1[3]);
    }
    const bool ok = __all_sync(0xffffffffu, sy.wait(&done, 0));
    tc_fence_after();
    __syncthreads();   // the tiles are free: the MMAs are done and z is formed
    // the record [n][65] staged over the tiles ((2 nb + 1) x 16 KB >= 260 n
    // bytes), then written out in order
    float *stage = reinterpret_cast<float *>(sm);
    const uint32_t lsel = (uint32_t)(warp * 32) << 16;
    for (int b = 0; b < nb; ++b) {
        const int f = b * 128 + warp * 32 + lane;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tS + lsel + b * kDv + h * 32, v);
            if (f < n)
#pragma unroll
                for (int e = 0; e < 32; ++e) stage[f * kW + h * 32 + e] = ok ? __uint_as_float(v[e]) : 0.f;
        }
        if (f < n) stage[f * kW + kDv] = zsum[f];
    }
    tc_fence_before();
    __syncthreads();
    float *r = rec + ((size_t)bh * NC + c) * (size_t)n * kW;
    const int total = n * kW;
    if ((n & 3) == 0) {   // the record starts on a 16-byte boundary
        for (int i = threadIdx.x; i < total / 4; i += blockDim.x)
            reinterpret_cast<float4 *>(r)[i] = reinterpret_cast<const float4 *>(stage)[i];
    } else {
        for (int i = threadIdx.x; i < total; i += blockDim.x) r[i] = stage[i];
    }
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_feat_error, 1);
    if (warp == 0) tmem_dealloc(tmem_base, tcols);
}

// ---------------------------------------------------------------- chunk output
// One CTA per (chunk c, head bh).  Warp 4 loads the hi and lo parts of Phi_Q and
// Phi_K (nbox boxes each) and V and issues the MMAs; warps 0-3 (TMEM lane
// quarter = warp) own query rows t = 32 warp + lane:
//   1. the chunk's scanned record (rows f = tid, tid + 128) into registers;
//   2. X = Phi_Q Phi_K^T from the three hi/lo products (M = 128 queries, N = 128
//      keys, K = 16 kst); once it is done, S_pre (bf16, MN-major B, rows =
//      features, zero past n) goes into the Phi_K,lo tile and z_pre (fp32) to
//      its array;
//   3. P = X where s <= t, in bf16 back to TMEM as the A operand of P V; D += P 1;
//   4. D += Phi_Q,hi(t) . z_pre;
//   5. N = Phi_Q,hi S_pre + P V -> O = N / D (0 where D = 0).
// TMEM: X [0, 128) | N [128, 192) | P [192, 256).
__global__ void __launch_bounds__(160, 1)
feat_output_kernel(const __grid_constant__ CUtensorMap tm_pq, const __grid_constant__ CUtensorMap tm_pql,
                   const __grid_constant__ CUtensorMap tm_pk, const __grid_constant__ CUtensorMap tm_pkl,
                   const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ rec,
                   bf16 *__restrict__ out, int T, int NC, int n, int nbox, int kst) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tpq = sm;                              // nbox atoms each: Phi_Q hi, lo (K-major A)
    uint8_t *tpql = tpq + nbox * kAtomBytes;
    uint8_t *tpk = tpql + nbox * kAtomBytes;        // Phi_K hi, lo (K-major B of X)
    uint8_t *tpkl = tpk + nbox * kAtomBytes;
    uint8_t *tv = tpkl + nbox * kAtomBytes;         // V tile (MN-major B of P V)
    uint8_t *spre = tpkl;                           // S_pre (16 kst rows of 128 bytes) after X
    __shared__ __align__(8) uint64_t full, spre_full, x_full, p_full, o_full;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float zpre[kFeatMax];

    const int c = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Sync sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&full, 1);
        mbar_init(&spre_full, 4);
        mbar_init(&x_full, 1);
        mbar_init(&p_full, 4);
        mbar_init(&o_full, 1);
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tX = tmem_base, tN = tmem_base + 128, tP = tmem_base + 192;

    if (warp == 4) {
        if (elect_lane0()) {
            mbar_arrive_expect_tx(&full, (uint32_t)(4 * nbox + 1) * kAtomBytes);
            for (int j = 0; j < nbox; ++j) {
                tma_load_3d(tpq + j * kAtomBytes, &tm_pq, j * kAtom, c * kTile, bh, &full);
                tma_load_3d(tpql + j * kAtomBytes, &tm_pql, j * kAtom, c * kTile, bh, &full);
                tma_load_3d(tpk + j * kAtomBytes, &tm_pk, j * kAtom, c * kTile, bh, &full);
                tma_load_3d(tpkl + j * kAtomBytes, &tm_pkl, j * kAtom, c * kTile, bh, &full);
            }
            tma_load_3d(tv, &tm_v, 0, c * kTile, bh, &full);
            constexpr uint32_t kIdX = idesc_bf16(128, kTile, false, false);
            constexpr uint32_t kIdN = idesc_bf16(128, kDv, false, true);
            const uint64_t dQ = smem_desc(smem_u32(tpq), 16, 1024, kSw128);   // K-major A
            const uint64_t dQl = smem_desc(smem_u32(tpql), 16, 1024, kSw128);
            const uint64_t dK = smem_desc(smem_u32(tpk), 16, 1024, kSw128);   // K-major B
            const uint64_t dKl = smem_desc(smem_u32(tpkl), 16, 1024, kSw128);
            const uint64_t dS = smem_desc(smem_u32(spre), kAtomBytes, 1024, kSw128);   // MN-major B
            const uint64_t dV = smem_desc(smem_u32(tv), kAtomBytes, 1024, kSw128);     // MN-major B
            bool ok = sy.wait(&full, 0);
            if (ok) {
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    const uint32_t o = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
                    mma_ss(tX, desc_add(dQ, o), desc_add(dK, o), kIdX, ks > 0 ? 1u : 0u);
                }
                for (int ks = 0; ks < kst; ++ks) {
                    const uint32_t o = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
                    mma_ss(tX, desc_add(dQ, o), desc_add(dKl, o), kIdX, 1u);
                }
                for (int ks = 0; ks < kst; ++ks) {
                    const uint32_t o = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
                    mma_ss(tX, desc_add(dQl, o), desc_add(dK, o), kIdX, 1u);
                }
                mma_commit(&x_full);
                ok = sy.wait(&spre_full, 0);
            }
            if (ok) {
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    const uint32_t o = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
                    mma_ss(tN, desc_add(dQ, o), desc_add(dS, ks * 2048), kIdN, ks > 0 ? 1u : 0u);
                }
                ok = sy.wait(&p_full, 0);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ts(tN, tP + ks * 8, desc_add(dV, ks * 2048), kIdN, 1u);
            }
            mma_commit(&o_full);
        }
    } else {
        // 1. record rows f = tid and tid + 128 into registers (all loads issued
        //    at once; rows past n are zero)
        const float *r = rec + ((size_t)bh * NC + c) * (size_t)n * kW;
        const int f0 = threadIdx.x, f1 = threadIdx.x + 128;
        float a0[kW], a1[kW];
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            a0[j] = f0 < n ? __ldg(r + (size_t)f0 * kW + j) : 0.f;
            a1[j] = f1 < n ? __ldg(r + (size_t)f1 * kW + j) : 0.f;
        }
        // 2. after X: S_pre over the Phi_K,lo tile, z_pre
        const bool xok = __all_sync(0xffffffffu, sy.wait(&x_full, 0));
        tc_fence_after();
        auto put_row = [&](int f, const float (&a)[kW]) {
            const uint32_t srow = smem_u32(spre + (f >> 3) * 1024 + (f & 7) * 128);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                st_shared_v4(srow + ((ch ^ (f & 7)) << 4), pack_bf16(a[8 * ch], a[8 * ch + 1]),
                             pack_bf16(a[8 * ch + 2], a[8 * ch + 3]), pack_bf16(a[8 * ch + 4], a[8 * ch + 5]),
                             pack_bf16(a[8 * ch + 6], a[8 * ch + 7]));
            zpre[f] = a[kDv];
        };
        if (f0 < kst * 16) put_row(f0, a0);
        if (f1 < kst * 16) put_row(f1, a1);
        fence_proxy_async_smem();
        __syncwarp();
        if (elect_lane0()) mbar_arrive(&spre_full);
        asm volatile("bar.sync 1, 128;" ::: "memory");   // z_pre complete for all four warps

        // 3. P = X masked to s <= t, row sums
        const int t = warp * 32 + lane;
        const uint32_t lsel = (uint32_t)(warp * 32) << 16;
        float den = 0.f;
        if (xok) {
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 4; ++h) {   // 32 keys at a time
                uint32_t v[32];
                tmem_ld32(tX + lsel + h * 32, v);
                uint32_t pw[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int s = 32 * h + 2 * j;
                    const float w0 = s <= t ? __uint_as_float(v[2 * j]) : 0.f;
                    const float w1 = s + 1 <= t ? __uint_as_float(v[2 * j + 1]) : 0.f;
                    den += w0;
                    den += w1;
                    pw[j] = pack_bf16(w0, w1);
                }
                tmem_st16(tP + lsel + h * 16, pw);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (elect_lane0()) mbar_arrive(&p_full);

        // 4. D += Phi_Q,hi(t) . z_pre (Phi_Q read back from its tile)
        if (__all_sync(0xffffffffu, sy.wait(&full, 0))) {
            float di = 0.f;
            for (int f8 = 0; f8 < (n + 7) / 8; ++f8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(tile_elem(tpq, t, 8 * f8));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    di = fmaf(__uint_as_float(w[e] << 16), zpre[8 * f8 + 2 * e], di);
                    di = fmaf(__uint_as_float(w[e] & 0xFFFF0000u), zpre[8 * f8 + 2 * e + 1], di);
                }
            }
            den += di;
        }

        // 5. O = N / D
        const bool ook = __all_sync(0xffffffffu, sy.wait(&o_full, 0));
        tc_fence_after();
        const float inv = den > 0.f ? 1.f / den : 0.f;
        uint32_t o[kDv / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tN + lsel + h * 32, v);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                o[h * 16 + e] = pack_bf16(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
        }
        const int64_t tok = (int64_t)c * kTile + t;
        if (ook && tok < T) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)bh * T + tok) * kDv);
#pragma unroll
            for (int c8 = 0; c8 < kDv / 8; ++c8)
                dst[c8] = make_uint4(o[4 * c8], o[4 * c8 + 1], o[4 * c8 + 2], o[4 * c8 + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_feat_error, 2);
    if (warp == 4) tmem_dealloc(tmem_base, 256);
}

// TMEM of the state kernel: 64 columns per block.  Its shared memory,
// (2 nb + 1) x 16 KB, admits at most 4 and 2 CTAs per SM for nb = 1 and 2, so
// the columns they hold stay within the SM's 512.
uint32_t state_tcols(const FeatPlan &p) { return p.nb == 1 ? 64u : 128u; }
size_t state_smem(const FeatPlan &p) { return (size_t)(2 * p.nb + 1) * kAtomBytes + 1024; }
// The output kernel holds 256 TMEM columns: its shared memory is at least 80 KB so
// that no more than two CTAs share an SM.  S_pre (16 kst rows of 128 bytes <=
// 8 KB per box) lies over the Phi_K,lo tile.
size_t output_smem(const FeatPlan &p) {
    const size_t b = (size_t)(4 * p.nbox + 1) * kAtomBytes + 1024;
    return b < (size_t)80 * 1024 ? (size_t)80 * 1024 : b;
}

}  // namespace

bool feat_supported(const FwdShape &s, const MapSpec &map, int cc_major, int cc_minor) {
    return s.dtype == 1 && cc_major == 10 && cc_minor == 3 && s.dv == kDv && s.d <= 64 &&
           map.n(s.d) <= kFeatMax && encoder() != nullptr;
}

size_t feat_workspace_bytes(const FwdShape &s, const MapSpec &map) {
    const FeatPlan p = feat_plan(s, map);
    const size_t rows = (size_t)s.BH() * s.T;
    const size_t rec = (size_t)s.BH() * ((size_t)p.NC + (size_t)(p.NC / 16 + 1)) * p.n * kW;
    return 4 * round256(rows * p.n8 * sizeof(bf16)) + sizeof(float) * rec;
}

cudaError_t feat_forward(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                         void *workspace, cudaStream_t stream, const MapSpec &map,
                         const StateOut &so) {
    const FeatPlan p = feat_plan(s, map);
    const int64_t rows = (int64_t)s.BH() * s.T;
    if (rows == 0) return cudaSuccess;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t phib = round256((size_t)rows * p.n8 * sizeof(bf16));
    bf16 *phiq = reinterpret_cast<bf16 *>(ws), *phik = reinterpret_cast<bf16 *>(ws + phib);
    bf16 *phiql = reinterpret_cast<bf16 *>(ws + 2 * phib), *phikl = reinterpret_cast<bf16 *>(ws + 3 * phib);
    float *rec = reinterpret_cast<float *>(ws + 4 * phib);
    float *part_ws = rec + (size_t)s.BH() * p.NC * p.n * kW;
    const int64_t want = (rows + kLiftRows - 1) / kLiftRows;
    const unsigned blocks = (unsigned)(want < 152 * 8 ? want : 152 * 8);
    const unsigned rblocks = (unsigned)((rows + 127) / 128);
    const size_t rsmem = (size_t)2 * 128 * p.n8 * sizeof(bf16);   // both parts of 128 rows
    // products per feature: 1 for the rank-one blocks, g for Sigma_g; the orthant map
    const int terms = map.kind == 3 ? -1 : map.kind == 2 ? map.g : 1;
    // Sigma_g with g >= 2 (several products per feature) has a compile-time lift;
    // the table lift's ordered stores serve the one-product maps better
    const int key = map.kind * 10000 + s.d * 100 + map.g;
    for (int side = 0; side < 2; ++side) {
        TraceScope tr("tc_feat_lift", stream);
        const bf16 *src = (const bf16 *)(side ? k : q);
        bf16 *dstp = side ? phik : phiq, *dlop = side ? phikl : phiql;
#define KATA_LIFT_ROWS(K, DD, GG)                                                                  \
    case K * 10000 + DD * 100 + GG:                                                                \
        cudaFuncSetAttribute(feat_lift_rows_kernel<K, DD, GG>,                                     \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsmem);             \
        feat_lift_rows_kernel<K, DD, GG><<<rblocks, 128, rsmem, stream>>>(src, dstp, dlop, rows,    \
                                                                          p.n8, map.eps, map.scale); \
        continue;
        switch (key) {
            KATA_LIFT_ROWS(2, 16, 2)
            KATA_LIFT_ROWS(2, 16, 4)
            KATA_LIFT_ROWS(2, 32, 2)
            KATA_LIFT_ROWS(2, 32, 4)
            KATA_LIFT_ROWS(2, 64, 4)
            default: break;
        }
#undef KATA_LIFT_ROWS
        switch (terms) {
            case -1: feat_lift_kernel<-1><<<blocks, kLiftThreads, 0, stream>>>(src, dstp, dlop, rows, s.d, p.n, p.n8, map); break;
            case 2: feat_lift_kernel<2><<<blocks, kLiftThreads, 0, stream>>>(src, dstp, dlop, rows, s.d, p.n, p.n8, map); break;
            case 4: feat_lift_kernel<4><<<blocks, kLiftThreads, 0, stream>>>(src, dstp, dlop, rows, s.d, p.n, p.n8, map); break;
            default: feat_lift_kernel<1><<<blocks, kLiftThreads, 0, stream>>>(src, dstp, dlop, rows, s.d, p.n, p.n8, map); break;
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap mpq, mpql, mpk, mpkl, mv;
    if (!make_map(mpq, phiq, p.n8, s.T, s.BH(), kAtom) || !make_map(mpk, phik, p.n8, s.T, s.BH(), kAtom) ||
        !make_map(mpql, phiql, p.n8, s.T, s.BH(), kAtom) ||
        !make_map(mpkl, phikl, p.n8, s.T, s.BH(), kAtom) || !make_map(mv, v, kDv, s.T, s.BH()))
        return cudaErrorInvalidValue;
    cudaFuncSetAttribute(feat_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)state_smem(p));
    cudaFuncSetAttribute(feat_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)output_smem(p));
    {
        TraceScope tr("tc_feat_state", stream);
        feat_state_kernel<<<dim3(p.NC, s.BH()), 128, state_smem(p), stream>>>(
            mpk, mv, rec, p.NC, p.n, p.nbox, p.nb, state_tcols(p));
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = scan_exclusive_launch(rec, s.BH(), p.NC, (int64_t)p.n * kW, "tc_feat_scan", stream, so, kW,
                              nullptr, part_ws);
    if (e != cudaSuccess) return e;
    {
        TraceScope tr("tc_feat_output", stream);
        feat_output_kernel<<<dim3(p.NC, s.BH()), 160, output_smem(p), stream>>>(
            mpq, mpql, mpk, mpkl, mv, rec, (bf16 *)out, s.T, p.NC, p.n, p.nbox, p.kst);
    }
    return cudaGetLastError();
}

int feat_take_error() {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_feat_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (h != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_feat_error, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return -1;
        }
    }
    return h;
}

}  // namespace kata
