// Quadratic (flash-style) KATA forward on tcgen05 (bf16, sm_103a).
//
// The direct form of the method ([KATA] Sec. 2 Eq. 2 with psi the rank-one PSD
// lift, so psi(q).psi(k) = (q.k)^2; the pages' O(T^2) "flash-style" kernel):
//   w_ts = (q_t . k_s)^2 for s <= t,  o_t = sum_s w_ts v_s / sum_s w_ts.
// No state: each 128-query tile walks the key tiles j <= its own, newest
// first, with
//   S = Q K_j^T (fp32 in TMEM), P = S^2 masked (bf16 in TMEM), O += P V_j,
// and the row sums of P in registers.  The weights are non-negative, so no
// running maximum is needed (unlike softmax attention).
//
// GatedKATA (the pages' multiplicative scalar state gate, S_t = gamma_t S_{t-1} +
// psi(k_t) v_t^T) weights pair (t, s) by a_ts = prod_{r=s+1}^{t} gamma_r.  For a
// key tile j below the query tile i the product splits into three factors, each
// at most 1: c_s (gates after s to the end of tile j), M_ij (whole tiles strictly
// between) and r_t (gates from the start of tile i to t).  c_s is folded into
// the keys, K'_s = sqrt(c_s) k_s (gate_prep_kernel), so S'^2 = c_s S^2; the P
// warps multiply by r_t M_ij, M_ij kept as a running product of tile gate
// products while the tiles are walked newest first.  The diagonal tile uses
// the plain keys and a_ts = 2^(l_t - l_s) from the tile-local cumulative log2
// of the gates (clamped at 2^-126, so a zero gate stays finite).
//
// Grid (heads, query tiles): CTAs launch in order of x fastest, so the heads'
// longest tiles (most key tiles) go first and the short ones fill the tail; 320 threads:
//   warp 0: TMA (the Q tile once, then K and V tiles through two rings: a K slot
//     is free once its S MMA is done, a V slot once its P V MMA is; one thread
//     polls both rings, so a K fetch never queues behind a V slot),
//   warp 1: MMA issue (one thread),
//   warps 2-9 ("P warps", TMEM lane quarter = warp % 4, key half = (warp - 2) / 4):
//     64 keys of a query row: S -> P and a partial row sum; the epilogue O / D
//     for 32 of the output columns (the two halves' sums meet in shared memory).
//     S is released as soon as it is in registers, so the next S MMA runs while
//     P is formed.
// TMEM (256 columns, two CTAs per SM): S [0,128) | P [128,192) | O [192,256).
#include "kata_tc_common.cuh"

namespace kata {

__device__ int g_quad_error = 0;   // sticky: bounded waits that expired

namespace {

// Ring depths: as deep as lets two CTAs share an SM's shared memory (97 KB at
// d = 64, 81 KB at d = 32).
template <int D>
struct QuadCfg {
    static constexpr int KST = 3;
    static constexpr int VST = D == 64 ? 2 : 3;
    static constexpr int QK_TILE = kTile * D * 2;   // 8 or 16 KB
    static constexpr int V_TILE = kTile * 64 * 2;   // 16 KB (dv = 64)
    static constexpr int SW = D == 64 ? kSw128 : kSw64;
    static constexpr int SBO = D * 2 * 8;            // 8 rows of the swizzled tile
    static constexpr int SMEM = (1 + KST) * QK_TILE + VST * V_TILE + 1024;
};

// Packed fp32 pairs (two lanes of one 64-bit register; sm_100 family).
__device__ __forceinline__ uint64_t f2_make(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_sq(uint64_t x) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %1;" : "=l"(r) : "l"(x));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t x, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Gate inputs of the gated variant (unused otherwise).
struct GateArgs {
    const float *lam2;    // [BH][T] cumulative log2 of the gates within each 128-token tile
    const float *gtile;   // [BH][NT] product of the gates of each tile
    int normalize;        // 1: O = N / D; 0: O = N
};

// Per 128-token tile of one head: the tile-local inclusive cumulative log2 of
// the gates, the scaled keys K'_s = sqrt(c_s) k_s with c_s the product of the
// gates after s to the end of the tile, and the tile's gate product.  Tokens
// past T count as gate 1.  One thread per token for the warp-shuffle scans; the
// key rows of the tile (contiguous) are then scaled in one coalesced sweep.
template <int D>
__global__ void __launch_bounds__(kTile)
gate_prep_kernel(const bf16 *__restrict__ k, const float *__restrict__ gamma,
                 bf16 *__restrict__ kp, float *__restrict__ lam2, float *__restrict__ gtile, int T,
                 int NT) {
    __shared__ float wsum[kTile / 32], wprod[kTile / 32], scale[kTile];
    const int j = blockIdx.x, bh = blockIdx.y, i = threadIdx.x;
    const int warp = i >> 5, lane = i & 31;
    const int t = j * kTile + i;
    const bool valid = t < T;
    const float g = valid ? gamma[(size_t)bh * T + t] : 1.f;
    float x = log2f(fmaxf(g, 1.17549435e-38f));   // log2 gamma, clamped at 2^-126
    float p = g;                                  // suffix product within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        const float z = __shfl_down_sync(0xffffffffu, p, o);
        if (lane >= o) x += y;
        if (lane + o < 32) p *= z;
    }
    float after = __shfl_down_sync(0xffffffffu, p, 1);   // gates after i within the warp
    if (lane == 31) after = 1.f;
    if (lane == 31) wsum[warp] = x;
    if (lane == 0) wprod[warp] = p;
    __syncthreads();
    for (int w = 0; w < warp; ++w) x += wsum[w];
    for (int w = warp + 1; w < kTile / 32; ++w) after *= wprod[w];
    if (i == 0) gtile[(size_t)bh * NT + j] = wprod[0] * wprod[1] * wprod[2] * wprod[3];
    if (valid) lam2[(size_t)bh * T + t] = x;
    scale[i] = sqrtf(after);
    __syncthreads();
    // rows t0 .. t0 + rows - 1 of this head: D / 8 16-byte pieces per row
    const int rows = min(kTile, T - j * kTile);
    const size_t base = ((size_t)bh * T + (size_t)j * kTile) * D;
    const uint4 *src = reinterpret_cast<const uint4 *>(k + base);
    uint4 *dst = reinterpret_cast<uint4 *>(kp + base);
    constexpr int kPer = D / 8;   // 16-byte pieces per thread (one tile has kTile * D / 8)
    uint4 u[kPer];
#pragma unroll
    for (int m = 0; m < kPer; ++m) {   // every load in flight before the first store
        const int e = i + m * kTile;
        if (e < rows * kPer) u[m] = src[e];
    }
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
        const int e = i + m * kTile;
        if (e >= rows * kPer) continue;
        const float sc = scale[e / kPer];
        uint32_t *w = reinterpret_cast<uint32_t *>(&u[m]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[c]);
            w[c] = pack_bf16(__low2float(b) * sc, __high2float(b) * sc);
        }
        dst[e] = u[m];
    }
}

template <int D, bool kGated>
__global__ void __launch_bounds__(320, 2)
quad_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kp,
            const __grid_constant__ CUtensorMap tm_o, int T, int NT, GateArgs ga) {
    using C = QuadCfg<D>;
    constexpr int DV = 64;
    constexpr int kPWarps = 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *tq = sm;
    uint8_t *tk = sm + C::QK_TILE;                        // [KST][QK_TILE]
    uint8_t *tv = tk + C::KST * C::QK_TILE;               // [VST][V_TILE]
    // q_full: the Q tile landed.  k_full[s] / k_empty[s]: K slot s holds K_j (TMA
    //   bytes) / the S MMA that read it is done; v_full / v_empty likewise for V_j
    //   and the P V MMA.  s_full: S = Q K_j^T is in TMEM; s_free: the P warps have
    //   read it.  p_full: P_j is in TMEM; p_free: the P V MMA that read it is
    //   done.  o_done: every MMA is done.
    __shared__ __align__(8) uint64_t q_full, k_full[C::KST], k_empty[C::KST], v_full[C::VST],
        v_empty[C::VST], s_full, s_free, p_full, p_free, o_done, fin_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float dpart[2][kTile];   // the two key halves' row sums
    __shared__ float lamd[kTile];       // gated: cumulative log2 gates of the diagonal tile

    const int qi = NT - 1 - (int)blockIdx.y;   // longest tiles first
    const int bh = blockIdx.x;
    const int nj = qi + 1;                      // key tiles 0 .. qi
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Sync sy{&abort_flag};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&q_full, 1);
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(&s_full, 1);
        mbar_init(&s_free, kPWarps);
        mbar_init(&p_full, kPWarps);
        mbar_init(&p_free, 1);
        mbar_init(&o_done, 1);
        mbar_init(&fin_bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base, tP = tmem_base + 128, tO = tmem_base + 192;

    if (warp == 0) {
        // ================= TMA producer
        if (elect_lane0()) {
            mbar_arrive_expect_tx(&q_full, C::QK_TILE);
            tma_load_3d(tq, &tm_q, 0, qi * kTile, bh, &q_full);
            // next K tile jk and next V tile jv (iteration order: key tile qi - jk),
            // each as soon as its slot is free; the idle spins between two fetches
            // are bounded like every other wait.  Gated: scaled keys below the
            // diagonal tile.
            int jk = 0, jv = 0;
            uint32_t it = 0;
            uint64_t t0 = globaltimer();
            while (jk < nj || jv < nj) {
                bool any = false;
                if (jk < nj) {
                    const int ks = jk % C::KST, ku = jk / C::KST;
                    if (ku == 0 || mbar_test_wait(&k_empty[ks], (ku - 1) & 1)) {
                        mbar_arrive_expect_tx(&k_full[ks], C::QK_TILE);
                        tma_load_3d(tk + ks * C::QK_TILE, (kGated && jk > 0) ? &tm_kp : &tm_k, 0,
                                    (qi - jk) * kTile, bh, &k_full[ks]);
                        ++jk;
                        any = true;
                    }
                }
                if (jv < nj) {
                    const int vs = jv % C::VST, vu = jv / C::VST;
                    if (vu == 0 || mbar_test_wait(&v_empty[vs], (vu - 1) & 1)) {
                        mbar_arrive_expect_tx(&v_full[vs], C::V_TILE);
                        tma_load_3d(tv + vs * C::V_TILE, &tm_v, 0, (qi - jv) * kTile, bh, &v_full[vs]);
                        ++jv;
                        any = true;
                    }
                }
                if (any) {
                    it = 0;
                    t0 = globaltimer();
                } else if (abort_flag) {
                    break;
                } else if (++it >= kSpinLimitIters || globaltimer() - t0 > kSpinLimitNs) {
                    abort_flag = 1;
                    break;
                }
            }
        }
    } else if (warp == 1) {
        // ================= MMA issue
        if (elect_lane0()) {
            constexpr uint32_t kIdQK = idesc_bf16(128, kTile, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(128, DV, false, true);
            const uint64_t dQ = smem_desc(smem_u32(tq), 16, C::SBO, C::SW);      // K-major A
            const uint64_t dK = smem_desc(smem_u32(tk), 16, C::SBO, C::SW);      // K-major B
            const uint64_t dV = smem_desc(smem_u32(tv), 16384, 1024, kSw128);    // MN-major B
            auto qk = [&](int j) {   // S = Q K_j^T
                const int ks0 = j % C::KST;
                const uint64_t b0 = desc_add(dK, ks0 * C::QK_TILE);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_ss(tS, desc_add(dQ, ks * 32), desc_add(b0, ks * 32), kIdQK, ks > 0);
                mma_commit(&s_full);
                mma_commit(&k_empty[ks0]);
            };
            bool ok = sy.wait(&q_full, 0) && sy.wait(&k_full[0], 0);
            if (ok) {
                tc_fence_after();
                qk(0);
            }
            for (int j = 0; j < nj && ok; ++j) {
                // S_{j+1} once the P warps have read S_j (they may still be writing P_j)
                if (j + 1 < nj) {
                    ok = sy.wait(&k_full[(j + 1) % C::KST], (j + 1) / C::KST) && sy.wait(&s_free, j);
                    if (!ok) break;
                    tc_fence_after();
                    qk(j + 1);
                }
                // O += P_j V_j
                const int vs = j % C::VST;
                ok = sy.wait(&v_full[vs], j / C::VST) && sy.wait(&p_full, j);
                if (!ok) break;
                tc_fence_after();
                const uint64_t b0 = desc_add(dV, vs * C::V_TILE);
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ts(tO, tP + ks * 8, desc_add(b0, ks * 2048), kIdPV, (j > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&p_free);
                mma_commit(&v_empty[vs]);
            }
            mma_commit(&o_done);
            mma_commit(&fin_bar);
            sy.wait(&fin_bar, 0);
        }
    } else {
        // ================= P warps: query row r = 32 * (warp % 4) + lane, keys
        // 64 h .. 64 h + 63 of each tile
        const int quarter = warp & 3, h = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lsel = (uint32_t)(quarter * 32) << 16;
        float dsum = 0.f;
        float rt = 1.f, M = 1.f;   // gated: r_t and the running M_ij
        if constexpr (kGated) {
            const int t0 = qi * kTile;
            for (int u = (int)threadIdx.x - 64; u < kTile; u += kPWarps * 32)
                lamd[u] = t0 + u < T ? ga.lam2[(size_t)bh * T + t0 + u] : 0.f;
            asm volatile("bar.sync 2, %0;" ::"r"(kPWarps * 32) : "memory");
            rt = exp2f(lamd[r]);
        }
        bool ok = true;
        // iteration j walks key tile qi - j (j = 0: the diagonal tile)
        for (int j = 0; j < nj && ok; ++j) {
            float gj = 1.f;   // gated: the product of the gates of this key tile
            if (kGated && j > 0) gj = ga.gtile[(size_t)bh * NT + qi - j];
            ok = __all_sync(0xffffffffu, sy.wait(&s_full, j));
            if (!ok) break;
            tc_fence_after();
            const bool diag = j == 0;   // keys past the query are masked on the diagonal tile
            uint32_t v[64], pw[32];
            tmem_ld64(tS + lsel + 64 * h, v);
            // S_j is in registers (the load has completed): the next S MMA may
            // overwrite it while P_j is formed
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&s_free);
            if (kGated && !diag) {
                // w = S'^2 r_t M_ij: packed square, packed scale, packed sum, convert
                const float f = rt * M;
                const uint64_t ff = f2_make(__float_as_uint(f), __float_as_uint(f));
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const uint64_t w = f2_mul(f2_sq(f2_make(v[2 * e], v[2 * e + 1])), ff);
                    acc[e & 3] = f2_add(acc[e & 3], w);
                    float w0, w1;
                    f2_split(w, w0, w1);
                    pw[e] = pack_bf16(w0, w1);
                }
                float a0, a1;
                f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                dsum += a0 + a1;
                M *= gj;
            } else if (kGated) {
                // diagonal tile: a_ts = 2^(l_t - l_s) for s <= t
                const float lr = lamd[r];
                float ds[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = 64 * h + 2 * e;
                    const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                    const float w0 = c <= r ? x0 * x0 * exp2f(lr - lamd[c]) : 0.f;
                    const float w1 = c + 1 <= r ? x1 * x1 * exp2f(lr - lamd[c + 1]) : 0.f;
                    ds[e & 3] += w0 + w1;
                    pw[e] = pack_bf16(w0, w1);
                }
                dsum += (ds[0] + ds[1]) + (ds[2] + ds[3]);
            } else if (!diag) {
                // packed pairs: one multiply, one add and one convert per two keys;
                // four accumulator chains so the adds overlap
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const uint64_t w = f2_sq(f2_make(v[2 * e], v[2 * e + 1]));
                    acc[e & 3] = f2_add(acc[e & 3], w);
                    float w0, w1;
                    f2_split(w, w0, w1);
                    pw[e] = pack_bf16(w0, w1);
                }
                float a0, a1;
                f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                dsum += a0 + a1;
            } else {
                float ds[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = 64 * h + 2 * e;
                    const float x0 = __uint_as_float(v[2 * e]), x1 = __uint_as_float(v[2 * e + 1]);
                    const float w0 = c <= r ? x0 * x0 : 0.f;
                    const float w1 = c + 1 <= r ? x1 * x1 : 0.f;
                    ds[e & 3] += w0 + w1;
                    pw[e] = pack_bf16(w0, w1);
                }
                dsum += (ds[0] + ds[1]) + (ds[2] + ds[3]);
            }
            // the P V MMA of the previous tile has read P
            ok = __all_sync(0xffffffffu, j == 0 || sy.wait(&p_free, j - 1));
            if (!ok) break;
            tc_fence_after();
            tmem_st32(tP + lsel + 32 * h, pw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (elect_lane0()) mbar_arrive(&p_full);
        }
        // epilogue: O = N / D (a zero denominator gives a zero row), staged
        // 128B-swizzled in V slot 0 (every P V MMA is done by then) and written by
        // one TMA store, which also clips the rows past T; every P warp reaches the
        // named barriers, also after a failed wait
        dpart[h][r] = dsum;
        asm volatile("bar.sync 1, %0;" ::"r"(kPWarps * 32) : "memory");
        if (ok && __all_sync(0xffffffffu, sy.wait(&o_done, 0))) {
            tc_fence_after();
            const float den = dpart[0][r] + dpart[1][r];
            const float inv = (kGated && !ga.normalize) ? 1.f : den > 0.f ? 1.f / den : 0.f;
            uint32_t v[32];
            tmem_ld32(tO + lsel + 32 * h, v);
            const uint32_t row = smem_u32(tv) + (uint32_t)r * 128u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t chunk = (uint32_t)(4 * h + c) ^ (uint32_t)(r & 7);
                st_shared_v4(row + (chunk << 4),
                             pack_bf16(__uint_as_float(v[8 * c + 0]) * inv, __uint_as_float(v[8 * c + 1]) * inv),
                             pack_bf16(__uint_as_float(v[8 * c + 2]) * inv, __uint_as_float(v[8 * c + 3]) * inv),
                             pack_bf16(__uint_as_float(v[8 * c + 4]) * inv, __uint_as_float(v[8 * c + 5]) * inv),
                             pack_bf16(__uint_as_float(v[8 * c + 6]) * inv, __uint_as_float(v[8 * c + 7]) * inv));
            }
            fence_proxy_async_smem();
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kPWarps * 32) : "memory");
        if (warp == 2 && lane == 0 && !abort_flag) {
            tma_store_3d(&tm_o, 0, qi * kTile, bh, tv);
            bulk_commit();
            bulk_wait_read_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag) atomicOr(&g_quad_error, 1);
    if (warp == 1) tmem_dealloc(tmem_base, 256);
}

template <int D>
cudaError_t quad_launch(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                        cudaStream_t stream, const float *gamma, int normalize, void *ws) {
    using C = QuadCfg<D>;
    CUtensorMap mq, mk, mv, mkp, mo;
    if (!make_map(mq, q, s.d, s.T, s.BH()) || !make_map(mk, k, s.d, s.T, s.BH()) ||
        !make_map(mv, v, s.dv, s.T, s.BH()) || !make_map(mo, out, s.dv, s.T, s.BH()))
        return cudaErrorInvalidValue;
    const int NT = (s.T + kTile - 1) / kTile;
    if (!gamma) {
        cudaFuncSetAttribute(quad_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
        TraceScope tr("tc_quadratic", stream);
        quad_kernel<D, false><<<dim3(s.BH(), NT), 320, C::SMEM, stream>>>(
            mq, mk, mv, mk, mo, s.T, NT, GateArgs{nullptr, nullptr, 1});
        return cudaGetLastError();
    }
    // workspace: K' [BH][T][d] bf16 | lam2 [BH][T] fp32 | tile gate products [BH][NT] fp32
    const size_t nk = (size_t)s.BH() * s.T * s.d;
    bf16 *kp = static_cast<bf16 *>(ws);
    float *lam2 = reinterpret_cast<float *>(kp + nk);
    float *gtile = lam2 + (size_t)s.BH() * s.T;
    if (!make_map(mkp, kp, s.d, s.T, s.BH())) return cudaErrorInvalidValue;
    {
        TraceScope tr("tc_gate_prep", stream);
        gate_prep_kernel<D><<<dim3(NT, s.BH()), kTile, 0, stream>>>(
            (const bf16 *)k, gamma, kp, lam2, gtile, s.T, NT);
    }
    cudaFuncSetAttribute(quad_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         C::SMEM);
    TraceScope tr("tc_quadratic_gated", stream);
    quad_kernel<D, true><<<dim3(s.BH(), NT), 320, C::SMEM, stream>>>(
        mq, mk, mv, mkp, mo, s.T, NT, GateArgs{lam2, gtile, normalize});
    return cudaGetLastError();
}

}  // namespace

cudaError_t gate_prep_launch(const void *k, const float *gamma, void *kp, float *lam2, float *gtile,
                             int BH, int T, int d, cudaStream_t stream) {
    if (d != 32 && d != 64) return cudaErrorInvalidValue;
    const int NT = (T + kTile - 1) / kTile;
    TraceScope tr("tc_gate_prep", stream);
    if (d == 32)
        gate_prep_kernel<32><<<dim3(NT, BH), kTile, 0, stream>>>((const bf16 *)k, gamma, (bf16 *)kp,
                                                                  lam2, gtile, T, NT);
    else
        gate_prep_kernel<64><<<dim3(NT, BH), kTile, 0, stream>>>((const bf16 *)k, gamma, (bf16 *)kp,
                                                                  lam2, gtile, T, NT);
    return cudaGetLastError();
}

bool quad_supported(const FwdShape &s, int cc_major, int cc_minor) {
    return s.dtype == 1 && cc_major == 10 && cc_minor == 3 && (s.d == 32 || s.d == 64) &&
           s.dv == 64 && (s.T + kTile - 1) / kTile <= 65535 && encoder() != nullptr;
}

cudaError_t quad_forward(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                         cudaStream_t stream, const float *gamma, int normalize, void *ws) {
    if ((size_t)s.BH() * s.T == 0) return cudaSuccess;
    return s.d == 64 ? quad_launch<64>(s, q, k, v, out, stream, gamma, normalize, ws)
                     : quad_launch<32>(s, q, k, v, out, stream, gamma, normalize, ws);
}

size_t quad_gated_workspace_bytes(const FwdShape &s) {
    const size_t NT = (s.T + kTile - 1) / kTile;
    return (size_t)s.BH() * ((size_t)s.T * s.d * 2 + (size_t)s.T * 4 + NT * 4);
}

int quad_take_error() {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_quad_error, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (h) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_quad_error, &zero, sizeof(int));
    }
    return h;
}

}  // namespace kata
