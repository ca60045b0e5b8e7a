// Shared pieces of the CUDA-core (fp32 FFMA) chunked kernels: the plain and
// reduced-map path (kata_simt.cu) and GatedKATA (kata_gated.cu).  Both tile a
// chunk's state record [n][dv + 1] in 128-feature rows x 32-column groups (the
// 33rd column is the normaliser) and stage state rows through shared memory.
#pragma once
#include "kata_internal.cuh"

namespace kata {
namespace simt {

constexpr int kColGroup = 32;     // value columns per block (plus the ones column)
constexpr int kStride = kColGroup + 1;
constexpr int kRow = 36;          // staged state rows: 33 values, 16-byte aligned
constexpr int kFeatTile = 128;    // features per chunk-state block
constexpr int kStageRows = 64;    // prefix rows staged per step in the output kernels

// acc[0..31] += a * row[0..31] for a 16-byte aligned shared-memory row: eight
// 16-byte loads per 32 FMAs (the rows are read by every thread at once).
__device__ __forceinline__ void fma_row32(float a, const float *row, float (&acc)[kStride]) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
#pragma unroll
    for (int u = 0; u < kColGroup / 4; ++u) {
        const float4 x = r4[u];
        acc[4 * u + 0] = fmaf(a, x.x, acc[4 * u + 0]);
        acc[4 * u + 1] = fmaf(a, x.y, acc[4 * u + 1]);
        acc[4 * u + 2] = fmaf(a, x.z, acc[4 * u + 2]);
        acc[4 * u + 3] = fmaf(a, x.w, acc[4 * u + 3]);
    }
}

// A state-kernel block's results (thread = feature ft * kFeatTile + threadIdx.x,
// acc = its 32 columns of group cg and its normaliser) into the record rows at
// `base` [n][W], through shared memory `os` [kFeatTile][kStride] so that each
// warp writes contiguous row segments.  Every thread of the block calls it.
__device__ __forceinline__ void store_state_rows(const float (&acc)[kStride], float *os,
                                                 float *base, int ft, int cg, int cols, int n,
                                                 int dv) {
    const int W = dv + 1;
    __syncthreads();
#pragma unroll
    for (int jj = 0; jj < kStride; ++jj) os[threadIdx.x * kStride + jj] = acc[jj];
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int r = warp; r < kFeatTile; r += blockDim.x / 32) {
        const int ff = ft * kFeatTile + r;
        if (ff >= n) break;
        float *row = base + (size_t)ff * W;
        if (lane < cols) row[cg * kColGroup + lane] = os[r * kStride + lane];
        if (cg == 0 && lane == 0) row[dv] = os[r * kStride + kColGroup];
    }
}

// Rows f0 .. f0 + nf - 1 of a state record sp [n][W] into `stg` [kStageRows][kRow]:
// the 32 columns of group cg (zero past `cols`) and the normaliser.  Block-wide.
__device__ __forceinline__ void stage_state_rows(const float *sp, float *stg, int f0, int nf,
                                                 int cg, int cols, int dv) {
    const int W = dv + 1;
    for (int e = threadIdx.x; e < nf * kStride; e += blockDim.x) {
        const int fr = e / kStride, jj = e % kStride;
        const float *row = sp + (size_t)(f0 + fr) * W;
        float val = 0.f;
        if (jj < cols) val = row[cg * kColGroup + jj];
        else if (jj == kColGroup) val = row[dv];
        stg[fr * kRow + jj] = val;
    }
}

}  // namespace simt
}  // namespace kata
