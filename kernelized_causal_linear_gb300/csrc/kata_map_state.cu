// The state of a reduced PSD map after the last token, composed from the
// full-map states its tensor route leaves (KATA paper, Sec. 4.1 "two reduced
// PSD families"; the state S = sum_t psi(k_t) v_t^T and z = sum_t psi(k_t) of
// Sec. 3 with the map's psi).
//
// Every feature sits in the packed order of the map's lift: each matrix
// row-major over its upper triangle, sqrt(2) on the off-diagonal entries, M_g's
// matrices block by block.  A full-map state of dimension dsrc in the same order
// holds, for the coordinate pair (i, j), sum_t c_ij k_ti k_tj v_t (c_ij = 1 on
// the diagonal, sqrt(2) off it).
//
//   KATA-M_g, psi(u) = (u_a u_a^T)_a: block a's features are those of the full
//   map of u_a.  The route runs block a as a sub-head whose first m = d / g
//   coordinates are u_a (the rest zero padding), so the block's feature (i, j)
//   is the sub-head's feature (i, j), i <= j < m.
//   KATA-Sigma_g, psi(u) = eps I + s sum_a u_a u_a^T: feature (i, j) is
//   eps [i = j] + s sum_a c_ij u_ai u_aj, so the map's state is
//   s sum_a S_a + eps [i = j] sum_t v_t, and z = s sum_a z_a + eps [i = j] T,
//   with S_a the full-map state of key block a.
#include "kata_internal.cuh"

namespace kata {
namespace {

constexpr int kDv = 64;   // the tensor routes' value width

// Row i of a packed upper triangle of dimension m: features (i, i..m-1), from
// i*m - i*(i-1)/2 on, contiguous, the first one diagonal.
__host__ __device__ __forceinline__ int row_start(int i, int m) { return i * m - i * (i - 1) / 2; }

// Grid (m, g or 1, BH): one CTA per map row (i), block (a, M_g only) and head;
// the row's m - i features x 64 columns are one contiguous run in the source
// and in the map's state, moved as float4.
__global__ void __launch_bounds__(256)
map_state_compose_kernel(const float *__restrict__ src, const float *__restrict__ src_z, int nsrc,
                         int dsrc, int kind, int m, float eps, float scale,
                         const float *__restrict__ eps_totals, float count,
                         float *__restrict__ state, float *__restrict__ z, int n) {
    const int i = blockIdx.x, a = blockIdx.y, bh = blockIdx.z;
    const int nm = m * (m + 1) / 2, ns = dsrc * (dsrc + 1) / 2, len = m - i;
    const int fd = (kind == 1 ? a * nm : 0) + row_start(i, m);   // the row in the map
    const int fs = row_start(i, dsrc);                             // the row in a source
    float4 *dst = reinterpret_cast<float4 *>(state + ((size_t)bh * n + fd) * kDv);
    const int n4 = len * (kDv / 4);
    if (kind == 1) {   // M_g: block a is source a's first m coordinates
        const size_t r = ((size_t)bh * nsrc + a) * ns + fs;
        const float4 *sp = reinterpret_cast<const float4 *>(src + r * kDv);
        for (int e = threadIdx.x; e < n4; e += blockDim.x) dst[e] = sp[e];
        for (int e = threadIdx.x; e < len; e += blockDim.x) z[(size_t)bh * n + fd + e] = src_z[r + e];
        return;
    }
    // Sigma_g: s times the key blocks' states summed in order, eps sum_t v_t on
    // the row's first (diagonal) feature
    const float4 *tv = reinterpret_cast<const float4 *>(eps_totals + (size_t)bh * kSigmaRec);
    for (int e = threadIdx.x; e < n4; e += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b = 0; b < nsrc; ++b) {
            const size_t r = ((size_t)bh * nsrc + b) * ns + fs;
            const float4 x = reinterpret_cast<const float4 *>(src + r * kDv)[e];
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
        float4 o = make_float4(scale * acc.x, scale * acc.y, scale * acc.z, scale * acc.w);
        if (e < kDv / 4) {
            const float4 t = tv[e];
            o = make_float4(o.x + eps * t.x, o.y + eps * t.y, o.z + eps * t.z, o.w + eps * t.w);
        }
        dst[e] = o;
    }
    for (int e = threadIdx.x; e < len; e += blockDim.x) {
        float acc = 0.f;
        for (int b = 0; b < nsrc; ++b) acc += src_z[((size_t)bh * nsrc + b) * ns + fs + e];
        z[(size_t)bh * n + fd + e] = scale * acc + (e == 0 ? eps * count : 0.f);
    }
}

}  // namespace

cudaError_t map_state_compose(const float *src_state, const float *src_z, int nsrc, int dsrc,
                              const MapSpec &map, int d, const float *eps_totals, int T,
                              float *state, float *z, int BH, cudaStream_t stream) {
    const int m = map.m(d), n = map.n(d);
    if ((map.kind != 1 && map.kind != 2) || nsrc != map.g || m > dsrc || BH < 1 || BH > 65535)
        return cudaErrorInvalidValue;
    if (map.kind == 2 && (m != dsrc || eps_totals == nullptr)) return cudaErrorInvalidValue;
    TraceScope tr("tc_map_state", stream);
    map_state_compose_kernel<<<dim3(m, map.kind == 1 ? map.g : 1, BH), 256, 0, stream>>>(
        src_state, src_z, nsrc, dsrc, map.kind, m, map.eps, map.scale, eps_totals, (float)T,
        state, z, n);
    return cudaGetLastError();
}

}  // namespace kata
