// The explicit-feature tensor-core path (kata_feat.cu): the chunked forward of a
// lift map whose packed features are few enough to be written out, on tcgen05.
#pragma once
#include "kata_internal.cuh"

namespace kata {

// Most packed features the path takes (three 64-feature boxes, two 128-feature
// state blocks; the output kernel holds four feature tiles): KATA-Sigma_4 at
// d = 64 (136), Sigma_2 / Sigma_4 / M_4 at d = 32, every map at d = 16, the
// orthant map.
constexpr int kFeatMax = 192;

// bf16, dv = 64, map.n(d) <= kFeatMax, sm_103a.
bool feat_supported(const FwdShape &s, const MapSpec &map, int cc_major, int cc_minor);
size_t feat_workspace_bytes(const FwdShape &s, const MapSpec &map);
// so: the state after the last token (row-major packed features of the map).
cudaError_t feat_forward(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                         void *workspace, cudaStream_t stream, const MapSpec &map,
                         const StateOut &so = StateOut{});
// Reads and clears the sticky error word of the path's kernels (nonzero: a
// bounded wait expired); -1 if it could not be read.
int feat_take_error();

}  // namespace kata
