// C ABI of libkata (declared and documented in include/kata.h): argument
// validation, path selection, workspace management and launches.
#include <cmath>
#include <mutex>

#include "../../include/kata.h"
#include "kata_feat.cuh"
#include "kata_dispatch.cuh"

using kata::FwdShape;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_d(int d) { return d == 16 || d == 32 || d == 64; }
bool valid_dv(int dv) { return dv == 16 || dv == 32 || dv == 64 || dv == 128; }
bool valid_C(int C) { return C == 32 || C == 64 || C == 128; }
bool valid_dtype(int t) { return t == KATA_F32 || t == KATA_BF16; }
size_t elem_size(int t) { return t == KATA_F32 ? 4 : 2; }

// A map the reduced-PSD entry points accept (see kata_fwd_chunked_map).
bool valid_map(int map, int d, int g, float eps, float scale) {
    if (map == KATA_MAP_ORTHANT)   // one feature per coordinate: g = 1, scale 1, eps >= 0
        return g == 1 && std::isfinite(eps) && eps >= 0.f && scale == 1.f;
    if (map < KATA_MAP_FULL || map > KATA_MAP_SUM) return false;
    if (!(g == 1 || g == 2 || g == 4) || d < g || d % g != 0) return false;
    if (!std::isfinite(eps) || !std::isfinite(scale) || eps < 0.f || scale <= 0.f) return false;
    if (map == KATA_MAP_FULL && g != 1) return false;
    if (map != KATA_MAP_SUM && (eps != 0.f || scale != 1.f)) return false;
    return true;
}

// The map descriptor of a validated (map, g, eps, scale).  KATA-M_1 is the full
// rank-one map (one block of width d), so it takes the full map's paths, whose
// intra-chunk weights are (q.k)^2 formed from q and k.
kata::MapSpec map_spec(int map, int g, float eps, float scale) {
    kata::MapSpec ms;
    ms.kind = (map == KATA_MAP_BLOCK && g == 1) ? KATA_MAP_FULL : map;
    ms.g = g;
    ms.eps = eps;
    ms.scale = scale;
    return ms;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_fwd_shape(int B, int H, int T, int d, int dv, int C, int dtype) {
    if (B < 1 || H < 1 || T < 1) return KATA_ERR_ARG;
    if (!valid_dtype(dtype)) return KATA_ERR_ARG;
    if ((int64_t)B * H > 65535) return KATA_ERR_UNSUPPORTED;   // grid.y limit
    if (!valid_d(d) || !valid_dv(dv) || !valid_C(C)) return KATA_ERR_UNSUPPORTED;
    return KATA_OK;
}

// Device properties cached per device (queried once).
struct DevInfo {
    int major = 0, minor = 0, sms = 0;
    bool ok = false;
};

int device_info(DevInfo &out) {
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    DevInfo &di = cache[dev];
    if (!di.ok) {
        if (cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return KATA_ERR_CUDA;
        }
        // Keep freed workspace in the stream-ordered pool between calls.
        cudaMemPool_t pool;
        if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
            uint64_t thr = UINT64_MAX;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
        }
        cudaGetLastError();
        di.ok = true;
    }
    out = di;
    return KATA_OK;
}

// Kernel families behind the public paths: KATA_PATH_TC covers both tensor-core
// variants (d = 32 with segments, d = 64 with the state split over four CTAs);
// kTc32Sub is KATA-M_2 at d = 64 as two d = 32 sub-heads, kTc32Sigma is
// KATA-Sigma_2 at d = 64 as four crosswise d = 32 sub-heads plus its eps terms,
// kTc32M4 is KATA-M_4 at d = 64 as four zero-padded d = 32 sub-heads;
// kTc32Adapt / kTc64Adapt run the other bf16 shapes (d = 16, dv != 64) on the
// two tensor-core paths through padded copies and 64-column parts of v.
// kFeat: a reduced map with at most kFeatMax packed features on the explicit-
// feature tensor path (kata_feat.cu).
// kTc32SubPad: KATA-M_2 at d = 32 as M_2 at d = 64 on the rows [u_1 0 | u_2 0].
// kTc32Sigma1 / kTc64Sigma1: KATA-Sigma_1 (eps I + s u u^T) at d = 32 / 64 as the
// full map on the d = 32 / d = 64 tensor path plus its eps terms.
enum Kernels { kSimt, kTc32, kTc64, kTc32Sub, kTc32Sigma, kTc32M4, kTc32Adapt, kTc64Adapt, kFeat,
               kTc32SubPad, kTc32Sigma1, kTc64Sigma1 };

Kernels from_fwd(kata::FwdKernels k) {
    switch (k) {
        case kata::FwdKernels::Tc32: return kTc32;
        case kata::FwdKernels::Tc64: return kTc64;
        case kata::FwdKernels::Tc32Adapt: return kTc32Adapt;
        case kata::FwdKernels::Tc64Adapt: return kTc64Adapt;
        default: return kSimt;
    }
}

Kernels select_kernels(const FwdShape &s, const DevInfo &di) {
    return from_fwd(kata::select_fwd_kernels(s, di.major, di.minor, di.sms));
}

// Kernels for a reduced map: KATA-M_2, KATA-Sigma_2 and KATA-M_4 at d = 64 are
// d = 32 sub-heads on the d = 32 tensor path (bf16, dv = 64); KATA-Sigma_1 is
// the full map plus its eps terms; the other maps with at most kFeatMax packed
// features (KATA-Sigma_4 at d = 64; Sigma_2, Sigma_4 and M_4 at d = 32; every
// map at d = 16; the orthant map) take the explicit-feature tensor path (bf16,
// dv = 64); the rest runs on CUDA cores.
// Every route exports the map's state.  The sub-head routes launch nsub
// sub-heads per head along grid.y, so they need B H nsub <= 65535.
Kernels select_map_kernels(const FwdShape &s, const DevInfo &di, const kata::MapSpec &map) {
    if (map.kind == KATA_MAP_FULL) return select_kernels(s, di);
    const int64_t bh = s.BH();
    if (s.d == 64 && map.kind == KATA_MAP_SUM && map.g == 1 &&
        kata::tc64_supported(s, di.major, di.minor, di.sms))
        return kTc64Sigma1;   // 2080 features
    if (s.d == 64) {
        FwdShape half = s;
        half.d = 32;
        if (kata::tc_supported(half, di.major, di.minor)) {
            if (map.kind == KATA_MAP_BLOCK && map.g == 2 && bh * 2 <= 65535) return kTc32Sub;
            if (map.kind == KATA_MAP_SUM && map.g == 2 && bh * 4 <= 65535) return kTc32Sigma;
            if (map.kind == KATA_MAP_BLOCK && map.g == 4 && bh * 4 <= 65535) return kTc32M4;
        }
    }
    if (kata::feat_supported(s, map, di.major, di.minor)) return kFeat;
    if (s.d == 32 && map.kind == KATA_MAP_BLOCK && map.g == 2 && bh * 2 <= 65535 &&
        kata::tc_supported(s, di.major, di.minor))
        return kTc32SubPad;   // 272 features: above the explicit-feature path's limit
    if (s.d == 32 && map.kind == KATA_MAP_SUM && map.g == 1 &&
        kata::tc_supported(s, di.major, di.minor))
        return kTc32Sigma1;   // 528 features
    return kSimt;
}

int select_path(const FwdShape &s, const DevInfo &di) {
    return select_kernels(s, di) == kSimt ? KATA_PATH_SIMT : KATA_PATH_TC;
}

kata::FwdKernels to_fwd(Kernels kn) {
    switch (kn) {
        case kTc32: return kata::FwdKernels::Tc32;
        case kTc64: return kata::FwdKernels::Tc64;
        case kTc32Adapt: return kata::FwdKernels::Tc32Adapt;
        case kTc64Adapt: return kata::FwdKernels::Tc64Adapt;
        default: return kata::FwdKernels::Simt;
    }
}

size_t workspace_for(const FwdShape &s, Kernels kn, const DevInfo &di, bool with_state = false) {
    return kata::fwd_workspace_bytes(s, to_fwd(kn), di.sms, with_state);
}

}  // namespace

namespace kata {

FwdKernels select_fwd_kernels(const FwdShape &s, int cc_major, int cc_minor, int num_sms) {
    if (s.dtype == KATA_F32) return FwdKernels::Simt;
    if (tc_supported(s, cc_major, cc_minor)) return FwdKernels::Tc32;
    if (tc64_supported(s, cc_major, cc_minor, num_sms)) return FwdKernels::Tc64;
    return adapt_kernels(s, cc_major, cc_minor, num_sms);
}

size_t fwd_workspace_bytes(const FwdShape &s, FwdKernels kn, int num_sms, bool with_state) {
    switch (kn) {
        case FwdKernels::Tc32: return tc_workspace_bytes(s, num_sms, with_state);
        case FwdKernels::Tc64: return tc64_workspace_bytes(s, with_state);
        case FwdKernels::Tc32Adapt:
        case FwdKernels::Tc64Adapt: return adapt_workspace_bytes(s, kn, num_sms, with_state);
        default: return simt_workspace_bytes(s);
    }
}

cudaError_t fwd_launch(const FwdShape &s, FwdKernels kn, const void *q, const void *k,
                       const void *v, void *out, void *workspace, int num_sms,
                       cudaStream_t stream, const StateOut &so) {
    switch (kn) {
        case FwdKernels::Tc32: return tc_forward(s, q, k, v, out, workspace, num_sms, stream, so);
        case FwdKernels::Tc64: return tc64_forward(s, q, k, v, out, workspace, stream, so);
        case FwdKernels::Tc32Adapt:
        case FwdKernels::Tc64Adapt:
            return adapt_forward(s, kn, q, k, v, out, workspace, num_sms, stream, so);
        default: return simt_forward(s, q, k, v, out, workspace, stream, so);
    }
}

}  // namespace kata

extern "C" {

int kata_feature_dim(int d) { return d < 1 ? -1 : d * (d + 1) / 2; }

const char *kata_status_str(int status) {
    switch (status) {
        case KATA_OK: return "ok";
        case KATA_ERR_ARG: return "invalid argument";
        case KATA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case KATA_ERR_CUDA: return "CUDA runtime error";
        case KATA_ERR_ALLOC: return "device workspace allocation failed";
        case KATA_ERR_TIMEOUT: return "bounded device-side wait expired";
        case KATA_ERR_SCRATCH_LIMIT:
            return "shape needs more scratch than the fixed no-allocation buffer holds";
        default: return "unknown status";
    }
}

int kata_fwd_workspace_size(int B, int H, int T, int d, int dv, int C, int dtype,
                            size_t *bytes) {
    if (!bytes) return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    const FwdShape s{B, H, T, d, dv, C, dtype};
    *bytes = workspace_for(s, select_kernels(s, di), di);
    return KATA_OK;
}

int kata_fwd_segments(int B, int H, int T, int d, int dv, int C, int dtype, int *seg_tokens) {
    int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    const FwdShape s{B, H, T, d, dv, C, dtype};
    const Kernels kn = select_kernels(s, di);
    if (kn == kTc32 || kn == kTc32Adapt) return kata::tc_segments(s, di.sms, seg_tokens);
    if (seg_tokens) *seg_tokens = T;
    return 1;
}

int kata_fwd_path(int B, int H, int T, int d, int dv, int C, int dtype) {
    if (check_fwd_shape(B, H, T, d, dv, C, dtype)) return KATA_PATH_NONE;
    DevInfo di;
    if (device_info(di)) return KATA_PATH_NONE;
    return select_path(FwdShape{B, H, T, d, dv, C, dtype}, di);
}

}  // extern "C"

namespace {
size_t round_up256(size_t b) { return (b + 255) & ~(size_t)255; }

// KATA-M_2 at d = 32 through the d = 64 sub-head route: q and k rows copied to
// [u_1 0 | u_2 0] (64 columns); the zero coordinates add nothing to either
// block's (q_a . k_a)^2.  Workspace: the padded q and k, then the route's.
FwdShape padded64(const FwdShape &s) {
    FwdShape c = s;
    c.d = 64;
    return c;
}

cudaError_t pad_run(const FwdShape &s, const void *q, const void *k, const void *v, void *out,
                    void *ws, const DevInfo &di, cudaStream_t st, const kata::StateOut &so) {
    const int64_t rows = (int64_t)s.BH() * s.T;
    const size_t np = round_up256((size_t)rows * 64 * 2);
    uint8_t *b = static_cast<uint8_t *>(ws);
    void *qp = b, *kp = b + np;
    cudaError_t e = cudaSuccess;
    for (int side = 0; side < 2; ++side) {   // [u_1 0 | u_2 0]
        const void *src = side ? k : q;
        void *dst = side ? kp : qp;
        if ((e = kata::part_copy_cols(src, 32, 0, 16, dst, 64, 0, rows, true, st)) != cudaSuccess ||
            (e = kata::part_copy_cols(src, 32, 16, 16, dst, 64, 32, rows, false, st)) != cudaSuccess)
            return e;
    }
    return kata::tc_forward(padded64(s), qp, kp, v, out, b + 2 * np, di.sms, st, so, 2);
}

// The routes whose map state is composed from full-map states (kata_map_state.cu):
// nsrc of dimension dsrc per head.  M_2 at d = 64 needs no composition: its two
// sub-heads' states are its two blocks, in its own order.
bool composed_state(Kernels kn, int &nsrc, int &dsrc) {
    switch (kn) {
        case kTc32SubPad: nsrc = 2; dsrc = 32; return true;    // M_2 at d = 32, blocks [u_a 0]
        case kTc32M4: nsrc = 4; dsrc = 32; return true;        // M_4 at d = 64, blocks [u_a 0]
        case kTc32Sigma: nsrc = 2; dsrc = 32; return true;     // Sigma_2 at d = 64: the key halves
        case kTc32Sigma1: nsrc = 1; dsrc = 32; return true;
        case kTc64Sigma1: nsrc = 1; dsrc = 64; return true;
        default: return false;
    }
}

// Scratch of a composed state, ahead of the route's: the sources' states and z,
// then the eps totals.
struct ComposeWs {
    size_t state, z, tot;
    size_t total() const { return state + z + tot; }
};
ComposeWs compose_ws(const FwdShape &s, int nsrc, int dsrc) {
    const size_t heads = (size_t)s.BH() * nsrc, ns = (size_t)dsrc * (dsrc + 1) / 2;
    return ComposeWs{round_up256(heads * ns * 64 * 4), round_up256(heads * ns * 4),
                     round_up256((size_t)s.BH() * kata::kSigmaRec * 4)};
}

// Workspace and launch of one kernel family for a (map, shape).
size_t route_ws(const FwdShape &s, Kernels kn, const DevInfo &di, const kata::MapSpec &map,
                bool with_state) {
    int nsrc = 0, dsrc = 0;
    const size_t pre = with_state && composed_state(kn, nsrc, dsrc) ? compose_ws(s, nsrc, dsrc).total() : 0;
    if (kn == kTc32SubPad)
        return pre + 2 * round_up256((size_t)s.BH() * s.T * 64 * 2) +
               kata::tc_workspace_bytes(padded64(s), di.sms, with_state, 2);
    return pre + (kn == kTc32Sub      ? kata::tc_workspace_bytes(s, di.sms, with_state, 2)
                  : kn == kTc32Sigma  ? kata::tc_workspace_bytes(s, di.sms, with_state, 4, &map)
                  : kn == kTc32Sigma1 ? kata::tc_workspace_bytes(s, di.sms, with_state, 1, &map)
                  : kn == kTc64Sigma1 ? kata::tc64_workspace_bytes(s, with_state, &map)
                  : kn == kTc32M4     ? kata::tc_m4_workspace_bytes(s, di.sms, with_state)
                  : kn == kFeat       ? kata::feat_workspace_bytes(s, map)
                  : map.kind == 0     ? workspace_for(s, kn, di, with_state)
                                      : kata::simt_workspace_bytes(s, map));
}

cudaError_t route_launch(const FwdShape &s, Kernels kn, const void *q, const void *k, const void *v,
                         void *out, void *ws, const DevInfo &di, cudaStream_t st,
                         const kata::StateOut &so, const kata::MapSpec &map) {
    if (kn == kTc32SubPad) return pad_run(s, q, k, v, out, ws, di, st, so);
    return kn == kTc32Sub      ? kata::tc_forward(s, q, k, v, out, ws, di.sms, st, so, 2)
           : kn == kTc32Sigma  ? kata::tc_forward(s, q, k, v, out, ws, di.sms, st, so, 4, &map)
           : kn == kTc32Sigma1 ? kata::tc_forward(s, q, k, v, out, ws, di.sms, st, so, 1, &map)
           : kn == kTc64Sigma1 ? kata::tc64_forward(s, q, k, v, out, ws, st, so, &map)
           : kn == kTc32M4    ? kata::tc_forward_m4(s, q, k, v, out, ws, di.sms, st, so)
           : kn == kFeat      ? kata::feat_forward(s, q, k, v, out, ws, st, map, so)
           : map.kind == 0    ? kata::fwd_launch(s, to_fwd(kn), q, k, v, out, ws, di.sms, st, so)
                              : kata::simt_forward(s, q, k, v, out, ws, st, so, map);
}

// The route, and with a state asked for on a composed route, its sources'
// states into scratch followed by the map's state from them.
cudaError_t route_run(const FwdShape &s, Kernels kn, const void *q, const void *k, const void *v,
                      void *out, void *ws, const DevInfo &di, cudaStream_t st,
                      const kata::StateOut &so, const kata::MapSpec &map) {
    int nsrc = 0, dsrc = 0;
    if (so.state == nullptr || !composed_state(kn, nsrc, dsrc))
        return route_launch(s, kn, q, k, v, out, ws, di, st, so, map);
    const ComposeWs c = compose_ws(s, nsrc, dsrc);
    uint8_t *b = static_cast<uint8_t *>(ws);
    kata::StateOut src;
    src.state = reinterpret_cast<float *>(b);
    src.z = reinterpret_cast<float *>(b + c.state);
    if (map.kind == KATA_MAP_SUM) src.eps_totals = reinterpret_cast<float *>(b + c.state + c.z);
    cudaError_t e = route_launch(s, kn, q, k, v, out, b + c.total(), di, st, src, map);
    if (e != cudaSuccess) return e;
    return kata::map_state_compose(src.state, src.z, nsrc, dsrc, map, s.d, src.eps_totals, s.T,
                                   so.state, so.z, s.BH(), st);
}

// A reduced map with bf16 inputs and dv in {16, 32, 128} whose route at dv = 64
// is a tensor path runs that route on 64-column parts of v (the last one
// zero-padded): each output column depends on its own v column and every part
// shares the weights, so the parts are independent forwards whose outputs are
// the result's columns and whose states are its column blocks.
bool map_parts(const FwdShape &s, const DevInfo &di, const kata::MapSpec &map, Kernels &core) {
    if (map.kind == KATA_MAP_FULL || s.dtype != KATA_BF16 || s.dv == 64) return false;
    FwdShape c = s;
    c.dv = 64;
    core = select_map_kernels(c, di, map);
    return core != kSimt;
}

// Workspace: [one v part] [its output] [its state and z] [the route's workspace].
size_t parts_ws(const FwdShape &s, Kernels core, const DevInfo &di, const kata::MapSpec &map,
                bool with_state) {
    FwdShape c = s;
    c.dv = 64;
    const size_t rows = (size_t)s.BH() * s.T, n = (size_t)map.n(s.d);
    const size_t vo = 2 * round_up256(rows * 64 * 2);
    const size_t sz = with_state ? round_up256((size_t)s.BH() * n * 64 * 4) +
                                       round_up256((size_t)s.BH() * n * 4)
                                 : 0;
    return vo + sz + route_ws(c, core, di, map, with_state);
}

cudaError_t parts_run(const FwdShape &s, Kernels core, const void *q, const void *k, const void *v,
                      void *out, void *ws, const DevInfo &di, cudaStream_t st,
                      const kata::StateOut &so, const kata::MapSpec &map) {
    FwdShape c = s;
    c.dv = 64;
    const int64_t rows = (int64_t)s.BH() * s.T;
    const size_t n = (size_t)map.n(s.d), half = round_up256((size_t)rows * 64 * 2);
    uint8_t *b = static_cast<uint8_t *>(ws);
    void *vp = b, *op = b + half;
    float *sp = reinterpret_cast<float *>(b + 2 * half);
    float *zp = sp + round_up256((size_t)s.BH() * n * 64 * 4) / 4;
    const bool with_state = so.state != nullptr;
    void *cw = b + 2 * half +
               (with_state ? round_up256((size_t)s.BH() * n * 64 * 4) + round_up256((size_t)s.BH() * n * 4)
                           : 0);
    kata::StateOut cso;
    if (with_state) {
        cso.state = sp;
        cso.z = zp;
    }
    cudaError_t e = cudaSuccess;
    for (int col = 0; col < s.dv; col += 64) {
        const int w = s.dv - col < 64 ? s.dv - col : 64;
        if ((e = kata::part_copy_cols(v, s.dv, col, w, vp, 64, 0, rows, true, st)) != cudaSuccess) return e;
        if ((e = route_run(c, core, q, k, vp, op, cw, di, st, cso, map)) != cudaSuccess) return e;
        if ((e = kata::part_copy_cols(op, 64, 0, w, out, s.dv, col, rows, false, st)) != cudaSuccess) return e;
        if (with_state && (e = kata::part_copy_state(sp, zp, (int)n, so.state, so.z, s.BH(), s.dv, col, w,
                                                     col == 0, st)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// Shared body of kata_fwd_chunked and kata_fwd_chunked_state.
int fwd_chunked_impl(const void *q, const void *k, const void *v, void *out, int B, int H, int T,
                     int d, int dv, int C, int dtype, kata_stream_t stream,
                     const kata::StateOut &so, const kata::MapSpec &map = kata::MapSpec{}) {
    if (!q || !k || !v || !out) return KATA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    const size_t es = elem_size(dtype);
    const size_t nqk = (size_t)B * H * T * d * es, nvo = (size_t)B * H * T * dv * es;
    if (overlap(out, nvo, q, nqk) || overlap(out, nvo, k, nqk) || overlap(out, nvo, v, nvo))
        return KATA_ERR_ARG;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    cudaGetLastError();

    const FwdShape s{B, H, T, d, dv, C, dtype};
    const bool with_state = so.state != nullptr;
    const Kernels kn = select_map_kernels(s, di, map);
    Kernels core = kSimt;
    const bool parts = kn == kSimt && map_parts(s, di, map, core);
    const size_t wsb = parts ? parts_ws(s, core, di, map, with_state)
                             : route_ws(s, kn, di, map, with_state);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (wsb && cudaMallocAsync(&ws, wsb, st) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_ALLOC;
    }
    cudaError_t e = parts ? parts_run(s, core, q, k, v, out, ws, di, st, so, map)
                          : route_run(s, kn, q, k, v, out, ws, di, st, so, map);
    if (ws) {
        const cudaError_t ef = cudaFreeAsync(ws, st);
        if (e == cudaSuccess) e = ef;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}
}  // namespace

extern "C" {

int kata_fwd_chunked(const void *q, const void *k, const void *v, void *out, int B, int H,
                     int T, int d, int dv, int C, int dtype, kata_stream_t stream) {
    return fwd_chunked_impl(q, k, v, out, B, H, T, d, dv, C, dtype, stream, kata::StateOut{});
}

int kata_map_feature_dim(int map, int d, int g) {
    if (d < 1 || d > 64 || !valid_map(map, d, g, 0.f, 1.f)) return -1;
    kata::MapSpec ms;
    ms.kind = map;
    ms.g = g;
    return ms.n(d);
}

int kata_fwd_path_map(int B, int H, int T, int d, int dv, int C, int dtype, int map, int g) {
    if (check_fwd_shape(B, H, T, d, dv, C, dtype)) return KATA_PATH_NONE;
    if (!valid_map(map, d, g, 0.f, 1.f)) return KATA_PATH_NONE;
    DevInfo di;
    if (device_info(di)) return KATA_PATH_NONE;
    const kata::MapSpec ms = map_spec(map, g, 0.f, 1.f);
    const FwdShape s{B, H, T, d, dv, C, dtype};
    Kernels core;
    return select_map_kernels(s, di, ms) == kSimt && !map_parts(s, di, ms, core)
               ? KATA_PATH_SIMT
               : KATA_PATH_TC;
}

int kata_fwd_chunked_map(const void *q, const void *k, const void *v, void *out, int B, int H,
                         int T, int d, int dv, int C, int dtype, int map, int g, float eps,
                         float scale, kata_stream_t stream) {
    if (!valid_map(map, d, g, eps, scale)) return KATA_ERR_ARG;
    return fwd_chunked_impl(q, k, v, out, B, H, T, d, dv, C, dtype, stream, kata::StateOut{},
                            map_spec(map, g, eps, scale));
}

// The quadratic form of a shape its kernels take through the rewritings of
// kata_adapt.cu (d = 16, dv != 64), with a stream-ordered workspace.
static int adapted_quadratic(const FwdShape &s, const void *q, const void *k, const void *v,
                             void *out, cudaStream_t st, const float *gamma, int normalize) {
    cudaGetLastError();
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, kata::adapt_quad_workspace_bytes(s, gamma != nullptr), st) !=
        cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_ALLOC;
    }
    cudaError_t e = kata::adapt_quad_forward(s, q, k, v, out, ws, st, gamma, normalize);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

int kata_fwd_chunked_map_state(const void *q, const void *k, const void *v, void *out,
                               float *state, float *z, int B, int H, int T, int d, int dv, int C,
                               int dtype, int map, int g, float eps, float scale,
                               kata_stream_t stream) {
    if (!valid_map(map, d, g, eps, scale)) return KATA_ERR_ARG;
    if (!state || !z) return KATA_ERR_ARG;
    if (!aligned16(state) || !aligned16(z)) return KATA_ERR_ARG;
    const int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    const kata::MapSpec ms = map_spec(map, g, eps, scale);
    const size_t es = elem_size(dtype), BH = (size_t)B * H, n = (size_t)ms.n(d);
    const size_t nqk = BH * T * d * es, nvo = BH * T * dv * es;
    const size_t ns = BH * n * dv * 4, nz = BH * n * 4;
    if (overlap(state, ns, z, nz) || overlap(state, ns, q, nqk) || overlap(state, ns, k, nqk) ||
        overlap(state, ns, v, nvo) || overlap(state, ns, out, nvo) || overlap(z, nz, q, nqk) ||
        overlap(z, nz, k, nqk) || overlap(z, nz, v, nvo) || overlap(z, nz, out, nvo))
        return KATA_ERR_ARG;
    kata::StateOut so;
    so.state = state;
    so.z = z;
    return fwd_chunked_impl(q, k, v, out, B, H, T, d, dv, C, dtype, stream, so, ms);
}

int kata_decode_step_map(float *state, float *z, const void *q, const void *k, const void *v,
                         void *out, int B, int H, int d, int dv, int dtype, int map, int g,
                         float eps, float scale, kata_stream_t stream) {
    if (!state || !z || !q || !k || !v || !out) return KATA_ERR_ARG;
    if (!aligned16(state) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
        !aligned16(v) || !aligned16(out))
        return KATA_ERR_ARG;
    if (B < 1 || H < 1 || !valid_dtype(dtype)) return KATA_ERR_ARG;
    if (!valid_d(d) || !valid_dv(dv)) return KATA_ERR_UNSUPPORTED;
    if (!valid_map(map, d, g, eps, scale)) return KATA_ERR_ARG;
    if ((int64_t)B * H > INT32_MAX) return KATA_ERR_UNSUPPORTED;
    kata::MapSpec ms;
    ms.kind = map;
    ms.g = g;
    ms.eps = eps;
    ms.scale = scale;
    const size_t n = (size_t)ms.n(d), BH = (size_t)B * H;
    if (overlap(state, BH * n * dv * 4, z, BH * n * 4) ||
        overlap(out, BH * dv * elem_size(dtype), state, BH * n * dv * 4))
        return KATA_ERR_ARG;
    cudaGetLastError();
    const cudaError_t e = kata::decode_map_launch(state, z, q, k, v, out, (int)BH, d, dv, dtype, ms,
                                                  reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

int kata_fwd_quadratic(const void *q, const void *k, const void *v, void *out, int B, int H,
                       int T, int d, int dv, int dtype, kata_stream_t stream) {
    if (!q || !k || !v || !out) return KATA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, 64, dtype);
    if (rc) return rc;
    const size_t es = elem_size(dtype);
    const size_t nqk = (size_t)B * H * T * d * es, nvo = (size_t)B * H * T * dv * es;
    if (overlap(out, nvo, q, nqk) || overlap(out, nvo, k, nqk) || overlap(out, nvo, v, nvo))
        return KATA_ERR_ARG;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    const FwdShape s{B, H, T, d, dv, 64, dtype};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (kata::quad_supported(s, di.major, di.minor)) {
        cudaGetLastError();
        if (kata::quad_forward(s, q, k, v, out, st) != cudaSuccess) {
            cudaGetLastError();
            return KATA_ERR_CUDA;
        }
        return KATA_OK;
    }
    if (!kata::adapt_quad_supported(s, di.major, di.minor)) return KATA_ERR_UNSUPPORTED;
    return adapted_quadratic(s, q, k, v, out, st, nullptr, 1);
}

int kata_fwd_quadratic_gated(const void *q, const void *k, const void *v, const float *gamma,
                             void *out, int B, int H, int T, int d, int dv, int dtype,
                             int normalize, kata_stream_t stream) {
    if (!q || !k || !v || !gamma || !out) return KATA_ERR_ARG;
    if (normalize != 0 && normalize != 1) return KATA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(gamma))
        return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, 64, dtype);
    if (rc) return rc;
    const size_t es = elem_size(dtype);
    const size_t nqk = (size_t)B * H * T * d * es, nvo = (size_t)B * H * T * dv * es;
    const size_t ng = (size_t)B * H * T * 4;
    if (overlap(out, nvo, q, nqk) || overlap(out, nvo, k, nqk) || overlap(out, nvo, v, nvo) ||
        overlap(out, nvo, gamma, ng))
        return KATA_ERR_ARG;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    const FwdShape s{B, H, T, d, dv, 64, dtype};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!kata::quad_supported(s, di.major, di.minor)) {
        if (!kata::adapt_quad_supported(s, di.major, di.minor)) return KATA_ERR_UNSUPPORTED;
        return adapted_quadratic(s, q, k, v, out, st, gamma, normalize);
    }
    cudaGetLastError();
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, kata::quad_gated_workspace_bytes(s), st) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_ALLOC;
    }
    cudaError_t e = kata::quad_forward(s, q, k, v, out, st, gamma, normalize, ws);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

// The quadratic form's crossover against the chunked form.  At d = 32 (and
// d = 16, which runs the d = 32 kernels) the chunked form's segments fill the GPU
// at any head count, and the quadratic form is faster up to T = 6144 (measured on
// GB300: 0.6x the chunked time at T = 4096, 1.37x at T = 8192).  At d = 64 the
// chunked kernels walk each head's chunks in order on four CTAs, so their time is
// ~T x 4.2e-5 ms per wave of 152 / 4 heads, while the quadratic form's is ~BH T^2
// x 1.0e-10 ms (both fitted to GB300 timings at 1 .. 128 heads, T = 2048 .. 65536):
// the quadratic form wins while BH T < 4.2e5 x waves.
static bool quadratic_is_faster(int BH, int T, int d, int num_sms) {
    if (d != 64) return T <= 6144;
    const int64_t waves = ((int64_t)4 * BH + num_sms - 1) / num_sms;
    return (int64_t)BH * T < (int64_t)420000 * waves;
}

int kata_fwd_form(int B, int H, int T, int d, int dv, int C, int dtype) {
    if (check_fwd_shape(B, H, T, d, dv, C, dtype)) return KATA_FORM_NONE;
    DevInfo di;
    if (device_info(di)) return KATA_FORM_NONE;
    const FwdShape s{B, H, T, d, dv, 64, dtype};
    const bool quad = kata::quad_supported(s, di.major, di.minor) ||
                      kata::adapt_quad_supported(s, di.major, di.minor);
    return (quad && quadratic_is_faster(B * H, T, d, di.sms)) ? KATA_FORM_QUADRATIC
                                                            : KATA_FORM_CHUNKED;
}

int kata_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int T, int d,
             int dv, int C, int dtype, kata_stream_t stream) {
    if (!q || !k || !v || !out) return KATA_ERR_ARG;
    const int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    if (kata_fwd_form(B, H, T, d, dv, C, dtype) == KATA_FORM_QUADRATIC)
        return kata_fwd_quadratic(q, k, v, out, B, H, T, d, dv, dtype, stream);
    return kata_fwd_chunked(q, k, v, out, B, H, T, d, dv, C, dtype, stream);
}

int kata_fwd_chunked_state(const void *q, const void *k, const void *v, void *out, float *state,
                           float *z, int B, int H, int T, int d, int dv, int C, int dtype,
                           kata_stream_t stream) {
    if (!state || !z) return KATA_ERR_ARG;
    if (!aligned16(state) || !aligned16(z)) return KATA_ERR_ARG;
    const int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    const size_t es = elem_size(dtype), BH = (size_t)B * H, n = (size_t)d * (d + 1) / 2;
    const size_t nqk = BH * T * d * es, nvo = BH * T * dv * es;
    const size_t ns = BH * n * dv * 4, nz = BH * n * 4;
    if (overlap(state, ns, z, nz) || overlap(state, ns, q, nqk) || overlap(state, ns, k, nqk) ||
        overlap(state, ns, v, nvo) || overlap(state, ns, out, nvo) || overlap(z, nz, q, nqk) ||
        overlap(z, nz, k, nqk) || overlap(z, nz, v, nvo) || overlap(z, nz, out, nvo))
        return KATA_ERR_ARG;
    kata::StateOut so;
    so.state = state;
    so.z = z;
    return fwd_chunked_impl(q, k, v, out, B, H, T, d, dv, C, dtype, stream, so);
}

int kata_fwd_chunked_host(const void *q, const void *k, const void *v, void *out, int B,
                          int H, int T, int d, int dv, int C, int dtype,
                          kata_stream_t stream) {
    if (!q || !k || !v || !out) return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    cudaGetLastError();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = elem_size(dtype);
    const int BH = B * H;
    const size_t hqk = (size_t)T * d * es, hvo = (size_t)T * dv * es;   // bytes per head
    const size_t nqk = BH * hqk, nvo = BH * hvo;
    // Heads are independent: for large transfers the heads are cut into groups so
    // that later groups are copied in while group g runs and group g - 1 is copied
    // out (two streams in, alternating groups; one out; the forward on the
    // caller's stream).  A group keeps the whole call's kernel path and still
    // fills the GPU.
    const FwdShape whole{1, BH, T, d, dv, C, dtype};
    const int path = select_path(whole, di);
    int ng = 1;
    if (2 * nqk + 2 * nvo >= ((size_t)64 << 20)) {
        for (int cand : {8, 4, 2}) {
            const int hg = BH / cand;
            if (BH % cand != 0 || hg < 1) continue;
            const FwdShape part{1, hg, T, d, dv, C, dtype};
            const bool fills = path == KATA_PATH_SIMT || hg * (int64_t)((T + 127) / 128) >= di.sms;
            if (select_path(part, di) == path && fills) {
                ng = cand;
                break;
            }
        }
    }
    const int hg = BH / ng;
    char *dq = nullptr, *dk = nullptr, *dvv = nullptr, *dout = nullptr;
    rc = KATA_OK;
    if (cudaMallocAsync((void **)&dq, nqk, st) != cudaSuccess ||
        cudaMallocAsync((void **)&dk, nqk, st) != cudaSuccess ||
        cudaMallocAsync((void **)&dvv, nvo, st) != cudaSuccess ||
        cudaMallocAsync((void **)&dout, nvo, st) != cudaSuccess) {
        cudaGetLastError();
        rc = KATA_ERR_ALLOC;
    }
    cudaStream_t sin2[2] = {nullptr, nullptr}, sout = nullptr;
    cudaEvent_t ready = nullptr, done = nullptr, ev_in[8] = {}, ev_run[8] = {};
    bool ev_ok = rc == KATA_OK &&
                 cudaStreamCreateWithFlags(&sin2[0], cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&sin2[1], cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&sout, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&done, cudaEventDisableTiming) == cudaSuccess;
    for (int g = 0; g < ng && ev_ok; ++g)
        ev_ok = cudaEventCreateWithFlags(&ev_in[g], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&ev_run[g], cudaEventDisableTiming) == cudaSuccess;
    if (rc == KATA_OK && !ev_ok) rc = KATA_ERR_CUDA;
    if (rc == KATA_OK) {
        // the buffers were allocated on the caller's stream: order the copy streams after it
        if (cudaEventRecord(ready, st) != cudaSuccess ||
            cudaStreamWaitEvent(sin2[0], ready, 0) != cudaSuccess ||
            cudaStreamWaitEvent(sin2[1], ready, 0) != cudaSuccess ||
            cudaStreamWaitEvent(sout, ready, 0) != cudaSuccess)
            rc = KATA_ERR_CUDA;
    }
    for (int g = 0; g < ng && rc == KATA_OK; ++g) {
        const size_t oq = (size_t)g * hg * hqk, ov = (size_t)g * hg * hvo;
        cudaStream_t sin = sin2[g & 1];
        if (cudaMemcpyAsync(dq + oq, (const char *)q + oq, hg * hqk, cudaMemcpyHostToDevice, sin) != cudaSuccess ||
            cudaMemcpyAsync(dk + oq, (const char *)k + oq, hg * hqk, cudaMemcpyHostToDevice, sin) != cudaSuccess ||
            cudaMemcpyAsync(dvv + ov, (const char *)v + ov, hg * hvo, cudaMemcpyHostToDevice, sin) != cudaSuccess ||
            cudaEventRecord(ev_in[g], sin) != cudaSuccess)
            rc = KATA_ERR_CUDA;
    }
    for (int g = 0; g < ng && rc == KATA_OK; ++g) {
        const size_t oq = (size_t)g * hg * hqk, ov = (size_t)g * hg * hvo;
        if (cudaStreamWaitEvent(st, ev_in[g], 0) != cudaSuccess) {
            rc = KATA_ERR_CUDA;
            break;
        }
        rc = kata_fwd_chunked(dq + oq, dk + oq, dvv + ov, dout + ov, 1, hg, T, d, dv, C, dtype, stream);
        if (rc != KATA_OK) break;
        if (cudaEventRecord(ev_run[g], st) != cudaSuccess || cudaStreamWaitEvent(sout, ev_run[g], 0) != cudaSuccess ||
            cudaMemcpyAsync((char *)out + ov, dout + ov, hg * hvo, cudaMemcpyDeviceToHost, sout) != cudaSuccess)
            rc = KATA_ERR_CUDA;
    }
    // the buffers are freed on the caller's stream after both copy streams are done
    for (cudaStream_t x : {sin2[0], sin2[1], sout})
        if (x && done && cudaEventRecord(done, x) == cudaSuccess) cudaStreamWaitEvent(st, done, 0);
    if (dq) cudaFreeAsync(dq, st);
    if (dk) cudaFreeAsync(dk, st);
    if (dvv) cudaFreeAsync(dvv, st);
    if (dout) cudaFreeAsync(dout, st);
    if (cudaStreamSynchronize(st) != cudaSuccess && rc == KATA_OK) rc = KATA_ERR_CUDA;
    for (cudaStream_t x : {sin2[0], sin2[1], sout})
        if (x && cudaStreamSynchronize(x) != cudaSuccess && rc == KATA_OK) rc = KATA_ERR_CUDA;
    for (int g = 0; g < 8; ++g) {
        if (ev_in[g]) cudaEventDestroy(ev_in[g]);
        if (ev_run[g]) cudaEventDestroy(ev_run[g]);
    }
    if (ready) cudaEventDestroy(ready);
    if (done) cudaEventDestroy(done);
    for (cudaStream_t x : {sin2[0], sin2[1], sout})
        if (x) cudaStreamDestroy(x);
    cudaGetLastError();
    return rc;
}

int kata_decode_step(float *state, float *z, const void *q, const void *k, const void *v,
                     void *out, int B, int H, int d, int dv, int dtype,
                     kata_stream_t stream) {
    if (!state || !z || !q || !k || !v || !out) return KATA_ERR_ARG;
    if (!aligned16(state) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
        !aligned16(v) || !aligned16(out))
        return KATA_ERR_ARG;
    if (B < 1 || H < 1 || !valid_dtype(dtype)) return KATA_ERR_ARG;
    if (!valid_d(d) || !valid_dv(dv)) return KATA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > INT32_MAX) return KATA_ERR_UNSUPPORTED;
    const size_t n = (size_t)d * (d + 1) / 2;
    const size_t BH = (size_t)B * H;
    if (overlap(state, BH * n * dv * 4, z, BH * n * 4) ||
        overlap(out, BH * dv * elem_size(dtype), state, BH * n * dv * 4))
        return KATA_ERR_ARG;
    cudaGetLastError();
    const cudaError_t e = kata::decode_launch(state, z, q, k, v, out, (int)BH, d, dv, dtype,
                                              reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

int kata_fwd_chunked_gated(const void *q, const void *k, const void *v, const float *gamma,
                           void *out, float *state, float *z, int B, int H, int T, int d, int dv,
                           int C, int dtype, int normalize, kata_stream_t stream) {
    if (!q || !k || !v || !gamma || !out) return KATA_ERR_ARG;
    if (!state != !z) return KATA_ERR_ARG;
    if (normalize != 0 && normalize != 1) return KATA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(gamma))
        return KATA_ERR_ARG;
    if (state && (!aligned16(state) || !aligned16(z))) return KATA_ERR_ARG;
    int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    const size_t es = elem_size(dtype), BH = (size_t)B * H, n = (size_t)d * (d + 1) / 2;
    const size_t nqk = BH * T * d * es, nvo = BH * T * dv * es, ng = BH * T * 4;
    if (overlap(out, nvo, q, nqk) || overlap(out, nvo, k, nqk) || overlap(out, nvo, v, nvo) ||
        overlap(out, nvo, gamma, ng))
        return KATA_ERR_ARG;
    if (state) {
        const size_t ns = BH * n * dv * 4, nz = BH * n * 4;
        const void *ins[5] = {q, k, v, gamma, out};
        const size_t lens[5] = {nqk, nqk, nvo, ng, nvo};
        if (overlap(state, ns, z, nz)) return KATA_ERR_ARG;
        for (int i = 0; i < 5; ++i)
            if (overlap(state, ns, ins[i], lens[i]) || overlap(z, nz, ins[i], lens[i]))
                return KATA_ERR_ARG;
    }
    DevInfo di;
    if ((rc = device_info(di))) return rc;
    cudaGetLastError();
    const FwdShape s{B, H, T, d, dv, C, dtype};
    const bool with_state = state != nullptr;
    const bool tc = kata::tc_supported(s, di.major, di.minor);
    const bool wide = !tc && kata::gated_wide_supported(s, di.major, di.minor, di.sms, with_state);
    const kata::GatedCore ad = tc || wide ? kata::GatedCore::None
                                          : kata::adapt_gated_core(s, di.major, di.minor, di.sms,
                                                                   with_state);
    const bool adapt = ad != kata::GatedCore::None;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    const size_t wsb = tc      ? kata::tc_gated_workspace_bytes(s, di.sms, with_state)
                       : wide  ? kata::gated_wide_workspace_bytes(s, with_state)
                       : adapt ? kata::adapt_gated_workspace_bytes(s, ad, di.sms, with_state)
                               : kata::gated_workspace_bytes(s);
    if (cudaMallocAsync(&ws, wsb, st) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_ALLOC;
    }
    kata::StateOut so;
    so.state = state;
    so.z = z;
    cudaError_t e =
        tc      ? kata::tc_forward_gated(s, q, k, v, gamma, out, ws, di.sms, st, so, normalize)
        : wide  ? kata::gated_wide_forward(s, q, k, v, gamma, out, ws, st, so, normalize)
        : adapt ? kata::adapt_gated_forward(s, ad, q, k, v, gamma, out, ws, di.sms, st, so,
                                            normalize)
                : kata::gated_forward(s, q, k, v, gamma, out, ws, st, so, normalize);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

// GatedKATA in whichever exact form is faster for the shape.  Per token the
// gated quadratic form costs work in proportion to T, the gated chunked form a
// constant.  Measured on GB300 (bf16, dv = 64, per token and head): at d = 32
// the chunked form runs on the tensor cores at 1.3 ns for every T, the
// quadratic form at 1.10 ns at T = 8192 and 1.90 ns at T = 16384, so they level
// near T = 10k.  At d = 64 the chunked call takes its output from the same gated
// quadratic kernel up to T = 262144 (7.1 ns at T = 65536), so the bound matters
// only past that, where the chunked form runs on CUDA cores at ~35 ns.
static int gated_quadratic_max_t(int d) { return d == 32 ? 10240 : 65536; }

int kata_fwd_path_gated(int B, int H, int T, int d, int dv, int C, int dtype) {
    if (check_fwd_shape(B, H, T, d, dv, C, dtype)) return KATA_PATH_NONE;
    DevInfo di;
    if (device_info(di)) return KATA_PATH_NONE;
    const FwdShape s{B, H, T, d, dv, C, dtype};
    return kata::tc_supported(s, di.major, di.minor) ||
                   kata::gated_wide_supported(s, di.major, di.minor, di.sms, false) ||
                   kata::adapt_gated_core(s, di.major, di.minor, di.sms, false) !=
                       kata::GatedCore::None
               ? KATA_PATH_TC
               : KATA_PATH_SIMT;
}

int kata_fwd_gated_form(int B, int H, int T, int d, int dv, int C, int dtype) {
    if (check_fwd_shape(B, H, T, d, dv, C, dtype)) return KATA_FORM_NONE;
    DevInfo di;
    if (device_info(di)) return KATA_FORM_NONE;
    const FwdShape s{B, H, T, d, dv, 64, dtype};
    const bool quad = kata::quad_supported(s, di.major, di.minor) ||
                      kata::adapt_quad_supported(s, di.major, di.minor);
    return (quad && T <= gated_quadratic_max_t(d < 32 ? 32 : d)) ? KATA_FORM_QUADRATIC
                                                                 : KATA_FORM_CHUNKED;
}

int kata_fwd_gated(const void *q, const void *k, const void *v, const float *gamma, void *out,
                   int B, int H, int T, int d, int dv, int C, int dtype, int normalize,
                   kata_stream_t stream) {
    if (!q || !k || !v || !gamma || !out) return KATA_ERR_ARG;
    const int rc = check_fwd_shape(B, H, T, d, dv, C, dtype);
    if (rc) return rc;
    if (kata_fwd_gated_form(B, H, T, d, dv, C, dtype) == KATA_FORM_QUADRATIC)
        return kata_fwd_quadratic_gated(q, k, v, gamma, out, B, H, T, d, dv, dtype, normalize,
                                        stream);
    return kata_fwd_chunked_gated(q, k, v, gamma, out, nullptr, nullptr, B, H, T, d, dv, C, dtype,
                                  normalize, stream);
}

int kata_decode_step_gated(float *state, float *z, const void *q, const void *k, const void *v,
                           const float *gamma, void *out, int B, int H, int d, int dv,
                           int dtype, int normalize, kata_stream_t stream) {
    if (!state || !z || !q || !k || !v || !gamma || !out) return KATA_ERR_ARG;
    if (normalize != 0 && normalize != 1) return KATA_ERR_ARG;
    if (!aligned16(state) || !aligned16(z) || !aligned16(q) || !aligned16(k) ||
        !aligned16(v) || !aligned16(out) || !aligned16(gamma))
        return KATA_ERR_ARG;
    if (B < 1 || H < 1 || !valid_dtype(dtype)) return KATA_ERR_ARG;
    if (!valid_d(d) || !valid_dv(dv)) return KATA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > INT32_MAX) return KATA_ERR_UNSUPPORTED;
    const size_t n = (size_t)d * (d + 1) / 2;
    const size_t BH = (size_t)B * H;
    if (overlap(state, BH * n * dv * 4, z, BH * n * 4) ||
        overlap(out, BH * dv * elem_size(dtype), state, BH * n * dv * 4) ||
        overlap(gamma, BH * 4, state, BH * n * dv * 4) || overlap(gamma, BH * 4, z, BH * n * 4))
        return KATA_ERR_ARG;
    cudaGetLastError();
    const cudaError_t e = kata::decode_launch(state, z, q, k, v, out, (int)BH, d, dv, dtype,
                                              reinterpret_cast<cudaStream_t>(stream), gamma,
                                              normalize);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

int kata_sync_status(kata_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    const int e = kata::tc_take_error(), e64 = kata::tc64_take_error(), eq = kata::quad_take_error(),
              ep = kata::pair_take_error(), ef = kata::feat_take_error();
    if (e < 0 || e64 < 0 || eq < 0 || ep < 0 || ef < 0) return KATA_ERR_CUDA;
    return (e | e64 | eq | ep | ef) ? KATA_ERR_TIMEOUT : KATA_OK;
}

int kata_test_arm_stall(void) {
    kata::tc_arm_stall();
    return KATA_OK;
}

int kata_lift_map(const void *x, float *phi, int64_t rows, int d, int dtype, int map, int g,
                  float eps, float scale, kata_stream_t stream) {
    if (!x || !phi || rows < 1 || d < 1 || !valid_dtype(dtype)) return KATA_ERR_ARG;
    if (d > 64) return KATA_ERR_UNSUPPORTED;
    if (!valid_map(map, d, g, eps, scale)) return KATA_ERR_ARG;
    if (!aligned16(x) || !aligned16(phi)) return KATA_ERR_ARG;
    kata::MapSpec ms;
    ms.kind = map;
    ms.g = g;
    ms.eps = eps;
    ms.scale = scale;
    cudaGetLastError();
    const cudaError_t e =
        kata::lift_launch(x, phi, rows, d, dtype, reinterpret_cast<cudaStream_t>(stream), ms);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

int kata_lift(const void *x, float *phi, int64_t rows, int d, int dtype, kata_stream_t stream) {
    if (!x || !phi || rows < 1 || d < 1 || !valid_dtype(dtype)) return KATA_ERR_ARG;
    if (d > 64) return KATA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(phi)) return KATA_ERR_ARG;
    cudaGetLastError();
    const cudaError_t e =
        kata::lift_launch(x, phi, rows, d, dtype, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}

}  // extern "C"
