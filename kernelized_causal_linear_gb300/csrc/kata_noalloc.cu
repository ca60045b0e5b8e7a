// kata_fwd_chunked_noalloc: the chunked forward without any device allocation.
//
// Some callers cannot allocate device memory at the point where they run the
// forward: code inside a framework that owns all device memory through its own
// pool (and forbids other allocators), real-time or embedded hosts that must
// not allocate after start-up, and callers replaying pre-recorded GPU work that
// may not contain allocations.  For them this entry point runs the same kernels
// as kata_fwd_chunked, but its scratch lives in one fixed-size device array
// that is part of this library's device image instead of being taken from the
// stream-ordered pool.
//
// Properties a user must know:
//   * Path and capacity: the call takes the kernel family kata_fwd_chunked
//     takes for the shape, and needs the scratch kata_fwd_workspace_size
//     reports for it.  Capacity is KATA_NOALLOC_SCRATCH_BYTES (32 MiB); a
//     shape that needs more is rejected with KATA_ERR_SCRATCH_LIMIT before any
//     device work.  Every bf16 shape of the d = 32 tensor path fits on a
//     152-SM GPU (its scratch is a few segment records per head).  The d = 64
//     tensor path keeps fp32 partial numerators of every token (about 1 KB per
//     token and head), so it fits up to roughly 32 K tokens x heads; the CUDA-
//     core path keeps every chunk's state, B*H*(NC + NC/16 + 1)*n*(dv+1)*4
//     bytes with NC = ceil(T/C).
//   * Memory: the array is part of this library's device code.  It is
//     reserved when that code is loaded on a device: under the default lazy
//     loading, at this entry point's first call there; with eager module
//     loading (CUDA_MODULE_LOADING=EAGER), on every device context the
//     process creates.  It stays reserved until the process exits.
//   * Set-up: the first call on each device (with that device current) looks
//     up the array's device address with cudaGetSymbolAddress, which may load
//     this part of the library's device code.  Make that first call before
//     any stream capture begins.
//   * Shared state: all calls use the same array and it keeps whatever the last
//     call left in it.  Nothing has to start at zero: every byte the kernels
//     read from it is written earlier in the same call.  Two calls whose work
//     overlaps on the GPU (for example on two streams without ordering between
//     them) race on the array and produce wrong results; order them.
//   * No call allocates: no cudaMalloc/cudaMallocAsync/cudaFree and no
//     allocating library routine.
#include <mutex>

#include "../../include/kata.h"
#include "kata_dispatch.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KATA_NOALLOC_SCRATCH_BYTES];

struct NoallocDevice {
    void *scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int major = 0, minor = 0, sms = 0;
    bool ready = false;
};

// Once per device, with that device current: resolve the array's address and
// read the properties the path selection needs.
int noalloc_setup(NoallocDevice &out) {
    static std::mutex mu;
    static NoallocDevice devs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    NoallocDevice &d = devs[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return KATA_ERR_CUDA;
        }
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return KATA_ERR_CUDA;
        }
        d.scratch = p;
        d.ready = true;
    }
    out = d;
    return KATA_OK;
}

bool is_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int kata_fwd_chunked_noalloc(const void *q, const void *k, const void *v, void *out,
                                        int B, int H, int T, int d, int dv, int C, int dtype,
                                        kata_stream_t stream) {
    // the argument rules of kata_fwd_chunked
    if (!q || !k || !v || !out) return KATA_ERR_ARG;
    if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(out))
        return KATA_ERR_ARG;
    if (B < 1 || H < 1 || T < 1) return KATA_ERR_ARG;
    if (dtype != KATA_F32 && dtype != KATA_BF16) return KATA_ERR_ARG;
    if ((int64_t)B * H > 65535) return KATA_ERR_UNSUPPORTED;
    if (!(d == 16 || d == 32 || d == 64) || !(dv == 16 || dv == 32 || dv == 64 || dv == 128) ||
        !(C == 32 || C == 64 || C == 128))
        return KATA_ERR_UNSUPPORTED;
    const size_t es = dtype == KATA_F32 ? 4 : 2;
    const size_t nqk = (size_t)B * H * T * d * es, nvo = (size_t)B * H * T * dv * es;
    if (ranges_overlap(out, nvo, q, nqk) || ranges_overlap(out, nvo, k, nqk) ||
        ranges_overlap(out, nvo, v, nvo))
        return KATA_ERR_ARG;

    NoallocDevice dev;
    int rc = noalloc_setup(dev);
    if (rc) return rc;
    cudaGetLastError();

    // the kernel family, and so the scratch size, kata_fwd_chunked takes for this shape
    const kata::FwdShape s{B, H, T, d, dv, C, dtype};
    const kata::FwdKernels kn = kata::select_fwd_kernels(s, dev.major, dev.minor, dev.sms);
    if (kata::fwd_workspace_bytes(s, kn, dev.sms) > (size_t)KATA_NOALLOC_SCRATCH_BYTES)
        return KATA_ERR_SCRATCH_LIMIT;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = kata::fwd_launch(s, kn, q, k, v, out, dev.scratch, dev.sms, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return KATA_OK;
}
