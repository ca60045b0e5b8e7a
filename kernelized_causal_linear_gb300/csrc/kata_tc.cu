// tcgen05 tensor-core path of the KATA chunked forward (bf16 inputs, sm_103a).
#include "kata_internal.cuh"

namespace kata {

bool tc_supported(const FwdShape &s, int cc_major, int cc_minor) {
    (void)s;
    (void)cc_major;
    (void)cc_minor;
    return false;
}

size_t tc_workspace_bytes(const FwdShape &s, int num_sms) {
    (void)s;
    (void)num_sms;
    return 0;
}

cudaError_t tc_forward(const FwdShape &s, const void *q, const void *k, const void *v,
                       void *out, void *workspace, int num_sms, cudaStream_t stream) {
    (void)s; (void)q; (void)k; (void)v; (void)out; (void)workspace; (void)num_sms;
    (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace kata
