// Per-stage device timing of libkata's launches (see kata_trace_begin in
// include/kata.h).  Each traced launch is bracketed by two CUDA events recorded
// on the launch's own stream; kata_trace_end reads them back.
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/kata.h"
#include "kata_internal.cuh"

namespace kata {
namespace {

struct Record {
    std::string stage;
    cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Record> g_records;

}  // namespace

TraceScope::TraceScope(const char *stage, cudaStream_t stream)
    : stage_(stage), stream_(stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_on) return;
    if (cudaEventCreate(&start_) != cudaSuccess) {
        cudaGetLastError();
        start_ = nullptr;
        return;
    }
    cudaEventRecord(start_, stream_);
}

TraceScope::~TraceScope() {
    if (!start_) return;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaEvent_t stop = nullptr;
    if (cudaEventCreate(&stop) != cudaSuccess) {
        cudaGetLastError();
        cudaEventDestroy(start_);
        return;
    }
    cudaEventRecord(stop, stream_);
    g_records.push_back(Record{stage_, start_, stop});
}

}  // namespace kata

extern "C" {

int kata_trace_begin(void) {
    std::lock_guard<std::mutex> lock(kata::g_mu);
    for (auto &r : kata::g_records) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    kata::g_records.clear();
    kata::g_on = true;
    return KATA_OK;
}

int kata_trace_end(kata_trace_stage *stages, int max_stages, int *n_stages) {
    if (max_stages < 0 || (max_stages > 0 && !stages)) return KATA_ERR_ARG;
    std::vector<kata::Record> recs;
    {
        std::lock_guard<std::mutex> lock(kata::g_mu);
        kata::g_on = false;
        recs.swap(kata::g_records);
    }
    std::vector<kata_trace_stage> agg;
    int rc = KATA_OK;
    for (auto &r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
            cudaGetLastError();
            rc = KATA_ERR_CUDA;
        }
        kata_trace_stage *slot = nullptr;
        for (auto &a : agg)
            if (r.stage == a.name) slot = &a;
        if (!slot) {
            kata_trace_stage s{};
            std::strncpy(s.name, r.stage.c_str(), sizeof(s.name) - 1);
            agg.push_back(s);
            slot = &agg.back();
        }
        slot->launches += 1;
        slot->total_ms += ms;
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    for (int i = 0; i < (int)agg.size() && i < max_stages; ++i) stages[i] = agg[i];
    if (n_stages) *n_stages = (int)agg.size();
    return rc;
}

}  // extern "C"
