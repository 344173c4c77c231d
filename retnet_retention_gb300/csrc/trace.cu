// Launch tracing: CUDA events recorded on the launching stream around every
// kernel the library enqueues, while tracing is enabled.  Used by the
// benchmark to time each kernel of a multi-kernel call (the segment-state,
// scan and output kernels of a long-sequence prefill) on the device clock.
#include <mutex>
#include <vector>

#include "launch.h"
#include "trace.h"

namespace la {

namespace {

struct Slot {
    const char* name;
    cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Slot> g_pool;   // created on enable, reused
size_t g_used = 0;

}  // namespace

TraceScope::TraceScope(const char* name, cudaStream_t s) : stream_(s), slot_(-1) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on || g_used >= g_pool.size()) return;
    slot_ = (int)g_used++;
    g_pool[slot_].name = name;
    cudaEventRecord(g_pool[slot_].start, stream_);
}

TraceScope::~TraceScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEventRecord(g_pool[slot_].stop, stream_);
}

}  // namespace la

extern "C" {

int la_trace_enable(int capacity) {
    using namespace la;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& s : g_pool) {
        cudaEventDestroy(s.start);
        cudaEventDestroy(s.stop);
    }
    g_pool.clear();
    g_used = 0;
    g_on = false;
    if (capacity <= 0) return LA_OK;
    g_pool.resize((size_t)capacity);
    for (auto& s : g_pool) {
        s.name = nullptr;
        if (cudaEventCreate(&s.start) != cudaSuccess || cudaEventCreate(&s.stop) != cudaSuccess) {
            g_pool.clear();
            return LA_ERR_CUDA;
        }
    }
    g_on = true;
    return LA_OK;
}

int la_trace_collect(la_trace_record* out, int max_records) {
    using namespace la;
    std::lock_guard<std::mutex> lk(g_mu);
    int n = 0;
    for (size_t i = 0; i < g_used && n < max_records; ++i) {
        Slot& s = g_pool[i];
        if (cudaEventSynchronize(s.stop) != cudaSuccess) return -LA_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, s.start, s.stop) != cudaSuccess) return -LA_ERR_CUDA;
        out[n].kernel = s.name;
        out[n].ms = ms;
        ++n;
    }
    g_used = 0;
    return n;
}

}  // extern "C"
