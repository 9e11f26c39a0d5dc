// Per-kernel timing for diagnostics.  While enabled, every kernel the library
// launches is bracketed by two CUDA events recorded on its own stream; the
// host reads the accumulated device time per kernel name afterwards.  Off by
// default; not for use under stream capture (event creation is not
// capturable).
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "gdr.h"
#include "launch.h"

namespace gdr {
namespace {

struct Rec {
    const char* name;
    cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

}  // namespace

KernelTimer::KernelTimer(const char* name, cudaStream_t s) : name_(name), stream_(s), a_(nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on) return;
    a_ = take_event();
    cudaEventRecord(static_cast<cudaEvent_t>(a_), stream_);
}

KernelTimer::~KernelTimer() {
    if (!a_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = take_event();
    cudaEventRecord(b, stream_);
    g_recs.push_back(Rec{name_, static_cast<cudaEvent_t>(a_), b});
}

}  // namespace gdr

using namespace gdr;

extern "C" {

int gdr_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_on = on != 0;
    return GDR_OK;
}

int gdr_profile_read(int max_kernels, char* names, size_t name_cap, double* total_ms, int* launches,
                     int* n_kernels) {
    std::vector<Rec> recs;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        recs.swap(g_recs);
    }
    std::map<std::string, std::pair<double, int>> agg;
    int rc = GDR_OK;
    for (const Rec& r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            rc = GDR_ERR_LAUNCH;
        auto& e = agg[r.name];
        e.first += ms;
        e.second += 1;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (const Rec& r : recs) {
            g_free.push_back(r.a);
            g_free.push_back(r.b);
        }
    }
    int i = 0;
    size_t used = 0;
    if (names && name_cap) names[0] = '\0';
    for (const auto& kv : agg) {
        if (i >= max_kernels) break;
        if (total_ms) total_ms[i] = kv.second.first;
        if (launches) launches[i] = kv.second.second;
        if (names && used + kv.first.size() + 2 < name_cap) {
            std::memcpy(names + used, kv.first.c_str(), kv.first.size());
            used += kv.first.size();
            names[used++] = ',';
            names[used] = '\0';
        }
        ++i;
    }
    if (n_kernels) *n_kernels = i;
    return rc;
}

}  // extern "C"
