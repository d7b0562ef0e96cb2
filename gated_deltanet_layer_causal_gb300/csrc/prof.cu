// Launch accounting and optional per-kernel timing.
//
// Every kernel launch of the library goes through a ProfScope: it bumps a
// launch counter and, while timing is enabled, brackets the launch with a pair
// of CUDA events recorded on the launch's own stream.  gdn_profile_report()
// waits for those events and returns, per kernel name, the number of timed
// launches and their total device time.  Timing is off by default and costs
// nothing then but the counter.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gdn.h"
#include "prof.h"

namespace gdn {
namespace {

struct Rec {
    const char* name;
    cudaEvent_t a, b;
};

std::atomic<long long> g_launches{0};
std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Rec> g_open;              // recorded, not yet reported
std::vector<cudaEvent_t> g_free;      // event pool
thread_local std::vector<Rec> t_stack;

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

void prof_begin(const char* name, cudaStream_t st) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r{name, take_event(), take_event()};
    cudaEventRecord(r.a, st);
    t_stack.push_back(r);
}

void prof_end(cudaStream_t st) {
    if (!g_enabled.load(std::memory_order_relaxed) || t_stack.empty()) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r = t_stack.back();
    t_stack.pop_back();
    cudaEventRecord(r.b, st);
    g_open.push_back(r);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

int64_t gdn_launch_count(void) { return (int64_t)g_launches.load(); }

gdn_status gdn_profile_enable(int32_t on) {
    g_enabled.store(on ? 1 : 0);
    return GDN_OK;
}

gdn_status gdn_profile_report(char* buf, size_t buf_bytes) {
    if (buf == nullptr || buf_bytes == 0) return GDN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    std::map<std::string, std::pair<long long, double>> acc;
    std::vector<std::string> order;
    for (const Rec& r : g_open) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return GDN_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return GDN_ERR_CUDA;
        auto it = acc.find(r.name);
        if (it == acc.end()) {
            order.push_back(r.name);
            acc[r.name] = {1, ms};
        } else {
            it->second.first += 1;
            it->second.second += ms;
        }
        g_free.push_back(r.a);
        g_free.push_back(r.b);
    }
    g_open.clear();
    size_t used = 0;
    buf[0] = 0;
    for (const std::string& n : order) {
        int w = std::snprintf(buf + used, buf_bytes - used, "%s %lld %.6f\n", n.c_str(),
                              acc[n].first, acc[n].second);
        if (w < 0 || (size_t)w >= buf_bytes - used) return GDN_ERR_INVALID_ARG;
        used += (size_t)w;
    }
    return GDN_OK;
}

}  // extern "C"
