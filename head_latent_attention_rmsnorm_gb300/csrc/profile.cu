// profile.cu -- launch accounting and opt-in per-kernel event timing of libmla.
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "mla_internal.h"

namespace mla {
namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_prof_on{false};
std::mutex g_mu;   // guards the event pool and the records (several host threads may launch)

struct Pair {
    cudaEvent_t a, b;
};
std::map<std::string, std::vector<Pair>> g_rec;
std::vector<cudaEvent_t> g_pool;
thread_local cudaEvent_t g_open = nullptr;

// Callers hold g_mu.
cudaEvent_t get_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Callers hold g_mu.
void recycle_all() {
    for (auto &kv : g_rec)
        for (auto &p : kv.second) {
            g_pool.push_back(p.a);
            g_pool.push_back(p.b);
        }
    g_rec.clear();
}

}  // namespace

void prof_begin(const char *, cudaStream_t st) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    g_open = get_event();
    if (g_open) cudaEventRecord(g_open, st);
}

void prof_end(const char *name, cudaStream_t st) {
    if (!g_prof_on.load(std::memory_order_relaxed) || !g_open) return;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaEvent_t b = get_event();
    if (!b) return;
    cudaEventRecord(b, st);
    g_rec[name].push_back(Pair{g_open, b});
    g_open = nullptr;
}

}  // namespace mla

extern "C" {

unsigned long long mla_launch_count(void) { return mla::g_launches.load(); }

void mla_profile_enable(int on) {
    mla::g_prof_on = on != 0;
    if (!on) {
        cudaDeviceSynchronize();
        std::lock_guard<std::mutex> lock(mla::g_mu);
        mla::recycle_all();
    }
}

void mla_profile_reset(void) {
    cudaDeviceSynchronize();
    std::lock_guard<std::mutex> lock(mla::g_mu);
    mla::recycle_all();
}

int mla_profile_kernel(const char *name, long long *launches, double *total_ms) {
    *launches = 0;
    *total_ms = 0.0;
    std::vector<mla::Pair> pairs;
    {
        std::lock_guard<std::mutex> lock(mla::g_mu);
        auto it = mla::g_rec.find(name);
        if (it == mla::g_rec.end()) return 0;
        pairs = it->second;
    }
    for (auto &p : pairs) {
        if (cudaEventSynchronize(p.b) != cudaSuccess) return -1;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return -1;
        *total_ms += ms;
        *launches += 1;
    }
    return 0;
}

}  // extern "C"
