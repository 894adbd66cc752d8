// profile.cu -- launch accounting and opt-in per-kernel event timing of libmla.
#include <atomic>
#include <map>
#include <string>
#include <vector>

#include "mla_internal.h"

namespace mla {
namespace {

std::atomic<unsigned long long> g_launches{0};
bool g_prof_on = false;

struct Pair {
    cudaEvent_t a, b;
};
std::map<std::string, std::vector<Pair>> g_rec;
std::vector<cudaEvent_t> g_pool;
thread_local cudaEvent_t g_open = nullptr;

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
    if (!g_prof_on) return;
    g_open = get_event();
    if (g_open) cudaEventRecord(g_open, st);
}

void prof_end(const char *name, cudaStream_t st) {
    if (!g_prof_on || !g_open) return;
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
        mla::recycle_all();
    }
}

void mla_profile_reset(void) {
    cudaDeviceSynchronize();
    mla::recycle_all();
}

int mla_profile_kernel(const char *name, long long *launches, double *total_ms) {
    *launches = 0;
    *total_ms = 0.0;
    auto it = mla::g_rec.find(name);
    if (it == mla::g_rec.end()) return 0;
    for (auto &p : it->second) {
        if (cudaEventSynchronize(p.b) != cudaSuccess) return -1;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return -1;
        *total_ms += ms;
        *launches += 1;
    }
    return 0;
}

}  // extern "C"
