// kda_profile.cu -- optional per-kernel device timing (kda_profile_enable / kda_profile_read).
//
// While enabled, each launch made through the C ABI is bracketed by CUDA events recorded on the
// launching stream.  Reading synchronises on the recorded events and sums elapsed time per kernel
// name.  Events are pooled and reused; nothing touches device memory.
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kda_internal.cuh"

namespace kda {

namespace {

struct Pending {
    int id;
    cudaEvent_t start, stop;
};
struct Acc {
    std::string name;
    int64_t launches;
    double ms;
};

std::mutex g_mu;
bool g_on = false;
int g_cur_id = -1;
cudaEvent_t g_cur_start = nullptr;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
std::vector<Acc> g_acc;

cudaEvent_t take_event()
{
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Folds every pending record into the accumulators (synchronises on their stop events).
bool drain_locked()
{
    bool ok = true;
    for (const Pending& p : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) {
            ok = false;
        } else {
            g_acc[p.id].launches += 1;
            g_acc[p.id].ms += ms;
        }
        g_pool.push_back(p.start);
        g_pool.push_back(p.stop);
    }
    g_pending.clear();
    return ok;
}

}  // namespace

void prof_start(const char* name, cudaStream_t s)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on) return;
    int id = -1;
    for (size_t i = 0; i < g_acc.size(); ++i) {
        if (g_acc[i].name == name) id = (int)i;
    }
    if (id < 0) {
        g_acc.push_back(Acc{name, 0, 0.0});
        id = (int)g_acc.size() - 1;
    }
    g_cur_id = id;
    g_cur_start = take_event();
    if (g_cur_start) cudaEventRecord(g_cur_start, s);
}

void prof_stop(cudaStream_t s)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on || g_cur_start == nullptr) return;
    cudaEvent_t stop = take_event();
    if (stop == nullptr) return;
    cudaEventRecord(stop, s);
    g_pending.push_back(Pending{g_cur_id, g_cur_start, stop});
    g_cur_start = nullptr;
    if (g_pending.size() > 8192) drain_locked();
}

}  // namespace kda

extern "C" {

kda_status_t kda_profile_enable(int enable)
{
    std::lock_guard<std::mutex> lk(kda::g_mu);
    kda::drain_locked();
    kda::g_acc.clear();
    kda::g_on = enable != 0;
    return KDA_OK;
}

int32_t kda_profile_read(kda_kernel_time_t* out, int32_t max_entries)
{
    std::lock_guard<std::mutex> lk(kda::g_mu);
    if (!kda::drain_locked()) return -1;
    const int32_t n = (int32_t)kda::g_acc.size();
    for (int32_t i = 0; i < n && i < max_entries && out; ++i) {
        std::memset(out[i].name, 0, sizeof(out[i].name));
        std::strncpy(out[i].name, kda::g_acc[i].name.c_str(), sizeof(out[i].name) - 1);
        out[i].launches = kda::g_acc[i].launches;
        out[i].total_ms = kda::g_acc[i].ms;
    }
    return n;
}

}  // extern "C"
