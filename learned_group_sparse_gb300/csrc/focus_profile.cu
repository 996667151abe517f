// Opt-in per-kernel timing: when enabled on a host thread, every kernel the
// library launches from that thread is bracketed by two CUDA events on its
// stream; focus_profile_read() sums the elapsed times per kernel name.
#include <cuda_runtime.h>
#include <string.h>

#include <string>
#include <vector>

#include "focus_internal.h"

namespace focus {

namespace {

struct Mark {
    const char *name;
    cudaEvent_t start, stop;
};

struct Profiler {
    bool enabled = false;
    std::vector<Mark> marks;
    std::vector<cudaEvent_t> pool;
    cudaEvent_t pending = nullptr;
    const char *pending_name = nullptr;

    cudaEvent_t take()
    {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};

thread_local Profiler g_prof;
thread_local long long *g_trace[3] = {nullptr, nullptr, nullptr};
thread_local long long *g_gtrace[2] = {nullptr, nullptr};
thread_local int g_gtrace_ctas = 0;

}  // namespace

long long *trace_buffer(int mode) { return (mode >= 0 && mode < 3) ? g_trace[mode] : nullptr; }

void gated_trace_buffer(int side, long long **buf, int *ctas)
{
    *buf = (side == 0 || side == 1) ? g_gtrace[side] : nullptr;
    *ctas = *buf ? g_gtrace_ctas : 0;
}

void prof_begin(const char *name, cudaStream_t s)
{
    if (!g_prof.enabled) return;
    g_prof.pending = g_prof.take();
    g_prof.pending_name = name;
    cudaEventRecord(g_prof.pending, s);
}

void prof_end(cudaStream_t s)
{
    if (!g_prof.enabled || !g_prof.pending) return;
    cudaEvent_t stop = g_prof.take();
    cudaEventRecord(stop, s);
    g_prof.marks.push_back({g_prof.pending_name, g_prof.pending, stop});
    g_prof.pending = nullptr;
}

}  // namespace focus

using namespace focus;

extern "C" {

void focus_profile_enable(int enable) { g_prof.enabled = enable != 0; }

void focus_trace_attention(long long *group_buf, long long *window_buf, long long *dense_buf)
{
    g_trace[0] = group_buf;
    g_trace[1] = window_buf;
    g_trace[2] = dense_buf;
}

void focus_trace_gated(long long *query_buf, long long *key_buf, int max_ctas)
{
    g_gtrace[0] = max_ctas > 0 ? query_buf : nullptr;
    g_gtrace[1] = max_ctas > 0 ? key_buf : nullptr;
    g_gtrace_ctas = max_ctas > 0 ? max_ctas : 0;
}

int focus_profile_read(char *names, int name_stride, double *total_ms, int *launches,
                       int max_entries)
{
    std::vector<std::string> keys;
    std::vector<double> ms;
    std::vector<int> cnt;
    for (const Mark &m : g_prof.marks) {
        float t = 0.f;
        if (cudaEventSynchronize(m.stop) != cudaSuccess) return -1;
        if (cudaEventElapsedTime(&t, m.start, m.stop) != cudaSuccess) return -1;
        size_t k = 0;
        while (k < keys.size() && keys[k] != m.name) ++k;
        if (k == keys.size()) {
            keys.emplace_back(m.name);
            ms.push_back(0.0);
            cnt.push_back(0);
        }
        ms[k] += t;
        cnt[k] += 1;
        g_prof.pool.push_back(m.start);
        g_prof.pool.push_back(m.stop);
    }
    g_prof.marks.clear();
    const int n = (int)keys.size() < max_entries ? (int)keys.size() : max_entries;
    for (int i = 0; i < n; ++i) {
        if (names && name_stride > 0) {
            strncpy(names + (size_t)i * name_stride, keys[i].c_str(), name_stride - 1);
            names[(size_t)i * name_stride + name_stride - 1] = 0;
        }
        if (total_ms) total_ms[i] = ms[i];
        if (launches) launches[i] = cnt[i];
    }
    return n;
}

}  // extern "C"
