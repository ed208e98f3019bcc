// rkv_prof.cu -- optional per-kernel timing with CUDA events recorded on the
// stream each kernel is launched on.  Off by default; when on, every launch the
// library makes is bracketed by two events, and rkv_profile_collect() reports the
// summed device time and the launch count per kernel name.
#include "rkv_internal.cuh"

#include <string.h>
#include <vector>

namespace rkv {

struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
};

static bool g_on = false;
static std::vector<ProfRec> g_recs;
static std::vector<cudaEvent_t> g_free;

static cudaEvent_t get_event()
{
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void prof_begin(const char *name, cudaStream_t s)
{
    if (!g_on) return;
    ProfRec r{name, get_event(), get_event()};
    if (!r.a || !r.b) return;
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
}

void prof_end(cudaStream_t s)
{
    if (!g_on || g_recs.empty()) return;
    cudaEventRecord(g_recs.back().b, s);
}

}  // namespace rkv

using namespace rkv;

extern "C" {

rkv_status rkv_profile_enable(int32_t on)
{
    for (auto &r : g_recs) {
        g_free.push_back(r.a);
        g_free.push_back(r.b);
    }
    g_recs.clear();
    g_on = on != 0;
    return RKV_OK;
}

int32_t rkv_profile_collect(char *names, int32_t name_len, float *total_ms, int32_t *launches,
                            int32_t max_entries)
{
    if (!names || !total_ms || !launches || max_entries <= 0 || name_len < 2) return -1;
    int n = 0;
    for (auto &r : g_recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
        int j = 0;
        for (; j < n; ++j)
            if (strncmp(names + (size_t)j * name_len, r.name, name_len - 1) == 0) break;
        if (j == n) {
            if (n == max_entries) continue;
            strncpy(names + (size_t)j * name_len, r.name, name_len - 1);
            names[(size_t)j * name_len + name_len - 1] = 0;
            total_ms[j] = 0.0f;
            launches[j] = 0;
            ++n;
        }
        total_ms[j] += ms;
        launches[j] += 1;
    }
    return n;
}

}  // extern "C"
