// gt_stats.cu -- launch statistics of the library's kernels.
//
// Every launch site opens a LaunchScope with a fixed kernel name.  The table
// counts launches per name at all times (one mutex-guarded increment per
// launch).  In timing mode each launch is also bracketed by two CUDA events on
// its stream, taken from a pool that grows on demand and is kept for reuse; the
// read call synchronizes the recorded end events and sums the elapsed times.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "gt_attn.h"
#include "gt_stats.cuh"

namespace gt {
namespace {

struct Entry {
    std::string name;
    int64_t launches = 0;
};

struct Timed {
    int entry;
    cudaEvent_t start, end;
};

struct Table {
    std::mutex mu;
    bool timing = false;
    std::vector<Entry> entries;
    std::vector<Timed> timed;
    std::vector<cudaEvent_t> pool;
};

Table& table() {
    static Table* t = new Table();   // never destroyed: launches may race process exit
    return *t;
}

cudaEvent_t take_event(Table& t) {
    if (!t.pool.empty()) {
        cudaEvent_t e = t.pool.back();
        t.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

int stats_begin(const char* name, cudaStream_t s) {
    Table& t = table();
    std::lock_guard<std::mutex> lock(t.mu);
    int idx = -1;
    for (size_t i = 0; i < t.entries.size(); ++i)
        if (t.entries[i].name == name) { idx = (int)i; break; }
    if (idx < 0) {
        t.entries.push_back(Entry{name, 0});
        idx = (int)t.entries.size() - 1;
    }
    t.entries[idx].launches += 1;
    if (!t.timing) return -1;
    Timed rec{idx, take_event(t), take_event(t)};
    if (!rec.start || !rec.end || cudaEventRecord(rec.start, s) != cudaSuccess) {
        if (rec.start) t.pool.push_back(rec.start);
        if (rec.end) t.pool.push_back(rec.end);
        return -1;
    }
    t.timed.push_back(rec);
    return (int)t.timed.size() - 1;
}

void stats_end(int slot, cudaStream_t s) {
    if (slot < 0) return;
    Table& t = table();
    std::lock_guard<std::mutex> lock(t.mu);
    if (slot < (int)t.timed.size()) cudaEventRecord(t.timed[slot].end, s);
}

}  // namespace gt

extern "C" {

int gt_kernel_stats_reset(int32_t timing) {
    gt::Table& t = gt::table();
    std::lock_guard<std::mutex> lock(t.mu);
    for (const gt::Timed& r : t.timed) {
        // an event still pending completes before it can be reused
        if (cudaEventSynchronize(r.end) != cudaSuccess) return GT_ERR_CUDA;
        t.pool.push_back(r.start);
        t.pool.push_back(r.end);
    }
    t.timed.clear();
    t.entries.clear();
    t.timing = timing != 0;
    return GT_OK;
}

int gt_kernel_stats_read(gt_kernel_stat* out, int32_t cap, int32_t* count) {
    if (cap < 0 || (cap > 0 && !out) || !count) return GT_ERR_INVALID_ARG;
    gt::Table& t = gt::table();
    std::lock_guard<std::mutex> lock(t.mu);
    std::vector<double> ms(t.entries.size(), 0.0);
    for (const gt::Timed& r : t.timed) {
        if (cudaEventSynchronize(r.end) != cudaSuccess) return GT_ERR_CUDA;
        float e = 0.f;
        if (cudaEventElapsedTime(&e, r.start, r.end) != cudaSuccess) return GT_ERR_CUDA;
        ms[r.entry] += e;
    }
    *count = (int32_t)t.entries.size();
    for (int32_t i = 0; i < cap && i < (int32_t)t.entries.size(); ++i) {
        memset(out[i].name, 0, sizeof(out[i].name));
        strncpy(out[i].name, t.entries[i].name.c_str(), sizeof(out[i].name) - 1);
        out[i].launches = t.entries[i].launches;
        out[i].total_ms = t.timing ? ms[i] : -1.0;
    }
    return GT_OK;
}

}  // extern "C"
