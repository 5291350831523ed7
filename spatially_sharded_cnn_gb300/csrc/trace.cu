// trace.cu -- per-kernel device timing.  While tracing is on, every launcher
// records a CUDA event on its stream before its first kernel and every launch
// records one after the kernel, so a kernel's device time is the interval from
// the event before it on the same stream to its own.  Launches into a stream
// that is being captured into a graph are not traced.  Host code only.
#include <string.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "common.cuh"

namespace hc {

std::atomic<int> g_trace_on{0};

namespace {

struct Rec {
    const char* name;
    cudaEvent_t a, b;
};

std::mutex g_mu;
std::vector<Rec> g_recs;
std::unordered_map<int, std::vector<cudaEvent_t>> g_pool;  // free events per device
std::unordered_map<cudaStream_t, cudaEvent_t> g_last;      // last event recorded on each stream
std::unordered_map<cudaEvent_t, int> g_dev_of;              // the device an event was created on

bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;  // not knowable (e.g. the legacy stream while another stream captures): skip
    }
    return cs != cudaStreamCaptureStatusNone;
}

// An event of the current device, recorded on st; nullptr if that failed.
cudaEvent_t record(cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaEvent_t e = nullptr;
    std::vector<cudaEvent_t>& pool = g_pool[dev];
    if (!pool.empty()) {
        e = pool.back();
        pool.pop_back();
    } else if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    } else {
        g_dev_of[e] = dev;
    }
    if (cudaEventRecord(e, st) != cudaSuccess) {
        cudaGetLastError();
        pool.push_back(e);
        return nullptr;
    }
    return e;
}

}  // namespace

void trace_begin(cudaStream_t st) {
    if (!g_trace_on.load(std::memory_order_relaxed) || capturing(st)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cudaEvent_t e = record(st)) g_last[st] = e;
}

void trace_launch(const char* name, cudaStream_t st) {
    if (!g_trace_on.load(std::memory_order_relaxed) || capturing(st)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t e = record(st);
    if (!e) return;
    auto it = g_last.find(st);
    if (it != g_last.end()) g_recs.push_back(Rec{name, it->second, e});
    g_last[st] = e;
}

}  // namespace hc

using namespace hc;

extern "C" {

hc_status hc_trace_enable(int on) {
    g_trace_on.store(on ? 1 : 0, std::memory_order_relaxed);
    return HC_OK;
}

hc_status hc_trace_collect(hc_trace_entry* out, int max_entries, int* n_entries) {
    if (!n_entries || max_entries < 0 || (max_entries > 0 && !out)) return HC_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    int n = 0;
    hc_status st = HC_OK;
    int cur = 0;
    cudaGetDevice(&cur);
    for (const Rec& r : g_recs) {
        float ms = 0.0f;
        const int dev = g_dev_of.count(r.b) ? g_dev_of[r.b] : cur;
        cudaSetDevice(dev);
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
            cudaGetLastError();
            st = HC_ERR_CUDA;
            continue;
        }
        int k = 0;
        while (k < n && strcmp(out[k].name, r.name) != 0) k++;
        if (k == n) {
            if (n == max_entries) continue;  // no room: the entry is dropped
            memset(&out[n], 0, sizeof(out[n]));
            strncpy(out[n].name, r.name, sizeof(out[n].name) - 1);
            n++;
        }
        out[k].launches += 1;
        out[k].total_ms += ms;
    }
    cudaSetDevice(cur);
    // every event goes back to its device's free list
    std::vector<cudaEvent_t> used;
    for (const Rec& r : g_recs) {
        used.push_back(r.a);
        used.push_back(r.b);
    }
    for (auto& kv : g_last) used.push_back(kv.second);
    std::sort(used.begin(), used.end());
    used.erase(std::unique(used.begin(), used.end()), used.end());
    for (cudaEvent_t e : used) g_pool[g_dev_of.count(e) ? g_dev_of[e] : cur].push_back(e);
    g_recs.clear();
    g_last.clear();
    *n_entries = n;
    return st;
}

}  // extern "C"
