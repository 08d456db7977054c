// Launch counting and optional per-launch CUDA-event timing.
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace muon {
namespace {

struct Record {
    int kind;
    cudaEvent_t start, stop;
};

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;
Record g_open{-1, nullptr, nullptr};
// launches the calling thread made since its capture_begin; -1 outside a capture
thread_local int64_t t_captured = -1;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void drop_records_locked() {
    for (const Record& r : g_records) {
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
    }
    g_records.clear();
}

// MUON_DEBUG, read once per process
bool debug_mode() {
    static const bool on = [] {
        const char* v = getenv("MUON_DEBUG");
        return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
    }();
    return on;
}

// Debug mode: waits for the launch and reports it by name if it failed.
void debug_check(int kind, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaPeekAtLastError();
    if (e != cudaSuccess) fprintf(stderr, "muon: kernel %s failed: %s\n", muon_kernel_name(kind), cudaGetErrorString(e));
}

}  // namespace

void launch_begin(int kind, cudaStream_t st) {
    if (t_captured >= 0) {
        ++t_captured;
        return;
    }
    nvtxRangePushA(muon_kernel_name(kind));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    g_open.kind = kind;
    g_open.start = take_event();
    g_open.stop = take_event();
    if (g_open.start) cudaEventRecord(g_open.start, st);
}

void launch_end(int kind, cudaStream_t st) {
    if (t_captured >= 0) return;
    nvtxRangePop();
    if (debug_mode()) debug_check(kind, st);
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_open.kind != kind || !g_open.start || !g_open.stop) return;
    cudaEventRecord(g_open.stop, st);
    g_records.push_back(g_open);
    g_open = Record{-1, nullptr, nullptr};
}

void capture_begin() { t_captured = 0; }

int64_t capture_end() {
    const int64_t n = t_captured < 0 ? 0 : t_captured;
    t_captured = -1;
    return n;
}

void count_replay(int64_t launches) { g_launches.fetch_add(launches, std::memory_order_relaxed); }

}  // namespace muon

using namespace muon;

extern "C" {

int64_t muon_launch_count(void) { return g_launches.load(); }

muon_status_t muon_set_timing(int32_t enable) {
    std::lock_guard<std::mutex> lock(g_mu);
    drop_records_locked();
    g_enabled.store(enable ? 1 : 0);
    return MUON_OK;
}

muon_status_t muon_timing_read(double* ms, int64_t* launches, int32_t nkinds) {
    if (nkinds < 0 || (nkinds > 0 && (!ms || !launches))) return MUON_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < nkinds; ++i) {
        ms[i] = 0.0;
        launches[i] = 0;
    }
    muon_status_t status = MUON_OK;
    for (const Record& r : g_records) {
        if (cudaEventSynchronize(r.stop) != cudaSuccess) {
            status = MUON_ERR_CUDA;
            continue;
        }
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) {
            status = MUON_ERR_CUDA;
            continue;
        }
        if (r.kind >= 0 && r.kind < nkinds) {
            ms[r.kind] += t;
            launches[r.kind] += 1;
        }
    }
    drop_records_locked();
    return status;
}

const char* muon_kernel_name(int32_t kind) {
    switch (kind) {
        case MUON_KERNEL_MOMENTUM_NORM: return "momentum_norm";
        case MUON_KERNEL_NORM_FINALIZE: return "norm_finalize";
        case MUON_KERNEL_X0_RESCALE: return "x0_rescale";
        case MUON_KERNEL_NS_SYRK: return "ns_syrk";
        case MUON_KERNEL_NS_POLY: return "ns_poly";
        case MUON_KERNEL_NS_UPDATE: return "ns_update";
        case MUON_KERNEL_FINAL_UPDATE: return "final_update";
        case MUON_KERNEL_ADAMW: return "adamw";
        case MUON_KERNEL_GRAD_GUARD: return "grad_guard";
        case MUON_KERNEL_DESC_UPLOAD: return "desc_upload";
        case MUON_KERNEL_STATS: return "stats";
    }
    return "unknown";
}

}  // extern "C"
