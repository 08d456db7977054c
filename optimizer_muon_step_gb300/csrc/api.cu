// C ABI of the Muon / AdamW step: validation, the execution plan, the
// workspace layout and the launch sequence.  Kernels live in
// elementwise.cu and ns_gemm.cu.
//
// Workspace layout of one chunk of n matrices (n * 8192 record bytes plus
// the X / Gram buffers of muon_workspace_bytes_per_matrix):
//   [0, 256)                 WsHeader: status word, gradient-guard results
//   [256, ...)               MatDesc[n]
//   [.., +n*4096)            norm partial sums, 1024 floats per matrix
//   [.., +n*2048)            statistics pass sums, 512 floats per matrix
//   [n*8192, ...)            per shape group of c matrices:
//                              X0[c], X1[c]  (each R(2 m' L(n')) bytes)
//                              A[c],  B[c]   (each R(2 m' L(m')) bytes)
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <numeric>
#include <vector>

#include "internal.h"

using namespace muon;

namespace {

constexpr int32_t kVersion = 300;  // 0.3.0

inline int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

struct DeviceInfo {
    int ok = -1;  // -1 unknown, 0 unsupported, 1 sm_103
    int num_sms = 0;
};

muon_status_t device_info(int* num_sms) {
    static std::mutex mu;
    static DeviceInfo info[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
    if (dev < 0 || dev >= 64) return MUON_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = info[dev];
    if (d.ok < 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MUON_ERR_CUDA;
        d.ok = (major == 10 && minor == 3) ? 1 : 0;
        d.num_sms = sms;
    }
    if (d.ok != 1) return MUON_ERR_NO_DEVICE;
    *num_sms = d.num_sms;
    return MUON_OK;
}

// ---------------------------------------------------------------------------
// Whose memory the caller's buffers are.  Every buffer the kernels read or
// write must be memory the current device owns: a device allocation made on
// it, or managed memory.  Host memory (pinned or pageable), another device's
// allocations and unknown addresses are refused with MUON_ERR_INVALID_ARG
// before anything is enqueued, so such a call ends in an error code rather
// than in a memory fault on the device.  Each driver query also looks up the
// bounds of the allocation holding the pointer and remembers them, so the
// views of one large buffer cost a single query.
// ---------------------------------------------------------------------------
typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

AddressRangeFn address_range_fn() {
    static AddressRangeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddressRangeFn>(ptr);
    });
    return fn;
}

class DeviceMemoryCheck {
  public:
    explicit DeviceMemoryCheck(int device) : dev_(device) {}

    // Whether the buffer starting at p (bytes long) is the current device's.
    bool owns(const void* p, size_t bytes) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        auto it = known_.upper_bound(lo);
        if (it != known_.begin()) {
            --it;
            if (lo >= it->first && lo + bytes <= it->second) return true;
        }
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();  // a refused query must not look like a failed launch later
            return false;
        }
        const bool mine = (a.type == cudaMemoryTypeDevice && a.device == dev_) || a.type == cudaMemoryTypeManaged;
        if (!mine) return false;
        CUdeviceptr base = 0;
        size_t size = 0;
        const AddressRangeFn range = address_range_fn();
        if (range && range(&base, &size, static_cast<CUdeviceptr>(lo)) == CUDA_SUCCESS && size > 0)
            known_[static_cast<uintptr_t>(base)] = static_cast<uintptr_t>(base) + size;
        return true;
    }

  private:
    int dev_;
    std::map<uintptr_t, uintptr_t> known_;  // verified allocations, start -> end
};

// Whether `st` is being captured into a graph.  A capture records launches
// only, so the memory checks are left out there (muon_step_graph_create
// checks before it captures); a stream whose state cannot be read counts as
// capturing.
bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

int64_t bytes_per_matrix(int64_t mp, int64_t np) {
    const int64_t x = round_up(2 * mp * round_up(np, 8), 256);
    const int64_t g = round_up(2 * mp * round_up(mp, 8), 256);
    return 2 * x + 2 * g + static_cast<int64_t>(kRecordBytes);
}

bool finite(float x) { return isfinite(x) != 0; }

muon_status_t check_hparams(const muon_hparams_t* hp) {
    if (!hp) return MUON_ERR_INVALID_ARG;
    if (!finite(hp->lr) || !finite(hp->weight_decay) || !finite(hp->momentum) || !finite(hp->ns_a) ||
        !finite(hp->ns_b) || !finite(hp->ns_c) || !finite(hp->norm_eps) || !finite(hp->rms_scale))
        return MUON_ERR_INVALID_ARG;
    if (hp->momentum < 0.f || hp->momentum > 1.f || hp->norm_eps < 0.f) return MUON_ERR_INVALID_ARG;
    if (hp->ns_steps < 0 || hp->ns_steps > 100) return MUON_ERR_INVALID_ARG;
    if (hp->nesterov != 0 && hp->nesterov != 1) return MUON_ERR_INVALID_ARG;
    if (hp->scale_mode != 0 && hp->scale_mode != 1) return MUON_ERR_INVALID_ARG;
    if (hp->skip_nonfinite != 0 && hp->skip_nonfinite != 1) return MUON_ERR_INVALID_ARG;
    if (!finite(hp->max_grad_norm) || hp->reserved0 != 0) return MUON_ERR_INVALID_ARG;
    if (hp->ns_coeffs)
        for (int i = 0; i < 3 * hp->ns_steps; ++i)
            if (!finite(hp->ns_coeffs[i])) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

// Per-step NS coefficients, 3 * steps floats.
std::vector<float> coeff_table(const muon_hparams_t* hp) {
    std::vector<float> t(3 * static_cast<size_t>(hp->ns_steps));
    for (int s = 0; s < hp->ns_steps; ++s) {
        t[3 * s] = hp->ns_coeffs ? hp->ns_coeffs[3 * s] : hp->ns_a;
        t[3 * s + 1] = hp->ns_coeffs ? hp->ns_coeffs[3 * s + 1] : hp->ns_b;
        t[3 * s + 2] = hp->ns_coeffs ? hp->ns_coeffs[3 * s + 2] : hp->ns_c;
    }
    return t;
}

// The update's scale factor (fp64, rounded to fp32): mode 0 matches AdamW's
// update RMS, rms_scale * sqrt(max(rows, cols)); mode 1 is the muP-style
// max(1, sqrt(d_out / d_in)) with (d_out, d_in) = (rows, cols).
float update_scale(const muon_hparams_t* hp, int64_t rows, int64_t cols) {
    if (hp->scale_mode == 1) {
        const double r = sqrt(static_cast<double>(rows) / static_cast<double>(cols));
        return static_cast<float>(r > 1.0 ? r : 1.0);
    }
    return static_cast<float>(static_cast<double>(hp->rms_scale) * sqrt(static_cast<double>(std::max(rows, cols))));
}

muon_status_t check_shapes(const muon_matrix_t* mats, int64_t count) {
    if (count < 0) return MUON_ERR_INVALID_ARG;
    if (count > 0 && !mats) return MUON_ERR_INVALID_ARG;
    if (count > (int64_t(1) << 30)) return MUON_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i) {
        const muon_matrix_t& m = mats[i];
        // m' and n' are used as int32 extents by the GEMM scheduler
        if (m.rows <= 0 || m.cols <= 0 || m.rows > (int64_t(1) << 30) || m.cols > (int64_t(1) << 30))
            return MUON_ERR_INVALID_ARG;
        if (m.rows * m.cols > (int64_t(1) << 40)) return MUON_ERR_INVALID_ARG;
    }
    return MUON_OK;
}

muon_status_t check_pointers(const muon_matrix_t* mats, int64_t count) {
    for (int64_t i = 0; i < count; ++i) {
        const muon_matrix_t& m = mats[i];
        if (!m.W || !m.G || !m.M || m.reserved != 0) return MUON_ERR_INVALID_ARG;
        if (m.g_dtype != MUON_F32 && m.g_dtype != MUON_BF16 && m.g_dtype != MUON_F16)
            return MUON_ERR_UNSUPPORTED_DTYPE;
        const uintptr_t g_align = m.g_dtype == MUON_F32 ? 4 : 2;
        if ((reinterpret_cast<uintptr_t>(m.W) & 3u) || (reinterpret_cast<uintptr_t>(m.M) & 3u) ||
            (reinterpret_cast<uintptr_t>(m.G) & (g_align - 1)))
            return MUON_ERR_MISALIGNED;
    }
    return MUON_OK;
}

// Every matrix's W, G and M, the workspace and the statistics array (when
// given) on the current device.
muon_status_t check_step_memory(const muon_matrix_t* mats, int64_t count, const void* workspace, size_t ws_bytes,
                                const void* stats) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
    DeviceMemoryCheck mem(dev);
    if (!mem.owns(workspace, ws_bytes)) return MUON_ERR_INVALID_ARG;
    if (stats && !mem.owns(stats, static_cast<size_t>(count) * sizeof(muon_matrix_stats_t)))
        return MUON_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i) {
        const muon_matrix_t& m = mats[i];
        const size_t n = static_cast<size_t>(m.rows * m.cols);
        const size_t g_bytes = m.g_dtype == MUON_F32 ? 4 : 2;
        if (!mem.owns(m.W, 4 * n) || !mem.owns(m.G, g_bytes * n) || !mem.owns(m.M, 4 * n))
            return MUON_ERR_INVALID_ARG;
    }
    return MUON_OK;
}

struct PlanRow {
    int32_t idx, transposed, group, slot, chunk;
    int64_t mp, np;
};

// Stable order by (m', n'); greedy chunks under ws_bytes.
muon_status_t build_plan(const muon_matrix_t* mats, int64_t count, int64_t ws_bytes, std::vector<PlanRow>& out) {
    std::vector<int32_t> order(static_cast<size_t>(count));
    std::iota(order.begin(), order.end(), 0);
    auto key = [&](int32_t i) {
        const int64_t r = mats[i].rows, c = mats[i].cols;
        return std::make_pair(std::min(r, c), std::max(r, c));
    };
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return key(a) < key(b); });
    out.clear();
    out.reserve(order.size());
    int32_t group = -1, chunk = 0, slot = 0;
    int64_t used = 0, pm = -1, pn = -1;
    for (size_t k = 0; k < order.size(); ++k) {
        const int32_t i = order[k];
        const auto mn = key(i);
        const int64_t need = bytes_per_matrix(mn.first, mn.second);
        if (need > ws_bytes) return MUON_ERR_WORKSPACE_TOO_SMALL;
        const bool new_group = mn.first != pm || mn.second != pn;
        if (new_group) ++group;
        if (k > 0 && used + need > ws_bytes) {
            ++chunk;
            used = 0;
            slot = 0;
        } else if (new_group) {
            slot = 0;
        }
        PlanRow row;
        row.idx = i;
        row.transposed = mats[i].rows > mats[i].cols ? 1 : 0;
        row.group = group;
        row.slot = slot++;
        row.chunk = chunk;
        row.mp = mn.first;
        row.np = mn.second;
        out.push_back(row);
        used += need;
        pm = mn.first;
        pn = mn.second;
    }
    return MUON_OK;
}

muon_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA; }

// Lays out one chunk's shape groups in the workspace.
struct ChunkLayout {
    std::vector<NsGroup> groups;
    std::vector<int64_t> first;  // per group: its first plan row, counted from the chunk start
    std::vector<int64_t> x0_of;  // per plan row in chunk: X0 address offset
    std::vector<int64_t> x1_of;
};

void layout_groups(const std::vector<PlanRow>& plan, size_t b, size_t e, uint8_t* base, ChunkLayout& L) {
    L.groups.clear();
    L.first.clear();
    L.x0_of.assign(e - b, 0);
    L.x1_of.assign(e - b, 0);
    uint8_t* cursor = base + (e - b) * kRecordBytes;
    size_t k = b;
    while (k < e) {
        size_t j = k;
        while (j < e && plan[j].mp == plan[k].mp && plan[j].np == plan[k].np) ++j;
        const int64_t c = static_cast<int64_t>(j - k);
        NsGroup g;
        g.mp = plan[k].mp;
        g.np = plan[k].np;
        g.ldx = round_up(g.np, 8);
        g.lda = round_up(g.mp, 8);
        g.x_stride = round_up(2 * g.mp * g.ldx, 256);
        g.g_stride = round_up(2 * g.mp * g.lda, 256);
        g.count = c;
        g.scale = nullptr;
        g.scale_stride = 0;
        g.X[0] = reinterpret_cast<uint16_t*>(cursor);
        g.X[1] = reinterpret_cast<uint16_t*>(cursor + c * g.x_stride);
        g.A = reinterpret_cast<uint16_t*>(cursor + 2 * c * g.x_stride);
        g.B = reinterpret_cast<uint16_t*>(cursor + 2 * c * g.x_stride + c * g.g_stride);
        for (size_t q = k; q < j; ++q) {
            L.x0_of[q - b] = reinterpret_cast<uint8_t*>(g.X[0]) - base + static_cast<int64_t>(q - k) * g.x_stride;
            L.x1_of[q - b] = reinterpret_cast<uint8_t*>(g.X[1]) - base + static_cast<int64_t>(q - k) * g.x_stride;
        }
        cursor += 2 * c * g.x_stride + 2 * c * g.g_stride;
        L.groups.push_back(g);
        L.first.push_back(static_cast<int64_t>(k - b));
        k = j;
    }
}

}  // namespace

extern "C" {

int32_t muon_version(void) { return kVersion; }

const char* muon_status_string(muon_status_t s) {
    switch (s) {
        case MUON_OK: return "ok";
        case MUON_ERR_INVALID_ARG: return "invalid argument";
        case MUON_ERR_UNSUPPORTED_DTYPE: return "unsupported gradient dtype";
        case MUON_ERR_MISALIGNED: return "misaligned pointer";
        case MUON_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MUON_ERR_CUDA: return "CUDA runtime error";
        case MUON_ERR_TIMEOUT: return "kernel timed out on a bounded wait";
        case MUON_ERR_NO_DEVICE: return "no sm_103 device is current";
        case MUON_STEP_SKIPPED: return "step skipped by the non-finite gradient guard";
    }
    return "unknown status";
}

size_t muon_workspace_bytes_per_matrix(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>(bytes_per_matrix(std::min(rows, cols), std::max(rows, cols)));
}

muon_status_t muon_workspace_size(const muon_matrix_t* mats, int64_t count, size_t budget_bytes,
                                  size_t* out_bytes) {
    if (!out_bytes) return MUON_ERR_INVALID_ARG;
    muon_status_t s = check_shapes(mats, count);
    if (s != MUON_OK) return s;
    int64_t total = 0, largest = 0;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t b = static_cast<int64_t>(muon_workspace_bytes_per_matrix(mats[i].rows, mats[i].cols));
        total += b;
        largest = std::max(largest, b);
    }
    const int64_t budget = static_cast<int64_t>(budget_bytes);
    *out_bytes = static_cast<size_t>(total <= budget ? total : std::max(budget, largest));
    return MUON_OK;
}

muon_status_t muon_plan(const muon_matrix_t* mats, int64_t count, size_t ws_bytes, muon_plan_entry_t* out) {
    muon_status_t s = check_shapes(mats, count);
    if (s != MUON_OK) return s;
    if (count > 0 && !out) return MUON_ERR_INVALID_ARG;
    std::vector<PlanRow> plan;
    s = build_plan(mats, count, static_cast<int64_t>(ws_bytes), plan);
    if (s != MUON_OK) return s;
    for (size_t k = 0; k < plan.size(); ++k) {
        out[k].mat_idx = plan[k].idx;
        out[k].transposed = plan[k].transposed;
        out[k].group_id = plan[k].group;
        out[k].slot = plan[k].slot;
        out[k].chunk_id = plan[k].chunk;
        out[k].reserved = 0;
        out[k].mp = plan[k].mp;
        out[k].np = plan[k].np;
    }
    return MUON_OK;
}

}  // extern "C"

namespace {

// The step, with per-matrix statistics when `stats` is non-null.
muon_status_t step_impl(const muon_matrix_t* mats, int64_t count, const muon_hparams_t* hp, void* workspace,
                        size_t ws_bytes, muon_matrix_stats_t* stats, void* stream) {
    NvtxScope range("muon_step");
    muon_status_t s = check_hparams(hp);
    if (s != MUON_OK) return s;
    s = check_shapes(mats, count);
    if (s != MUON_OK) return s;
    if (count == 0) return MUON_OK;
    s = check_pointers(mats, count);
    if (s != MUON_OK) return s;
    if (!workspace) return MUON_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
    int num_sms = 0;
    s = device_info(&num_sms);
    if (s != MUON_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!capturing(st)) {
        s = check_step_memory(mats, count, workspace, ws_bytes, stats);
        if (s != MUON_OK) return s;
    }

    std::vector<PlanRow> plan;
    s = build_plan(mats, count, static_cast<int64_t>(ws_bytes), plan);
    if (s != MUON_OK) return s;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    WsHeader* header = reinterpret_cast<WsHeader*>(ws);
    bool header_cleared = false;  // the call's first record upload clears the header

    const bool clip_on = hp->max_grad_norm > 0.f;
    const bool guard_on = clip_on || hp->skip_nonfinite;
    const MomentumScalars ms{hp->momentum, 1.0f - hp->momentum, hp->nesterov, clip_on ? 1 : 0,
                             guard_on ? header : nullptr};
    const UpdateScalars us{hp->lr, hp->weight_decay, guard_on ? header : nullptr};
    const std::vector<float> coeffs = coeff_table(hp);
    ChunkLayout L;
    std::vector<MatDesc> descs;
    MatDesc* d_descs = reinterpret_cast<MatDesc*>(ws + kHeaderBytes);
    int max_tiles = 1;       // flat tiles, every matrix (gradient guard)
    int max_wide_tiles = 0;  // flat tiles of the wide matrices (momentum pass)
    int max_units = 0;       // tall-pass units (momentum pass)
    int64_t max_final_units = 0;  // tall units of the final update
    int tall_units[3] = {0, 0, 0};  // the same, over tall matrices per gradient type (muon_dtype_t)
    int wide_tiles[3] = {0, 0, 0};  // flat tiles of the wide matrices per gradient type
    float* o_partials = nullptr;  // statistics pass: kStatsTiles sums per matrix after the norm partials

    // Fills `descs` and the layout for plan rows [b, e) and uploads them (by
    // kernel parameters: no host buffer outlives the call, so the sequence
    // can be captured into a graph).
    auto prepare_chunk = [&](size_t b, size_t e) -> muon_status_t {
        const int n = static_cast<int>(e - b);
        layout_groups(plan, b, e, ws, L);
        float* d_partials = reinterpret_cast<float*>(
            ws + kHeaderBytes + round_up(static_cast<int64_t>(n) * static_cast<int64_t>(sizeof(MatDesc)), 256));
        o_partials = d_partials + static_cast<int64_t>(n) * kMaxNormTiles;
        descs.assign(n, MatDesc{});
        max_tiles = 1;
        max_wide_tiles = max_units = 0;
        max_final_units = 0;
        tall_units[0] = tall_units[1] = tall_units[2] = 0;
        wide_tiles[0] = wide_tiles[1] = wide_tiles[2] = 0;
        for (int k = 0; k < n; ++k) {
            const PlanRow& row = plan[b + k];
            const muon_matrix_t& m = mats[row.idx];
            MatDesc& d = descs[k];
            d.W = m.W;
            d.G = m.G;
            d.M = m.M;
            d.X0 = reinterpret_cast<uint16_t*>(ws + L.x0_of[k]);
            d.O = reinterpret_cast<const uint16_t*>(ws + ((hp->ns_steps & 1) ? L.x1_of[k] : L.x0_of[k]));
            d.partials = d_partials + static_cast<int64_t>(k) * kMaxNormTiles;
            d.rows = m.rows;
            d.cols = m.cols;
            d.ldx = round_up(row.np, 8);
            const int64_t nel = m.rows * m.cols;
            int64_t tl = 8192;
            int64_t nt = (nel + tl - 1) / tl;
            if (nt > kMaxNormTiles) {
                tl = round_up((nel + kMaxNormTiles - 1) / kMaxNormTiles, 8);
                nt = (nel + tl - 1) / tl;
            }
            d.tile_len = tl;
            d.ntiles = static_cast<int32_t>(nt);
            d.g_kind = m.g_dtype;
            d.transposed = row.transposed;
            d.vec = ((reinterpret_cast<uintptr_t>(m.W) | reinterpret_cast<uintptr_t>(m.G) |
                      reinterpret_cast<uintptr_t>(m.M)) & 15u) == 0 ? 1 : 0;
            d.scale = 0.f;
            d.update_scale = update_scale(hp, m.rows, m.cols);
            d.stats = stats ? stats + row.idx : nullptr;
            if (d.transposed) {
                // units of tall_kc x tall_kr 64x64 tiles, at most kMaxNormTiles
                const int64_t rt = (m.rows + 63) / 64, ct = (m.cols + 63) / 64;
                const int64_t kc = (ct + kMaxNormTiles - 1) / kMaxNormTiles;
                const int64_t cu = (ct + kc - 1) / kc;
                const int64_t kr = (rt + kMaxNormTiles / cu - 1) / (kMaxNormTiles / cu);
                d.tall_kc = static_cast<int32_t>(kc);
                d.tall_kr = static_cast<int32_t>(kr);
                d.nparts = static_cast<int32_t>(cu * ((rt + kr - 1) / kr));
                max_units = std::max(max_units, d.nparts);
                max_final_units = std::max(max_final_units, final_update_tall_units(m.rows, m.cols));
                tall_units[d.g_kind] = std::max(tall_units[d.g_kind], d.nparts);
            } else {
                d.nparts = d.ntiles;
                max_wide_tiles = std::max(max_wide_tiles, d.ntiles);
                wide_tiles[d.g_kind] = std::max(wide_tiles[d.g_kind], d.ntiles);
            }
            max_tiles = std::max(max_tiles, d.ntiles);
        }
        // the first NS step applies each matrix's ns_scale, read from its record
        for (size_t gi = 0; gi < L.groups.size(); ++gi) {
            L.groups[gi].scale = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(d_descs + L.first[gi]) +
                                                                offsetof(MatDesc, ns_scale));
            L.groups[gi].scale_stride = static_cast<int64_t>(sizeof(MatDesc) / sizeof(float));
        }
        WsHeader* clear = header_cleared ? nullptr : header;
        header_cleared = true;
        return from_cuda(launch_desc_upload(d_descs, descs.data(), n, clear, st));
    };

    // chunk boundaries
    std::vector<std::pair<size_t, size_t>> chunks;
    for (size_t b = 0; b < plan.size();) {
        size_t e = b;
        while (e < plan.size() && plan[e].chunk == plan[b].chunk) ++e;
        chunks.emplace_back(b, e);
        b = e;
    }

    // Gradient guard over every matrix of the call, before any state changes.
    if (guard_on) {
        for (const auto& c : chunks) {
            s = prepare_chunk(c.first, c.second);
            if (s != MUON_OK) return s;
            const int n = static_cast<int>(c.second - c.first);
            s = from_cuda(launch_grad_stats(d_descs, n, max_tiles, header, st));
            if (s != MUON_OK) return s;
            s = from_cuda(launch_grad_stats_reduce(d_descs, n, header, st));
            if (s != MUON_OK) return s;
        }
        s = from_cuda(launch_grad_decide(header, hp->max_grad_norm, hp->skip_nonfinite, st));
        if (s != MUON_OK) return s;
    }

    for (size_t ci = 0; ci < chunks.size(); ++ci) {
        NvtxScope chunk_range("muon_step chunk");
        const size_t b = chunks[ci].first, e = chunks[ci].second;
        const int n = static_cast<int>(e - b);
        if (!(guard_on && chunks.size() == 1)) {  // a single chunk is still in place from the guard
            s = prepare_chunk(b, e);
            if (s != MUON_OK) return s;
        }
        s = from_cuda(launch_momentum_norm(d_descs, n, wide_tiles, tall_units, ms, st));
        if (s != MUON_OK) return s;
        // with no NS step X0 is the result, so it is normalised in place
        s = from_cuda(launch_norm_finalize(d_descs, n, hp->norm_eps, hp->ns_steps == 0 ? 1 : 0, st));
        if (s != MUON_OK) return s;
        s = from_cuda(ns_run(L.groups.data(), static_cast<int>(L.groups.size()), hp->ns_steps, coeffs.data(),
                             &header->status, num_sms, st));
        if (s != MUON_OK) return s;
        s = from_cuda(launch_final_update(d_descs, n, max_wide_tiles, max_final_units, us, st));
        if (s != MUON_OK) return s;
        if (stats) {
            s = from_cuda(launch_step_stats(d_descs, n, o_partials, guard_on ? header : nullptr, st));
            if (s != MUON_OK) return s;
        }
    }
    return MUON_OK;
}

}  // namespace

extern "C" {

muon_status_t muon_step_batched(const muon_matrix_t* mats, int64_t count, const muon_hparams_t* hp,
                                void* workspace, size_t ws_bytes, void* stream) {
    return step_impl(mats, count, hp, workspace, ws_bytes, nullptr, stream);
}

muon_status_t muon_step_batched_stats(const muon_matrix_t* mats, int64_t count, const muon_hparams_t* hp,
                                      void* workspace, size_t ws_bytes, muon_matrix_stats_t* stats, void* stream) {
    if (!stats) return MUON_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(stats) & 7u) return MUON_ERR_MISALIGNED;
    return step_impl(mats, count, hp, workspace, ws_bytes, stats, stream);
}

}  // extern "C"

// A captured step: the instantiated graph and what one replay launches.
struct muon_graph_s {
    cudaGraphExec_t exec;  // null for a step of no matrices
    int64_t launches;      // this library's kernels in one replay
};

extern "C" {

muon_status_t muon_step_graph_create(const muon_matrix_t* mats, int64_t count, const muon_hparams_t* hp,
                                     void* workspace, size_t ws_bytes, muon_graph_t* out) {
    NvtxScope range("muon_step_graph_create");
    if (!out) return MUON_ERR_INVALID_ARG;
    *out = nullptr;
    // the host-side checks of the step, so that a bad call captures nothing
    muon_status_t s = check_hparams(hp);
    if (s != MUON_OK) return s;
    s = check_shapes(mats, count);
    if (s != MUON_OK) return s;
    std::unique_ptr<muon_graph_s> g(new (std::nothrow) muon_graph_s{nullptr, 0});
    if (!g) return MUON_ERR_INVALID_ARG;
    if (count > 0) {
        s = check_pointers(mats, count);
        if (s != MUON_OK) return s;
        if (!workspace) return MUON_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
        int num_sms = 0;
        s = device_info(&num_sms);
        if (s != MUON_OK) return s;
        s = check_step_memory(mats, count, workspace, ws_bytes, nullptr);
        if (s != MUON_OK) return s;
        // kernel attributes are set outside the capture
        if (ns_prepare_device() != cudaSuccess) return MUON_ERR_CUDA;
        cudaStream_t cs = nullptr;
        if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MUON_ERR_CUDA;
        cudaGraph_t graph = nullptr;
        s = from_cuda(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
        if (s == MUON_OK) {
            capture_begin();
            s = muon_step_batched(mats, count, hp, workspace, ws_bytes, cs);
            g->launches = capture_end();
            const cudaError_t e = cudaStreamEndCapture(cs, &graph);
            if (s == MUON_OK && e != cudaSuccess) s = MUON_ERR_CUDA;
        }
        if (s == MUON_OK && cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) {
            g->exec = nullptr;
            s = MUON_ERR_CUDA;
        }
        if (graph) cudaGraphDestroy(graph);
        cudaStreamDestroy(cs);
        if (s != MUON_OK) return s;
    }
    *out = g.release();
    return MUON_OK;
}

muon_status_t muon_step_graph_launch(muon_graph_t graph, void* stream) {
    if (!graph) return MUON_ERR_INVALID_ARG;
    if (!graph->exec) return MUON_OK;
    if (cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess) return MUON_ERR_CUDA;
    count_replay(graph->launches);
    return MUON_OK;
}

muon_status_t muon_step_graph_destroy(muon_graph_t graph) {
    if (!graph) return MUON_OK;
    // an executable graph still in flight is freed when it completes
    const bool ok = !graph->exec || cudaGraphExecDestroy(graph->exec) == cudaSuccess;
    delete graph;
    return ok ? MUON_OK : MUON_ERR_CUDA;
}

muon_status_t muon_newton_schulz(const uint16_t* X_in, uint16_t* X_out, int64_t count, int64_t mp, int64_t np,
                                 int32_t ns_steps, const float* coeff_in, int32_t ncoeff_sets, void* workspace,
                                 size_t ws_bytes, void* stream) {
    NvtxScope range("muon_newton_schulz");
    if (count < 0 || mp <= 0 || np <= 0 || mp > np || ns_steps < 0 || ns_steps > 100) return MUON_ERR_INVALID_ARG;
    if (np > (int64_t(1) << 30)) return MUON_ERR_INVALID_ARG;
    if (ns_steps > 0 && (!coeff_in || (ncoeff_sets != 1 && ncoeff_sets != ns_steps))) return MUON_ERR_INVALID_ARG;
    std::vector<float> coeffs(3 * static_cast<size_t>(ns_steps));
    for (int st = 0; st < ns_steps; ++st)
        for (int j = 0; j < 3; ++j) {
            const float v = coeff_in[(ncoeff_sets == 1 ? 0 : 3 * st) + j];
            if (!finite(v)) return MUON_ERR_INVALID_ARG;
            coeffs[3 * st + j] = v;
        }
    if (count == 0) return MUON_OK;
    if (!X_in || !X_out || !workspace) return MUON_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X_in) | reinterpret_cast<uintptr_t>(X_out)) & 1u) return MUON_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
    const int64_t per = bytes_per_matrix(mp, np);
    if (per > static_cast<int64_t>(ws_bytes)) return MUON_ERR_WORKSPACE_TOO_SMALL;
    int num_sms = 0;
    muon_status_t s = device_info(&num_sms);
    if (s != MUON_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!capturing(st)) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
        DeviceMemoryCheck mem(dev);
        const size_t x_bytes = static_cast<size_t>(count * mp * np) * 2;
        if (!mem.owns(X_in, x_bytes) || !mem.owns(X_out, x_bytes) || !mem.owns(workspace, ws_bytes))
            return MUON_ERR_INVALID_ARG;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    s = from_cuda(cudaMemsetAsync(ws, 0, sizeof(WsHeader), st));
    if (s != MUON_OK) return s;
    const int64_t per_chunk = static_cast<int64_t>(ws_bytes) / per;
    const size_t row_bytes = static_cast<size_t>(np) * 2;
    for (int64_t first = 0; first < count; first += per_chunk) {
        const int64_t cnt = std::min(per_chunk, count - first);
        NsGroup g;
        g.mp = mp;
        g.np = np;
        g.ldx = round_up(np, 8);
        g.lda = round_up(mp, 8);
        g.x_stride = round_up(2 * mp * g.ldx, 256);
        g.g_stride = round_up(2 * mp * g.lda, 256);
        g.count = cnt;
        g.scale = nullptr;
        g.scale_stride = 0;
        uint8_t* cursor = ws + cnt * static_cast<int64_t>(kRecordBytes);
        g.X[0] = reinterpret_cast<uint16_t*>(cursor);
        g.X[1] = reinterpret_cast<uint16_t*>(cursor + cnt * g.x_stride);
        g.A = reinterpret_cast<uint16_t*>(cursor + 2 * cnt * g.x_stride);
        g.B = reinterpret_cast<uint16_t*>(cursor + 2 * cnt * g.x_stride + cnt * g.g_stride);
        // With rows a multiple of 8 wide the workspace rows are unpadded, so
        // each matrix is one contiguous run and one strided copy moves the
        // whole chunk (a matrix per copy "row", its pitch below the 2 GiB a
        // copy pitch may reach); ragged widths copy matrix by matrix, row
        // pitch and all.
        const size_t mat_bytes = row_bytes * static_cast<size_t>(mp);
        const bool whole = g.ldx == np && g.x_stride < (int64_t(1) << 31);
        if (whole) {
            s = from_cuda(cudaMemcpy2DAsync(g.X[0], g.x_stride, X_in + first * mp * np, mat_bytes, mat_bytes, cnt,
                                            cudaMemcpyDeviceToDevice, st));
            if (s != MUON_OK) return s;
        } else {
            for (int64_t k = 0; k < cnt; ++k) {
                s = from_cuda(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(g.X[0]) + k * g.x_stride, g.ldx * 2,
                                                X_in + (first + k) * mp * np, row_bytes, row_bytes, mp,
                                                cudaMemcpyDeviceToDevice, st));
                if (s != MUON_OK) return s;
            }
        }
        s = from_cuda(ns_run(&g, 1, ns_steps, coeffs.data(), status, num_sms, st));
        if (s != MUON_OK) return s;
        const uint16_t* res = g.X[ns_steps & 1];
        if (whole) {
            s = from_cuda(cudaMemcpy2DAsync(X_out + first * mp * np, mat_bytes, res, g.x_stride, mat_bytes, cnt,
                                            cudaMemcpyDeviceToDevice, st));
            if (s != MUON_OK) return s;
        } else {
            for (int64_t k = 0; k < cnt; ++k) {
                s = from_cuda(cudaMemcpy2DAsync(X_out + (first + k) * mp * np, row_bytes,
                                                reinterpret_cast<const uint8_t*>(res) + k * g.x_stride, g.ldx * 2,
                                                row_bytes, mp, cudaMemcpyDeviceToDevice, st));
                if (s != MUON_OK) return s;
            }
        }
    }
    return MUON_OK;
}

}  // extern "C"

namespace {

// AdamW hyper-parameters and step count -> the kernels' scalars, with the
// bias corrections 1 - beta^step computed in fp64 and rounded to fp32.
muon_status_t adamw_scalars(const adamw_hparams_t* hp, int64_t step, AdamwScalars* sc) {
    if (!hp || step < 1) return MUON_ERR_INVALID_ARG;
    if (!finite(hp->lr) || !finite(hp->beta1) || !finite(hp->beta2) || !finite(hp->eps) ||
        !finite(hp->weight_decay))
        return MUON_ERR_INVALID_ARG;
    if (hp->beta1 < 0.f || hp->beta1 >= 1.f || hp->beta2 < 0.f || hp->beta2 >= 1.f || hp->eps < 0.f)
        return MUON_ERR_INVALID_ARG;
    sc->lr = hp->lr;
    sc->beta1 = hp->beta1;
    sc->beta2 = hp->beta2;
    sc->one_minus_beta1 = 1.0f - hp->beta1;
    sc->one_minus_beta2 = 1.0f - hp->beta2;
    sc->bc1 = static_cast<float>(1.0 - pow(static_cast<double>(hp->beta1), static_cast<double>(step)));
    sc->bc2 = static_cast<float>(1.0 - pow(static_cast<double>(hp->beta2), static_cast<double>(step)));
    sc->eps = hp->eps;
    sc->weight_decay = hp->weight_decay;
    if (!(sc->bc1 > 0.f) || !(sc->bc2 > 0.f)) return MUON_ERR_INVALID_ARG;
    return MUON_OK;
}

// One AdamW tensor's pointer checks: non-null, 4-byte aligned.
muon_status_t check_adamw_tensor(const float* p, const float* g, const float* m, const float* v) {
    if (!p || !g || !m || !v) return MUON_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(m) |
         reinterpret_cast<uintptr_t>(v)) & 3u)
        return MUON_ERR_MISALIGNED;
    return MUON_OK;
}

// One AdamW call's buffers on the current device (left out under capture).
muon_status_t check_adamw_memory(const adamw_tensor_t* tensors, int64_t count, cudaStream_t st) {
    if (capturing(st)) return MUON_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
    DeviceMemoryCheck mem(dev);
    for (int64_t i = 0; i < count; ++i) {
        const adamw_tensor_t& x = tensors[i];
        if (x.n == 0) continue;
        const size_t bytes = static_cast<size_t>(x.n) * 4u;
        if (!mem.owns(x.p, bytes) || !mem.owns(x.g, bytes) || !mem.owns(x.m, bytes) || !mem.owns(x.v, bytes))
            return MUON_ERR_INVALID_ARG;
    }
    return MUON_OK;
}

// Whether byte ranges [start, end) are pairwise disjoint (sorted in place).
bool disjoint(std::vector<std::pair<uintptr_t, uintptr_t>>& ranges) {
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second) return false;
    return true;
}

}  // namespace

extern "C" {

muon_status_t adamw_step(float* p, const float* g, float* m, float* v, int64_t n, const adamw_hparams_t* hp,
                         int64_t step, void* stream) {
    NvtxScope range("adamw_step");
    AdamwScalars sc;
    muon_status_t s = adamw_scalars(hp, step, &sc);
    if (s != MUON_OK) return s;
    if (n < 0) return MUON_ERR_INVALID_ARG;
    if (n == 0) return MUON_OK;
    s = check_adamw_tensor(p, g, m, v);
    if (s != MUON_OK) return s;
    // the four buffers must be pairwise disjoint
    const uintptr_t len = static_cast<uintptr_t>(n) * 4u;
    std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
    for (const void* b : {static_cast<const void*>(p), static_cast<const void*>(g), static_cast<const void*>(m),
                          static_cast<const void*>(v)})
        ranges.emplace_back(reinterpret_cast<uintptr_t>(b), reinterpret_cast<uintptr_t>(b) + len);
    if (!disjoint(ranges)) return MUON_ERR_INVALID_ARG;
    int num_sms = 0;
    s = device_info(&num_sms);
    if (s != MUON_OK) return s;
    adamw_tensor_t one;
    one.p = p;
    one.g = g;
    one.m = m;
    one.v = v;
    one.n = n;
    s = check_adamw_memory(&one, 1, static_cast<cudaStream_t>(stream));
    if (s != MUON_OK) return s;
    return from_cuda(launch_adamw(p, g, m, v, n, sc, num_sms, static_cast<cudaStream_t>(stream)));
}

muon_status_t adamw_step_batched(const adamw_tensor_t* tensors, int64_t count, const adamw_hparams_t* hp,
                                 int64_t step, void* stream) {
    NvtxScope range("adamw_step_batched");
    AdamwScalars sc;
    muon_status_t s = adamw_scalars(hp, step, &sc);
    if (s != MUON_OK) return s;
    if (count < 0 || (count > 0 && !tensors)) return MUON_ERR_INVALID_ARG;
    std::vector<std::pair<uintptr_t, uintptr_t>> ranges;
    for (int64_t i = 0; i < count; ++i) {
        const adamw_tensor_t& x = tensors[i];
        if (x.n < 0 || x.n > (int64_t(1) << 40)) return MUON_ERR_INVALID_ARG;
        if (x.n == 0) continue;
        s = check_adamw_tensor(x.p, x.g, x.m, x.v);
        if (s != MUON_OK) return s;
        const uintptr_t len = static_cast<uintptr_t>(x.n) * 4u;
        for (const void* b : {static_cast<const void*>(x.p), static_cast<const void*>(x.g),
                              static_cast<const void*>(x.m), static_cast<const void*>(x.v)})
            ranges.emplace_back(reinterpret_cast<uintptr_t>(b), reinterpret_cast<uintptr_t>(b) + len);
    }
    if (ranges.empty()) return MUON_OK;
    if (!disjoint(ranges)) return MUON_ERR_INVALID_ARG;
    int num_sms = 0;
    s = device_info(&num_sms);
    if (s != MUON_OK) return s;
    s = check_adamw_memory(tensors, count, static_cast<cudaStream_t>(stream));
    if (s != MUON_OK) return s;
    return from_cuda(launch_adamw_multi(tensors, count, sc, num_sms, static_cast<cudaStream_t>(stream)));
}

muon_status_t muon_check_bounded_wait(void* workspace, int64_t limit_us, void* stream) {
    if (!workspace || limit_us < 1 || limit_us > 10000000) return MUON_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_ERR_MISALIGNED;
    int num_sms = 0;
    muon_status_t s = device_info(&num_sms);
    if (s != MUON_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!capturing(st)) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
        DeviceMemoryCheck mem(dev);
        if (!mem.owns(workspace, sizeof(WsHeader))) return MUON_ERR_INVALID_ARG;
    }
    WsHeader* header = static_cast<WsHeader*>(workspace);
    s = from_cuda(cudaMemsetAsync(header, 0, sizeof(WsHeader), st));
    if (s != MUON_OK) return s;
    return from_cuda(launch_wait_probe(&header->status, static_cast<long long>(limit_us) * 1000, st));
}

muon_status_t muon_query_status(void* workspace, void* stream) {
    if (!workspace) return MUON_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MUON_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
    if (host != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MUON_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
        return static_cast<muon_status_t>(host);
    }
    return MUON_OK;
}

}  // extern "C"
