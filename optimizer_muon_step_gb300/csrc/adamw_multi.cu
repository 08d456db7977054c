// Multi-tensor AdamW: one launch updates up to kBatch tensors.
//
// The tensor table travels in the kernel's parameter block (no host buffer
// outlives the call).  The launch's threads stride, as the single-tensor
// kernel does over one buffer, over the concatenation of every tensor's
// float4 groups (tensors whose four buffers are 16-byte aligned), then over
// the concatenation of the remaining single elements (those tensors' tails
// and every element of the other tensors).  A thread's index only grows, so
// it finds the tensor of each index by advancing through the table's
// offsets.  Large tensors are thus read in the same contiguous sweep as by
// the single-tensor kernel, and small ones are spread over all CTAs.  Each
// element goes through adamw_elem, the same rounded fp32 sequence as the
// single-tensor kernels, so the results equal adamw_step's bit for bit.
#include <memory>
#include <new>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 448;  // tensors per launch

struct AdamwBatch {
    AdamwScalars s;
    int32_t count;
    int64_t vec_begin[kBatch + 1];  // tensor t's float4 groups: [vec_begin[t], vec_begin[t + 1])
    int64_t sc_begin[kBatch + 1];   // its single elements: [sc_begin[t], sc_begin[t + 1])
    int64_t sc_first[kBatch];       // element index of its first single element
    float* p[kBatch];
    const float* g[kBatch];
    float* m[kBatch];
    float* v[kBatch];
};
static_assert(sizeof(AdamwBatch) <= 32764, "kernel parameter limit");

__global__ void __launch_bounds__(kThreads) adamw_multi_kernel(const __grid_constant__ AdamwBatch b) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t nvec = b.vec_begin[b.count];
    int t = 0;
    for (int64_t j = first; j < nvec; j += stride) {
        while (j >= b.vec_begin[t + 1]) ++t;
        const int64_t i = 4 * (j - b.vec_begin[t]);
        // every byte is touched once: streaming (evict-first) loads and stores
        float4 pp = __ldcs(reinterpret_cast<const float4*>(b.p[t] + i));
        const float4 gg = __ldcs(reinterpret_cast<const float4*>(b.g[t] + i));
        float4 mm = __ldcs(reinterpret_cast<const float4*>(b.m[t] + i));
        float4 vv = __ldcs(reinterpret_cast<const float4*>(b.v[t] + i));
        adamw_elem(pp.x, gg.x, mm.x, vv.x, b.s);
        adamw_elem(pp.y, gg.y, mm.y, vv.y, b.s);
        adamw_elem(pp.z, gg.z, mm.z, vv.z, b.s);
        adamw_elem(pp.w, gg.w, mm.w, vv.w, b.s);
        __stcs(reinterpret_cast<float4*>(b.p[t] + i), pp);
        __stcs(reinterpret_cast<float4*>(b.m[t] + i), mm);
        __stcs(reinterpret_cast<float4*>(b.v[t] + i), vv);
    }
    const int64_t nsc = b.sc_begin[b.count];
    t = 0;
    for (int64_t j = first; j < nsc; j += stride) {
        while (j >= b.sc_begin[t + 1]) ++t;
        const int64_t i = b.sc_first[t] + (j - b.sc_begin[t]);
        float pp = b.p[t][i], mm = b.m[t][i], vv = b.v[t][i];
        adamw_elem(pp, b.g[t][i], mm, vv, b.s);
        b.p[t][i] = pp;
        b.m[t][i] = mm;
        b.v[t][i] = vv;
    }
}

}  // namespace

cudaError_t launch_adamw_multi(const adamw_tensor_t* tensors, int64_t count, AdamwScalars s, int num_sms,
                               cudaStream_t st) {
    for (int64_t off = 0; off < count; off += kBatch) {
        const int n = static_cast<int>(count - off < kBatch ? count - off : kBatch);
        std::unique_ptr<AdamwBatch> b(new (std::nothrow) AdamwBatch());
        if (!b) return cudaErrorMemoryAllocation;
        b->s = s;
        b->count = n;
        int64_t nvec = 0, nsc = 0;
        for (int k = 0; k < n; ++k) {
            const adamw_tensor_t& x = tensors[off + k];
            const bool aligned = ((reinterpret_cast<uintptr_t>(x.p) | reinterpret_cast<uintptr_t>(x.g) |
                                   reinterpret_cast<uintptr_t>(x.m) | reinterpret_cast<uintptr_t>(x.v)) & 15u) == 0;
            const int64_t groups = aligned ? x.n / 4 : 0;
            b->vec_begin[k] = nvec;
            b->sc_begin[k] = nsc;
            b->sc_first[k] = 4 * groups;
            b->p[k] = x.p;
            b->g[k] = x.g;
            b->m[k] = x.m;
            b->v[k] = x.v;
            nvec += groups;
            nsc += x.n - 4 * groups;
        }
        b->vec_begin[n] = nvec;
        b->sc_begin[n] = nsc;
        const int64_t work = nvec > nsc ? nvec : nsc;
        if (work == 0) continue;
        const int64_t cap = static_cast<int64_t>(num_sms) * 8;
        const int64_t blocks = (work + kThreads - 1) / kThreads;
        const int grid = static_cast<int>(blocks < cap ? blocks : cap);
        launch_begin(MUON_KERNEL_ADAMW, st);
        adamw_multi_kernel<<<grid, kThreads, 0, st>>>(*b);
        launch_end(MUON_KERNEL_ADAMW, st);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace muon
