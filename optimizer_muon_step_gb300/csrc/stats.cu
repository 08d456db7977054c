// Per-matrix statistics of a Muon step, on request (muon_step_batched_stats):
//
//   u_norm      ||u||_F of the look-ahead, from the momentum pass's fp32
//               tile sums of u^2 (the norm the step normalised by), summed
//               in fp64
//   update_rms  the RMS of scale * O, the RMS-matched update before lr and
//               decay.  "Kimi K2 ... what is worth noting" (section 3.1)
//               matches it to AdamW's update RMS of 0.2-0.4.
//
// Two launches per workspace chunk, after the final update: a pass over each
// matrix's NS output O (wide, bf16, row stride ldx) in row tiles, writing
// one fp32 sum of fl(scale * o)^2 per tile, then one warp per matrix adding
// the tile sums in a fixed order in fp64.  Nothing here is on the step's
// own data path: W, M and O are only read.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// One CTA per (row tile, matrix).  Rows per tile: ceil(m' / kStatsTiles).
// Each thread sums fl(fl(scale * o)^2) over its share of the tile in fp32,
// then the block adds the 256 thread sums in a fixed tree order.
__global__ void __launch_bounds__(kThreads) stats_o_kernel(const MatDesc* __restrict__ descs,
                                                           float* __restrict__ o_partials) {
    const MatDesc& d = descs[blockIdx.y];
    if (d.stats == nullptr) return;
    const int64_t mp = d.rows < d.cols ? d.rows : d.cols;
    const int64_t np = d.rows < d.cols ? d.cols : d.rows;
    const int64_t rows_per = (mp + kStatsTiles - 1) / kStatsTiles;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per;
    if (r0 >= mp) return;
    const int64_t r1 = r0 + rows_per < mp ? r0 + rows_per : mp;
    const float sc = d.update_scale;
    const int64_t ldx = d.ldx;  // a multiple of 8: every row starts 16-byte aligned
    const int64_t nvec = np / 8;
    float acc = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        const uint16_t* row = d.O + r * ldx;
        for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
            const uint4 q = *reinterpret_cast<const uint4*>(row + 8 * v);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = __fmul_rn(sc, bf16_bits_to_f32(w[k] & 0xffffu));
                const float hi = __fmul_rn(sc, bf16_bits_to_f32(w[k] >> 16));
                acc = __fadd_rn(acc, __fmul_rn(lo, lo));
                acc = __fadd_rn(acc, __fmul_rn(hi, hi));
            }
        }
        for (int64_t c = 8 * nvec + threadIdx.x; c < np; c += kThreads) {
            const float x = __fmul_rn(sc, bf16_bits_to_f32(row[c]));
            acc = __fadd_rn(acc, __fmul_rn(x, x));
        }
    }
    __shared__ float sums[kThreads];
    sums[threadIdx.x] = acc;
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) sums[threadIdx.x] = __fadd_rn(sums[threadIdx.x], sums[threadIdx.x + s]);
        __syncthreads();
    }
    if (threadIdx.x == 0) o_partials[static_cast<int64_t>(blockIdx.y) * kStatsTiles + blockIdx.x] = sums[0];
}

// One warp per matrix: lane l adds tile sums l, l + 32, ... in fp64, then
// the lanes combine in a fixed butterfly order.
__global__ void __launch_bounds__(kThreads) stats_finalize_kernel(const MatDesc* __restrict__ descs, int count,
                                                                  const float* __restrict__ o_partials,
                                                                  const WsHeader* __restrict__ header) {
    const int m = static_cast<int>((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (m >= count) return;
    const MatDesc& d = descs[m];
    if (d.stats == nullptr) return;
    if (header != nullptr && header->skip) {
        if (lane == 0) {
            d.stats->u_norm = nan("");
            d.stats->update_rms = nan("");
        }
        return;
    }
    const int64_t mp = d.rows < d.cols ? d.rows : d.cols;
    const int64_t rows_per = (mp + kStatsTiles - 1) / kStatsTiles;
    const int otiles = static_cast<int>((mp + rows_per - 1) / rows_per);
    double su = 0.0, so = 0.0;
    for (int i = lane; i < d.nparts; i += 32) su += static_cast<double>(d.partials[i]);
    for (int i = lane; i < otiles; i += 32) so += static_cast<double>(o_partials[static_cast<int64_t>(m) * kStatsTiles + i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        su += __shfl_xor_sync(0xffffffffu, su, off);
        so += __shfl_xor_sync(0xffffffffu, so, off);
    }
    if (lane == 0) {
        d.stats->u_norm = sqrt(su);
        d.stats->update_rms = sqrt(so / (static_cast<double>(d.rows) * static_cast<double>(d.cols)));
    }
}

}  // namespace

cudaError_t launch_step_stats(const MatDesc* descs, int count, float* o_partials, const WsHeader* header,
                              cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    for (int off = 0; off < count; off += 65535) {
        const int n = count - off < 65535 ? count - off : 65535;
        launch_begin(MUON_KERNEL_STATS, st);
        stats_o_kernel<<<dim3(kStatsTiles, n), kThreads, 0, st>>>(descs + off,
                                                                   o_partials + static_cast<int64_t>(off) * kStatsTiles);
        launch_end(MUON_KERNEL_STATS, st);
    }
    const int per = kThreads / 32;
    launch_begin(MUON_KERNEL_STATS, st);
    stats_finalize_kernel<<<(count + per - 1) / per, kThreads, 0, st>>>(descs, count, o_partials, header);
    launch_end(MUON_KERNEL_STATS, st);
    return cudaGetLastError();
}

}  // namespace muon
