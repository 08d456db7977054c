// Element-wise stages of the Muon step and the AdamW step (HBM-bound).
//
//   momentum_norm   M = mu M + (1-mu) G;  u = (1-mu) G + mu M;  per-tile sum
//                   u^2;  X0 = bf16(u) in the wide orientation (a tiled
//                   shared-memory transpose for tall matrices)
//   norm_finalize   s = 1 / (sqrt(sum u^2) + eps) per matrix (fp64 sum); the
//                   first NS step applies s to X0 (s^2 to X0 X0^T), so the
//                   normalised input s * bf16(u) is never stored; a matrix
//                   whose norm lies outside [2^-40, 2^40] has a power of
//                   two moved from s into X0 (exact)
//   final_update    W = W - lr (wd W + scale O)
//   grad guard      global sum of G^2 and non-finite count; clip factor
//                   and skip decision
//   adamw           AdamW on flat buffers
//   desc_upload     the per-matrix records into the workspace, carried as
//                   kernel parameters
//
// Formulas follow "LLM training series, part 2: optimizers" (mhpq.cn):
// momentum as an exponential moving average (section 2.1), Adam with bias
// correction (section 2.3), decoupled weight decay (section 3.1).  Every
// arithmetic step is an explicitly rounded fp32 intrinsic (__fmul_rn,
// __fadd_rn, ...) so no multiply-add is contracted and the results are
// reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include <memory>
#include <new>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;  // tile edge of the tall momentum and the final-update kernels

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// A 2-byte gradient element as fp32 (exact): bf16 or fp16 bits.
__device__ __forceinline__ float half_g_to_f32(uint32_t h, int g_kind) {
    return g_kind == MUON_F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
                              : __uint_as_float(h << 16);
}

// Two packed 2-byte gradient elements (the lower-addressed one in the low
// half) as fp32.
__device__ __forceinline__ void unpack_g2(uint32_t w, int g_kind, float& lo, float& hi) {
    if (g_kind == MUON_F16) {
        lo = __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
        hi = __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    } else {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
}

// Element i of a gradient of type g_kind (muon_dtype_t) as fp32.
__device__ __forceinline__ float load_g(const void* G, int g_kind, int64_t i) {
    return g_kind == MUON_F32 ? static_cast<const float*>(G)[i]
                              : half_g_to_f32(static_cast<const uint16_t*>(G)[i], g_kind);
}

// The gradient as the momentum sees it: clip * G when global-norm clipping
// is on (clip read once per CTA from the workspace header), else G.
__device__ __forceinline__ float scaled_g(float g, int scale_g, float clip) {
    return scale_g ? __fmul_rn(clip, g) : g;
}

// Momentum update and Nesterov look-ahead for one element.
__device__ __forceinline__ float momentum_elem(float g, float& m, const MomentumScalars& s) {
    float gterm = __fmul_rn(s.one_minus_mu, g);
    float mnew = __fadd_rn(__fmul_rn(s.mu, m), gterm);
    m = mnew;
    return s.nesterov ? __fadd_rn(gterm, __fmul_rn(s.mu, mnew)) : mnew;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    if (warp == 0) {
        t = lane < (kThreads / 32) ? red[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    return t;
}

// ---------------------------------------------------------------------------
// Momentum pass, wide matrices (rows <= cols, X0 = u): momentum, look-ahead,
// X0 = bf16(u) and a per-tile sum of squares.
// grid = (max tiles, matrices); each CTA handles one contiguous tile.
// ---------------------------------------------------------------------------
// One instance per gradient type (KIND, a muon_dtype_t), whose conversion
// it compiles in.
template <int KIND>
__global__ void __launch_bounds__(kThreads) momentum_norm_kernel(const MatDesc* __restrict__ descs,
                                                                 MomentumScalars s) {
    __shared__ float red[kThreads / 32];
    pdl_wait_then_release();
    const MatDesc& d = descs[blockIdx.y];
    const int tile = blockIdx.x;
    // tall matrices: momentum_tall_kernel; other gradient types: their instance
    if (d.transposed || tile >= d.ntiles || d.g_kind != KIND) return;
    if (s.header && s.header->skip) return;  // the non-finite guard skips the step
    const float clip = s.scale_g ? s.header->clip : 1.f;
    const int64_t n = d.rows * d.cols;
    const int64_t start = static_cast<int64_t>(tile) * d.tile_len;
    const int64_t end = min(n, start + d.tile_len);
    float* __restrict__ M = d.M;
    const void* G = d.G;
    constexpr int g_kind = KIND;
    uint16_t* __restrict__ X0 = d.X0;
    const int64_t cols = d.cols, ldx = d.ldx;
    const bool x_flat = ldx == cols;  // X0 rows packed: X0 index = element index
    float acc = 0.f;
    int64_t scalar_from = start;
    if (d.vec) {
        const int64_t nvec = (end - start) >> 3;
        for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
            const int64_t i = start + (v << 3);
            float g[8];
            if constexpr (KIND != MUON_F32) {
                uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(G) + i));
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) unpack_g2(w[j], KIND, g[2 * j], g[2 * j + 1]);
            } else {
                const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(G) + i);
                float4 a = __ldg(gp), b = __ldg(gp + 1);
                g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
                g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
            }
            float4* mp = reinterpret_cast<float4*>(M + i);
            float4 m0 = mp[0], m1 = mp[1];
            float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            uint32_t xb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float u = momentum_elem(scaled_g(g[j], s.scale_g, clip), m[j], s);
                acc = fmaf(u, u, acc);
                xb[j] = f32_to_bf16(u);
            }
            mp[0] = make_float4(m[0], m[1], m[2], m[3]);
            mp[1] = make_float4(m[4], m[5], m[6], m[7]);
            if (x_flat) {
                *reinterpret_cast<uint4*>(X0 + i) = make_uint4(xb[0] | (xb[1] << 16), xb[2] | (xb[3] << 16),
                                                               xb[4] | (xb[5] << 16), xb[6] | (xb[7] << 16));
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) X0[((i + j) / cols) * ldx + (i + j) % cols] = static_cast<uint16_t>(xb[j]);
            }
        }
        scalar_from = start + (nvec << 3);
    }
    for (int64_t i = scalar_from + threadIdx.x; i < end; i += kThreads) {
        float m = M[i];
        float u = momentum_elem(scaled_g(load_g(G, g_kind, i), s.scale_g, clip), m, s);
        M[i] = m;
        acc = fmaf(u, u, acc);
        X0[(i / cols) * ldx + i % cols] = f32_to_bf16(u);
    }
    float total = block_sum(acc, red);
    if (threadIdx.x == 0) d.partials[tile] = total;
}

// ---------------------------------------------------------------------------
// Momentum pass, tall matrices (rows > cols, X0 = u^T): the same step
// over 64x64 tiles, bf16(u) staged in shared memory and written transposed.
// A CTA ("unit") covers tall_kc column tiles x tall_kr row tiles and writes
// one partial.  grid = (max units, matrices).
// Thread (tx, ty) covers rows ty + 16 i (i < 4) and columns 4 tx .. 4 tx + 3.
// ---------------------------------------------------------------------------
// kPrefetch (2-byte gradients, bf16 or fp16): the next full tile's G and M are loaded into
// registers right after the current tile's momentum step, so they are in
// flight during its barriers and transposed X0 stores; four CTAs fit an SM
// (at most 64 registers a thread).  Without it (fp32 gradients, whose tiles
// already carry twice the bytes) six CTAs fit (at most 40 registers).
// Measured: prefetching made the bf16 pass 6% faster and the fp32 one 8%
// slower; at the unbounded 118 registers only two CTAs fit and the kernel
// ran at a third of HBM bandwidth.  Each instance handles the tall matrices
// of one gradient type (KIND, a muon_dtype_t), whose conversion it compiles
// in.
template <int KIND>
__global__ void __launch_bounds__(kThreads, KIND != MUON_F32 ? 4 : 6) momentum_tall_kernel(
    const MatDesc* __restrict__ descs, MomentumScalars s) {
    constexpr bool kPrefetch = KIND != MUON_F32;
    __shared__ uint16_t tileT[kTile][kTile + 2];
    __shared__ float red[kThreads / 32];
    pdl_wait_then_release();
    const MatDesc& d = descs[blockIdx.y];
    const int unit = blockIdx.x;
    if (!d.transposed || unit >= d.nparts || d.g_kind != KIND) return;
    if (s.header && s.header->skip) return;
    const float clip = s.scale_g ? s.header->clip : 1.f;
    const int64_t rows = d.rows, cols = d.cols;
    const int64_t ctiles = (cols + kTile - 1) / kTile;
    const int64_t cunits = (ctiles + d.tall_kc - 1) / d.tall_kc;
    const int64_t ct_begin = (unit % cunits) * d.tall_kc;
    const int64_t ct_end = min(ctiles, ct_begin + d.tall_kc);
    const int64_t rt_begin = (unit / cunits) * d.tall_kr;
    const int64_t rt_end = min((rows + kTile - 1) / kTile, rt_begin + d.tall_kr);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float* __restrict__ M = d.M;
    const void* G = d.G;
    constexpr int g_kind = KIND;
    uint16_t* __restrict__ X0 = d.X0;
    const int64_t ldx = d.ldx;
    const int64_t nr = rt_end - rt_begin;
    const int64_t ntl = nr > 0 && ct_end > ct_begin ? (ct_end - ct_begin) * nr : 0;
    // tile t of the unit: column tile ct_begin + t / nr, row tile rt_begin + t % nr
    auto origin = [&](int64_t t, int64_t& r0, int64_t& c0) {
        c0 = (ct_begin + t / nr) * kTile;
        r0 = (rt_begin + t % nr) * kTile;
    };
    auto is_full = [&](int64_t r0, int64_t c0) {
        return d.vec && (cols % 4 == 0) && r0 + kTile <= rows && c0 + kTile <= cols;
    };
    // row ty + 16 i of a full tile, columns 4 tx .. 4 tx + 3
    auto load_row = [&](int i, int64_t r0, int64_t c0, float4& m4, float (&g)[4]) {
        const int64_t off = (r0 + ty + 16 * i) * cols + c0 + 4 * tx;
        m4 = *reinterpret_cast<const float4*>(M + off);
        if constexpr (KIND != MUON_F32) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(G) + off));
            unpack_g2(raw.x, KIND, g[0], g[1]);
            unpack_g2(raw.y, KIND, g[2], g[3]);
        } else {
            const float4 g4 = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(G) + off));
            g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
        }
    };
    // kPrefetch: the registers of one whole full tile
    float4 mreg[4];
    float greg[4][4];
    auto load_full = [&](int64_t r0, int64_t c0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) load_row(i, r0, c0, mreg[i], greg[i]);
    };
    float acc = 0.f;
    bool loaded = false;  // the registers hold tile t
    for (int64_t t = 0; t < ntl; ++t) {
        int64_t r0, c0;
        origin(t, r0, c0);
        const bool full = is_full(r0, c0);
        if (kPrefetch && full && !loaded) load_full(r0, c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rl = ty + 16 * i;
            const int64_t r = r0 + rl;
            const int64_t c = c0 + 4 * tx;
            uint16_t b[4] = {0, 0, 0, 0};
            if (full) {
                float4 m4;
                float gv[4];
                if (kPrefetch) {
                    m4 = mreg[i];
#pragma unroll
                    for (int j = 0; j < 4; ++j) gv[j] = greg[i][j];
                } else {
                    load_row(i, r0, c0, m4, gv);
                }
                float m[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float u = momentum_elem(scaled_g(gv[j], s.scale_g, clip), m[j], s);
                    acc = fmaf(u, u, acc);
                    b[j] = f32_to_bf16(u);
                }
                *reinterpret_cast<float4*>(M + r * cols + c) = make_float4(m[0], m[1], m[2], m[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (r < rows && c + j < cols) {
                        const int64_t off = r * cols + c + j;
                        float m = M[off];
                        const float u = momentum_elem(scaled_g(load_g(G, g_kind, off), s.scale_g, clip), m, s);
                        M[off] = m;
                        acc = fmaf(u, u, acc);
                        b[j] = f32_to_bf16(u);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) tileT[4 * tx + j][rl] = b[j];
        }
        // the next tile's loads go out before this tile's barriers and stores
        loaded = false;
        if (kPrefetch && t + 1 < ntl) {
            int64_t r1, c1;
            origin(t + 1, r1, c1);
            if (is_full(r1, c1)) {
                load_full(r1, c1);
                loaded = true;
            }
        }
        __syncthreads();
        // X0 row = original column, X0 column = original row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int cl = ty + 16 * i;
            const int64_t xr = c0 + cl;
            const int64_t xc = r0 + 4 * tx;
            if (xr >= cols) continue;
            if (full) {
                const uint2 packed =
                    make_uint2(tileT[cl][4 * tx] | (static_cast<uint32_t>(tileT[cl][4 * tx + 1]) << 16),
                               tileT[cl][4 * tx + 2] | (static_cast<uint32_t>(tileT[cl][4 * tx + 3]) << 16));
                *reinterpret_cast<uint2*>(X0 + xr * ldx + xc) = packed;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (xc + j < rows) X0[xr * ldx + xc + j] = tileT[cl][4 * tx + j];
            }
        }
        __syncthreads();
    }
    const float total = block_sum(acc, red);
    if (threadIdx.x == 0) d.partials[unit] = total;
}

// Norms for which the first NS step applies the scale itself: products of
// two bf16(u) elements of typical size ||u||^2 / (m n) stay far inside the
// normal fp32 range for any matrix up to 2^31 elements.
constexpr double kNormLo = 9.094947017729282e-13;  // 2^-40
constexpr double kNormHi = 1.099511627776e12;      // 2^40

// One warp per matrix: fp64 sum of the partials in a fixed order.
__global__ void __launch_bounds__(kThreads) norm_finalize_kernel(MatDesc* __restrict__ descs,
                                                                 int count, float eps, int force_rescale) {
    pdl_wait_then_release();
    const int k = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (k >= count) return;
    const MatDesc& d = descs[k];
    double s = 0.0;
    for (int i = lane; i < d.nparts; i += 32) s += static_cast<double>(d.partials[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
        const double norm = sqrt(s);
        const float scale = static_cast<float>(1.0 / (norm + static_cast<double>(eps)));
        MatDesc& out = descs[k];
        out.scale = scale;
        out.rescaled = 0;
        out.rescale_factor = 1.f;
        out.ns_scale = scale;
        if (force_rescale) {
            out.rescaled = 1;
            out.rescale_factor = scale;
            out.ns_scale = 1.f;
        } else if (norm > 0.0 && isfinite(norm) && (norm < kNormLo || norm > kNormHi)) {
            // 2^k ||u|| in [0.5, 1): X0 elements stay at most 1 in size
            int e = 0;
            frexp(norm, &e);
            out.rescaled = 1;
            out.rescale_factor = ldexpf(1.f, -e);
            out.ns_scale = ldexpf(scale, e);
        }
    }
}

// X0 = bf16(X0 * rescale_factor) for the matrices norm_finalize flagged.  A
// fixed grid first scans the flags together, then walks the flagged matrices.
constexpr int kRescaleCtas = 304;

__global__ void __launch_bounds__(kThreads) x0_rescale_kernel(const MatDesc* __restrict__ descs, int count) {
    pdl_wait_then_release();
    int flagged = 0;
    for (int k = threadIdx.x; k < count; k += kThreads) flagged |= descs[k].rescaled;
    if (!__syncthreads_or(flagged)) return;  // the usual case: nothing to do
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int k = 0; k < count; ++k) {
        const MatDesc& d = descs[k];
        if (!d.rescaled) continue;
        const float scale = d.rescale_factor;
        const int64_t mp = d.transposed ? d.cols : d.rows;
        const int64_t np = d.transposed ? d.rows : d.cols;
        const int64_t ldx = d.ldx;
        uint16_t* __restrict__ X0 = d.X0;
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; e < mp * np; e += stride) {
            uint16_t* x = X0 + (e / np) * ldx + e % np;
            *x = f32_to_bf16(__fmul_rn(bf16_to_f32(*x), scale));
        }
    }
}

// ---------------------------------------------------------------------------
// Final update: W = W - lr (wd W + scale O), O read from the wide buffer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float update_elem(float w, float o, float sc, const UpdateScalars& u) {
    float decay = __fmul_rn(u.weight_decay, w);
    float step = __fmul_rn(sc, o);
    float delta = __fmul_rn(u.lr, __fadd_rn(decay, step));
    return __fsub_rn(w, delta);
}

// Final update of wide matrices (rows <= cols, O in the caller's layout) over
// the momentum pass's flat tiles: one CTA per tile of tile_len elements,
// 8 elements a thread per iteration.  grid = (max tiles, matrices).
__global__ void __launch_bounds__(kThreads) final_update_wide_kernel(const MatDesc* __restrict__ descs,
                                                                     UpdateScalars us) {
    pdl_wait_then_release();
    const MatDesc& d = descs[blockIdx.y];
    const int tile = blockIdx.x;
    if (d.transposed || tile >= d.ntiles) return;
    if (us.header && us.header->skip) return;
    const float sc = d.update_scale;
    float* __restrict__ W = d.W;
    const uint16_t* __restrict__ O = d.O;
    const int64_t cols = d.cols, ldx = d.ldx;
    const int64_t n = d.rows * cols;
    const int64_t start = static_cast<int64_t>(tile) * d.tile_len;
    const int64_t end = min(n, start + d.tile_len);
    int64_t scalar_from = start;
    if (d.vec && ldx == cols) {
        const int64_t nvec = (end - start) >> 3;
        for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
            const int64_t i = start + (v << 3);
            float4* wp = reinterpret_cast<float4*>(W + i);
            float4 a = wp[0], b = wp[1];
            const uint4 o = *reinterpret_cast<const uint4*>(O + i);
            a.x = update_elem(a.x, __uint_as_float(o.x << 16), sc, us);
            a.y = update_elem(a.y, __uint_as_float(o.x & 0xffff0000u), sc, us);
            a.z = update_elem(a.z, __uint_as_float(o.y << 16), sc, us);
            a.w = update_elem(a.w, __uint_as_float(o.y & 0xffff0000u), sc, us);
            b.x = update_elem(b.x, __uint_as_float(o.z << 16), sc, us);
            b.y = update_elem(b.y, __uint_as_float(o.z & 0xffff0000u), sc, us);
            b.z = update_elem(b.z, __uint_as_float(o.w << 16), sc, us);
            b.w = update_elem(b.w, __uint_as_float(o.w & 0xffff0000u), sc, us);
            wp[0] = a;
            wp[1] = b;
        }
        scalar_from = start + (nvec << 3);
    }
    for (int64_t i = scalar_from + threadIdx.x; i < end; i += kThreads)
        W[i] = update_elem(W[i], bf16_to_f32(O[(i / cols) * ldx + i % cols]), sc, us);
}

// Final update of tall matrices (rows > cols, O holds the transpose): a CTA
// takes one 64-column tile by up to kFinalRowTiles 64-row tiles (units in
// column-tile order), O^T staged through shared memory.  The next tile's O
// and W are loaded into registers right after the current tile's update, so
// they are in flight during its barrier.  grid = (max units, matrices).
constexpr int kFinalRowTiles = 4;

inline __host__ __device__ int64_t final_tall_units(int64_t rows, int64_t cols) {
    const int64_t rt = (rows + kTile - 1) / kTile;
    return (cols + kTile - 1) / kTile * ((rt + kFinalRowTiles - 1) / kFinalRowTiles);
}

__global__ void __launch_bounds__(kThreads, 4) final_update_tall_kernel(const MatDesc* __restrict__ descs,
                                                                        UpdateScalars us) {
    __shared__ uint16_t tileT[kTile][kTile + 2];
    pdl_wait_then_release();
    const MatDesc& d = descs[blockIdx.y];
    const int unit = blockIdx.x;
    if (!d.transposed) return;
    const int64_t rows = d.rows, cols = d.cols, ldx = d.ldx;
    if (unit >= final_tall_units(rows, cols)) return;
    if (us.header && us.header->skip) return;
    const float sc = d.update_scale;
    float* __restrict__ W = d.W;
    const uint16_t* __restrict__ O = d.O;
    // tile counts fit 32 bits: rows, cols <= 2^30
    const int ctiles = static_cast<int>((cols + kTile - 1) / kTile);
    const int64_t c0u = static_cast<int64_t>(unit % ctiles) * kTile;
    const int rt_begin = (unit / ctiles) * kFinalRowTiles;
    const int rt_end = min(static_cast<int>((rows + kTile - 1) / kTile), rt_begin + kFinalRowTiles);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int ntl = rt_end - rt_begin;
    auto origin = [&](int t, int64_t& r0, int64_t& c0) {
        c0 = c0u;
        r0 = static_cast<int64_t>(rt_begin + t) * kTile;
    };
    auto is_full = [&](int64_t r0, int64_t c0) {
        return d.vec && (cols % 4 == 0) && r0 + kTile <= rows && c0 + kTile <= cols;
    };
    // registers of one full tile: O rows c0 + ty + 16 i, columns r0 + 4 tx ..;
    // W rows r0 + ty + 16 i, columns c0 + 4 tx ..
    uint2 oreg[4];
    float4 wreg[4];
    auto load_full = [&](int64_t r0, int64_t c0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            oreg[i] = *reinterpret_cast<const uint2*>(O + (c0 + ty + 16 * i) * ldx + r0 + 4 * tx);
            wreg[i] = *reinterpret_cast<const float4*>(W + (r0 + ty + 16 * i) * cols + c0 + 4 * tx);
        }
    };
    bool loaded = false;  // the registers hold tile t
    for (int t = 0; t < ntl; ++t) {
        int64_t r0, c0;
        origin(t, r0, c0);
        const bool full = is_full(r0, c0);
        if (full && !loaded) load_full(r0, c0);
        // stage O^T: O rows c0.., columns r0..
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int cl = ty + 16 * i;
            if (full) {
                tileT[cl][4 * tx] = oreg[i].x & 0xffffu;
                tileT[cl][4 * tx + 1] = oreg[i].x >> 16;
                tileT[cl][4 * tx + 2] = oreg[i].y & 0xffffu;
                tileT[cl][4 * tx + 3] = oreg[i].y >> 16;
            } else {
                const int64_t orow = c0 + cl;
                const int64_t ocol = r0 + 4 * tx;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tileT[cl][4 * tx + j] = (orow < cols && ocol + j < rows) ? O[orow * ldx + ocol + j] : 0;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rl = ty + 16 * i;
            const int64_t r = r0 + rl;
            const int64_t c = c0 + 4 * tx;
            if (full) {
                float4 w4 = wreg[i];
                w4.x = update_elem(w4.x, bf16_to_f32(tileT[4 * tx][rl]), sc, us);
                w4.y = update_elem(w4.y, bf16_to_f32(tileT[4 * tx + 1][rl]), sc, us);
                w4.z = update_elem(w4.z, bf16_to_f32(tileT[4 * tx + 2][rl]), sc, us);
                w4.w = update_elem(w4.w, bf16_to_f32(tileT[4 * tx + 3][rl]), sc, us);
                *reinterpret_cast<float4*>(W + r * cols + c) = w4;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (r < rows && c + j < cols)
                        W[r * cols + c + j] = update_elem(W[r * cols + c + j], bf16_to_f32(tileT[4 * tx + j][rl]), sc, us);
            }
        }
        // the next tile's loads go out before this tile's closing barrier
        loaded = false;
        if (t + 1 < ntl) {
            int64_t r1, c1;
            origin(t + 1, r1, c1);
            if (is_full(r1, c1)) {
                load_full(r1, c1);
                loaded = true;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Gradient guard ("LLM training series, part 2: optimizers", section 5.4:
// skip a step whose gradients hold Inf/NaN; clip by the global norm).
// ---------------------------------------------------------------------------
// Each CTA sums kGuardTiles consecutive momentum tiles of one matrix: the
// sum goes to the first tile's partial, zeros to the others.
constexpr int kGuardTiles = 4;

__global__ void __launch_bounds__(kThreads) grad_stats_kernel(const MatDesc* __restrict__ descs,
                                                              WsHeader* __restrict__ header) {
    __shared__ float red[kThreads / 32];
    const MatDesc& d = descs[blockIdx.y];
    const int tile = blockIdx.x * kGuardTiles;
    if (tile >= d.ntiles) return;
    const int last = min(d.ntiles, tile + kGuardTiles);
    const int64_t n = d.rows * d.cols;
    const int64_t start = static_cast<int64_t>(tile) * d.tile_len;
    const int64_t end = min(n, static_cast<int64_t>(last) * d.tile_len);
    const void* G = d.G;
    const int g_kind = d.g_kind;
    float acc = 0.f;
    unsigned int bad = 0;
    int64_t scalar_from = start;
    if (d.vec) {
        const int64_t nvec = (end - start) >> 3;
        for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
            const int64_t i = start + (v << 3);
            float g[8];
            if (g_kind != MUON_F32) {
                uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(G) + i));
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                if (g_kind == MUON_F16) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) unpack_g2(w[j], MUON_F16, g[2 * j], g[2 * j + 1]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) unpack_g2(w[j], MUON_BF16, g[2 * j], g[2 * j + 1]);
                }
            } else {
                const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(G) + i);
                float4 a = __ldg(gp), b = __ldg(gp + 1);
                g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
                g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                acc = fmaf(g[j], g[j], acc);
                bad += isfinite(g[j]) ? 0u : 1u;
            }
        }
        scalar_from = start + (nvec << 3);
    }
    for (int64_t i = scalar_from + threadIdx.x; i < end; i += kThreads) {
        const float g = load_g(G, g_kind, i);
        acc = fmaf(g, g, acc);
        bad += isfinite(g) ? 0u : 1u;
    }
    const float total = block_sum(acc, red);
    if (threadIdx.x == 0) {
        d.partials[tile] = total;
        for (int t = tile + 1; t < last; ++t) d.partials[t] = 0.f;
    }
    if (bad) atomicAdd(&header->nonfinite, static_cast<unsigned long long>(bad));
}

// One warp per matrix sums its partials in fp64 in a fixed order (lane
// strides, then a fixed shuffle tree) into the matrix's record.
__global__ void __launch_bounds__(kThreads) grad_stats_reduce_kernel(MatDesc* __restrict__ descs, int count) {
    const int k = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (k >= count) return;
    MatDesc& d = descs[k];
    double s = 0.0;
    for (int i = lane; i < d.ntiles; i += 32) s += static_cast<double>(d.partials[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) d.gsum = s;
}

// One warp adds the matrices' sums to header->sumsq: lane l sums matrices
// l, l + 32, ... in order, then a fixed shuffle tree, so the total does not
// depend on scheduling.
__global__ void __launch_bounds__(32) grad_stats_total_kernel(const MatDesc* __restrict__ descs, int count,
                                                             WsHeader* __restrict__ header) {
    const int lane = threadIdx.x;
    double s = 0.0;
    for (int k = lane; k < count; k += 32) s += descs[k].gsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) header->sumsq += s;
}

__global__ void grad_decide_kernel(WsHeader* __restrict__ header, float max_grad_norm, int32_t skip_nonfinite) {
    if (threadIdx.x != 0) return;
    float clip = 1.f;
    if (max_grad_norm > 0.f) {
        const double c = static_cast<double>(max_grad_norm) / (sqrt(header->sumsq) + 1e-6);
        clip = static_cast<float>(c < 1.0 ? c : 1.0);
    }
    header->clip = clip;
    const int32_t skip = (skip_nonfinite && header->nonfinite > 0) ? 1 : 0;
    header->skip = skip;
    if (skip) atomicCAS(&header->status, 0, static_cast<int>(MUON_STEP_SKIPPED));
}

// ---------------------------------------------------------------------------
// AdamW
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) adamw_vec_kernel(float4* __restrict__ p, const float4* __restrict__ g,
                                                             float4* __restrict__ m, float4* __restrict__ v,
                                                             int64_t nvec, AdamwScalars s) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec; i += stride) {
        float4 pp = __ldcs(p + i), gg = __ldcs(g + i), mm = __ldcs(m + i), vv = __ldcs(v + i);
        adamw_elem(pp.x, gg.x, mm.x, vv.x, s);
        adamw_elem(pp.y, gg.y, mm.y, vv.y, s);
        adamw_elem(pp.z, gg.z, mm.z, vv.z, s);
        adamw_elem(pp.w, gg.w, mm.w, vv.w, s);
        __stcs(p + i, pp);
        __stcs(m + i, mm);
        __stcs(v + i, vv);
    }
}

__global__ void __launch_bounds__(kThreads) adamw_scalar_kernel(float* __restrict__ p, const float* __restrict__ g,
                                                                float* __restrict__ m, float* __restrict__ v,
                                                                int64_t begin, int64_t n, AdamwScalars s) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride) {
        float pp = p[i], mm = m[i], vv = v[i];
        adamw_elem(pp, g[i], mm, vv, s);
        p[i] = pp;
        m[i] = mm;
        v[i] = vv;
    }
}

inline unsigned grid_for(int64_t work, int64_t per_block, int64_t cap) {
    int64_t b = (work + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return static_cast<unsigned>(b);
}

// Per-matrix records passed by value: one launch carries up to K of them in
// its parameter block (kernel parameters may take up to 32764 bytes on
// sm_70 and later), so the upload reads no host buffer after the launch and
// a captured graph keeps the records in its kernel node.
template <int K>
struct DescBatch {
    MatDesc* dst;
    WsHeader* zero_header;  // cleared by this launch before the records land; null: left alone
    int32_t count;
    MatDesc d[K];
};
constexpr int kUploadSmall = 8;
constexpr int kUploadLarge = 224;
static_assert(sizeof(DescBatch<kUploadLarge>) <= 32764, "kernel parameter limit");
static_assert(sizeof(MatDesc) % 4 == 0, "word copy");

template <int K>
__global__ void __launch_bounds__(kThreads) desc_upload_kernel(const __grid_constant__ DescBatch<K> b) {
    constexpr int kWords = static_cast<int>(sizeof(MatDesc) / 4);
    pdl_wait_then_release();
    if (b.zero_header) {
        uint32_t* h = reinterpret_cast<uint32_t*>(b.zero_header);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(WsHeader) / 4); i += blockDim.x) h[i] = 0u;
    }
    const uint32_t* src = reinterpret_cast<const uint32_t*>(b.d);
    uint32_t* dst = reinterpret_cast<uint32_t*>(b.dst);
    for (int i = threadIdx.x; i < b.count * kWords; i += blockDim.x) dst[i] = src[i];
}
static_assert(sizeof(WsHeader) % 4 == 0, "word clear");

template <int K>
cudaError_t upload_batch(MatDesc* d_descs, const MatDesc* descs, int count, WsHeader* zero_header,
                         cudaStream_t st) {
    std::unique_ptr<DescBatch<K>> b(new (std::nothrow) DescBatch<K>());
    if (!b) return cudaErrorMemoryAllocation;
    b->dst = d_descs;
    b->zero_header = zero_header;
    b->count = count;
    memcpy(b->d, descs, sizeof(MatDesc) * static_cast<size_t>(count));
    launch_begin(MUON_KERNEL_DESC_UPLOAD, st);
    cudaError_t e = launch_pdl(desc_upload_kernel<K>, dim3(1), dim3(kThreads), 0, st, *b);
    launch_end(MUON_KERNEL_DESC_UPLOAD, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

}  // namespace

cudaError_t launch_desc_upload(MatDesc* d_descs, const MatDesc* descs, int count, WsHeader* zero_header,
                               cudaStream_t st) {
    for (int done = 0; done < count;) {
        const int left = count - done;
        const int n = left < kUploadLarge ? left : kUploadLarge;
        WsHeader* z = done == 0 ? zero_header : nullptr;
        const cudaError_t e = n <= kUploadSmall ? upload_batch<kUploadSmall>(d_descs + done, descs + done, n, z, st)
                                                : upload_batch<kUploadLarge>(d_descs + done, descs + done, n, z, st);
        if (e != cudaSuccess) return e;
        done += n;
    }
    return cudaSuccess;
}

// wide_tiles[k]: largest ntiles over the wide matrices, tall_units[k]:
// largest nparts over the tall matrices, whose gradient type is k (a
// muon_dtype_t; 0 when there are none of that type).
cudaError_t launch_momentum_norm(const MatDesc* descs, int count, const int* wide_tiles, const int* tall_units,
                                 MomentumScalars s, cudaStream_t st) {
    cudaError_t err = cudaSuccess;
    auto keep = [&](cudaError_t e) { if (err == cudaSuccess) err = e; };
    for (int off = 0; off < count; off += 65535) {
        int n = count - off < 65535 ? count - off : 65535;
        if (wide_tiles[MUON_BF16] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_norm_kernel<MUON_BF16>, dim3(wide_tiles[MUON_BF16], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
        if (wide_tiles[MUON_F16] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_norm_kernel<MUON_F16>, dim3(wide_tiles[MUON_F16], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
        if (wide_tiles[MUON_F32] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_norm_kernel<MUON_F32>, dim3(wide_tiles[MUON_F32], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
        if (tall_units[MUON_BF16] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_tall_kernel<MUON_BF16>, dim3(tall_units[MUON_BF16], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
        if (tall_units[MUON_F16] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_tall_kernel<MUON_F16>, dim3(tall_units[MUON_F16], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
        if (tall_units[MUON_F32] > 0) {
            launch_begin(MUON_KERNEL_MOMENTUM_NORM, st);
            keep(launch_pdl(momentum_tall_kernel<MUON_F32>, dim3(tall_units[MUON_F32], n), dim3(kThreads), 0, st,
                            descs + off, s));
            launch_end(MUON_KERNEL_MOMENTUM_NORM, st);
        }
    }
    keep(cudaGetLastError());
    return err;
}

int64_t final_update_tall_units(int64_t rows, int64_t cols) { return final_tall_units(rows, cols); }

cudaError_t launch_norm_finalize(MatDesc* descs, int count, float eps, int force_rescale, cudaStream_t st) {
    const int per = kThreads / 32;
    launch_begin(MUON_KERNEL_NORM_FINALIZE, st);
    cudaError_t err = launch_pdl(norm_finalize_kernel, dim3((count + per - 1) / per), dim3(kThreads), 0, st, descs,
                                 count, eps, force_rescale);
    launch_end(MUON_KERNEL_NORM_FINALIZE, st);
    launch_begin(MUON_KERNEL_X0_RESCALE, st);
    const cudaError_t e2 = launch_pdl(x0_rescale_kernel, dim3(kRescaleCtas), dim3(kThreads), 0, st, descs, count);
    launch_end(MUON_KERNEL_X0_RESCALE, st);
    if (err == cudaSuccess) err = e2;
    if (err == cudaSuccess) err = cudaGetLastError();
    return err;
}

cudaError_t launch_final_update(const MatDesc* descs, int count, int max_wide_tiles, int64_t max_tall_units,
                                UpdateScalars s, cudaStream_t st) {
    if (max_tall_units > 0x7fffffff) return cudaErrorInvalidValue;
    cudaError_t err = cudaSuccess;
    auto keep = [&](cudaError_t e) { if (err == cudaSuccess) err = e; };
    for (int off = 0; off < count; off += 65535) {
        int n = count - off < 65535 ? count - off : 65535;
        if (max_wide_tiles > 0) {
            launch_begin(MUON_KERNEL_FINAL_UPDATE, st);
            keep(launch_pdl(final_update_wide_kernel, dim3(max_wide_tiles, n), dim3(kThreads), 0, st, descs + off, s));
            launch_end(MUON_KERNEL_FINAL_UPDATE, st);
        }
        if (max_tall_units > 0) {
            launch_begin(MUON_KERNEL_FINAL_UPDATE, st);
            keep(launch_pdl(final_update_tall_kernel, dim3(static_cast<unsigned>(max_tall_units), n), dim3(kThreads), 0,
                            st, descs + off, s));
            launch_end(MUON_KERNEL_FINAL_UPDATE, st);
        }
    }
    keep(cudaGetLastError());
    return err;
}

cudaError_t launch_grad_stats(const MatDesc* descs, int count, int max_tiles, WsHeader* header,
                              cudaStream_t st) {
    for (int off = 0; off < count; off += 65535) {
        int n = count - off < 65535 ? count - off : 65535;
        launch_begin(MUON_KERNEL_GRAD_GUARD, st);
        grad_stats_kernel<<<dim3((max_tiles + kGuardTiles - 1) / kGuardTiles, n), kThreads, 0, st>>>(descs + off,
                                                                                                  header);
        launch_end(MUON_KERNEL_GRAD_GUARD, st);
    }
    return cudaGetLastError();
}

cudaError_t launch_grad_stats_reduce(MatDesc* descs, int count, WsHeader* header, cudaStream_t st) {
    const int per = kThreads / 32;
    launch_begin(MUON_KERNEL_GRAD_GUARD, st);
    grad_stats_reduce_kernel<<<(count + per - 1) / per, kThreads, 0, st>>>(descs, count);
    launch_end(MUON_KERNEL_GRAD_GUARD, st);
    launch_begin(MUON_KERNEL_GRAD_GUARD, st);
    grad_stats_total_kernel<<<1, 32, 0, st>>>(descs, count, header);
    launch_end(MUON_KERNEL_GRAD_GUARD, st);
    return cudaGetLastError();
}

cudaError_t launch_grad_decide(WsHeader* header, float max_grad_norm, int32_t skip_nonfinite, cudaStream_t st) {
    launch_begin(MUON_KERNEL_GRAD_GUARD, st);
    grad_decide_kernel<<<1, 32, 0, st>>>(header, max_grad_norm, skip_nonfinite);
    launch_end(MUON_KERNEL_GRAD_GUARD, st);
    return cudaGetLastError();
}

cudaError_t launch_adamw(float* p, const float* g, float* m, float* v, int64_t n, AdamwScalars s,
                         int num_sms, cudaStream_t st) {
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    const bool aligned = ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(g) |
                           reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
    int64_t done = 0;
    if (aligned) {
        const int64_t nvec = n / 4;
        if (nvec > 0) {
            launch_begin(MUON_KERNEL_ADAMW, st);
            adamw_vec_kernel<<<grid_for(nvec, kThreads, cap), kThreads, 0, st>>>(
                reinterpret_cast<float4*>(p), reinterpret_cast<const float4*>(g),
                reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), nvec, s);
            launch_end(MUON_KERNEL_ADAMW, st);
        }
        done = nvec * 4;
    }
    if (done < n) {
        launch_begin(MUON_KERNEL_ADAMW, st);
        adamw_scalar_kernel<<<grid_for(n - done, kThreads, cap), kThreads, 0, st>>>(p, g, m, v, done, n, s);
        launch_end(MUON_KERNEL_ADAMW, st);
    }
    return cudaGetLastError();
}

}  // namespace muon
