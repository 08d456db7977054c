// Library-internal declarations shared by the CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

#include "muon_step.h"

namespace muon {

// Per-matrix record the element-wise kernels read (device copy lives in the
// workspace).  All buffers are row-major.  X buffers hold the wide
// (m' x n') orientation with row stride `ldx`.
struct MatDesc {
    float* W;
    const void* G;
    float* M;
    uint16_t* X0;        // NS input, bf16 bits
    const uint16_t* O;   // NS output, bf16 bits (X0 or X1)
    float* partials;     // per-tile sums of u^2 (kMaxNormTiles entries)
    int64_t rows, cols;  // caller's orientation
    int64_t ldx;         // row stride of X0 / O in elements
    int64_t tile_len;    // elements per flat tile (multiple of 8): wide momentum pass, gradient guard
    int32_t ntiles;      // flat tiles
    int32_t g_kind;      // G's element type: 0 fp32, 1 bf16, 2 fp16 (muon_dtype_t)
    int32_t transposed;  // 1: rows > cols, X holds the transpose
    int32_t vec;         // 1: W, G, M are 16-byte aligned
    float scale;         // 1 / (||u||_F + eps), written by the finalize kernel
    float update_scale;  // rms_scale * sqrt(n')
    int32_t nparts;      // partials the momentum pass writes (flat tiles, or tall units)
    int32_t tall_kr;     // tall pass: 64-row tiles per unit
    int32_t tall_kc;     // tall pass: 64-column tiles per unit
    int32_t rescaled;    // 1: X0 is multiplied in place by rescale_factor before NS
    float rescale_factor;
    float ns_scale;      // factor the first NS step applies to X0
    double gsum;         // gradient guard: sum of G^2 over the matrix (fp64)
    muon_matrix_stats_t* stats;  // this matrix's statistics entry (device), or null
};

constexpr int kMaxNormTiles = 1024;
constexpr int kStatsTiles = 512;          // row tiles of the statistics pass per matrix
constexpr size_t kRecordBytes = 8192;     // per matrix, see muon_step.h
constexpr size_t kHeaderBytes = 256;
// a matrix's record and partials fit its kRecordBytes (header and rounding
// covered by the slack); the NS kernels index ns_scale in float strides
static_assert(sizeof(MatDesc) + sizeof(float) * (kMaxNormTiles + kStatsTiles) + 512 <= kRecordBytes,
              "record overflow");
static_assert(sizeof(MatDesc) % sizeof(float) == 0, "record stride");

// Start of the workspace: status word and the gradient guard's results.
struct WsHeader {
    int32_t status;               // muon_status_t recorded by kernels
    int32_t pad0;
    double sumsq;                 // sum of G^2 over every matrix of the call
    unsigned long long nonfinite; // non-finite gradient elements
    float clip;                   // gradient scale (1 when clipping is off)
    int32_t skip;                 // 1: the non-finite guard skips the step
};

struct MomentumScalars {
    float mu, one_minus_mu;
    int32_t nesterov;
    int32_t scale_g;              // 1: multiply G by header->clip first
    const WsHeader* header;       // guard results (device)
};

struct UpdateScalars {
    float lr, weight_decay;
    const WsHeader* header;       // skip flag (device); may be null
};

struct AdamwScalars {
    float lr, beta1, beta2, one_minus_beta1, one_minus_beta2;
    float bc1, bc2, eps, weight_decay;
};

// ---- programmatic dependent launch ------------------------------------------
// The kernels of one step form a chain on one stream.  Those launched with
// launch_pdl may be scheduled before the kernel ahead of them has finished:
// each runs pdl_wait_then_release() before it touches global memory, which
// waits until every kernel ahead of it has completed and its writes are
// visible, and then lets the kernel behind it launch.  A chained kernel's
// CTAs can thus start on idle SMs, and run any prologue that touches only
// shared memory, TMEM and kernel parameters, while the kernel ahead
// finishes.  Waiting before releasing keeps at most one kernel ahead.  After
// a non-kernel stream operation (memset, copy, event) the launch falls back
// to plain stream order.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One AdamW element ("LLM training series, part 2: optimizers", sections 2.3
// and 3.1), each operation a separately rounded fp32 op in this order:
//   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g g
//   p = p - lr ((m / bc1) / (sqrt(v / bc2) + eps) + wd p)
__device__ __forceinline__ void adamw_elem(float& p, float g, float& m, float& v, const AdamwScalars& s) {
    const float mi = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.one_minus_beta1, g));
    const float g2 = __fmul_rn(g, g);
    const float vi = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.one_minus_beta2, g2));
    const float m_hat = __fdiv_rn(mi, s.bc1);
    const float v_hat = __fdiv_rn(vi, s.bc2);
    const float den = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
    const float upd = __fdiv_rn(m_hat, den);
    const float decay = __fmul_rn(s.weight_decay, p);
    p = __fsub_rn(p, __fmul_rn(s.lr, __fadd_rn(upd, decay)));
    m = mi;
    v = vi;
}
#endif

// ---- launch accounting (timing.cu) -----------------------------------------
// Every kernel launch is bracketed by launch_begin / launch_end: they count
// launches, open and close an NVTX range named for the kernel kind, and,
// when timing is enabled, record CUDA events on the stream.  With the
// environment variable MUON_DEBUG set to a nonzero value, launch_end also
// synchronises the stream (unless it is being captured) and reports a
// failed kernel by name on stderr.
void launch_begin(int kind, cudaStream_t st);
void launch_end(int kind, cudaStream_t st);
// Between capture_begin and capture_end the calling thread's launches go
// into a graph: they are counted apart (capture_end returns the count) and
// never timed.  count_replay adds a replayed graph's launches to the total.
void capture_begin();
int64_t capture_end();
void count_replay(int64_t launches);

// An NVTX range over a scope of host code (an API call).
struct NvtxScope {
    explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope&) = delete;
    NvtxScope& operator=(const NvtxScope&) = delete;
};

// ---- per-matrix records (elementwise.cu) ----------------------------------
// Writes descs[0..count) to d_descs on `st` through kernel parameters, so the
// upload needs no host buffer that outlives the call (stream-capture safe).
// With zero_header non-null the first upload kernel also clears that
// workspace header (status word, guard results) before writing records: a
// step starts with a clean header and no memset in its launch chain.
cudaError_t launch_desc_upload(MatDesc* d_descs, const MatDesc* descs, int count, WsHeader* zero_header,
                               cudaStream_t st);

// ---- element-wise kernels (elementwise.cu) --------------------------------
// Momentum pass: M updated, X0 = bf16(u) in the wide orientation (tall
// matrices through a tiled transpose), per-unit sums of u^2 into the
// partials.  wide_tiles[k] bounds ntiles over the wide matrices and
// tall_units[k] nparts over the tall ones whose gradient type is k (3
// entries each, one per muon_dtype_t).
cudaError_t launch_momentum_norm(const MatDesc* descs, int count, const int* wide_tiles, const int* tall_units,
                                 MomentumScalars s, cudaStream_t st);
// Norm: scale = 1 / (||u|| + eps) per matrix; the first NS step applies
// ns_scale to X0 = bf16(u).  Normally ns_scale = scale.  A norm outside the
// range where products of bf16(u) elements stay normal fp32 numbers moves
// a power of two 2^k from the scale into X0 (X0 *= 2^k, ns_scale = scale *
// 2^-k: exact, the NS result is unchanged).  With `force_rescale` (no NS
// step follows) X0 = bf16(X0 * scale) and ns_scale = 1.
cudaError_t launch_norm_finalize(MatDesc* descs, int count, float eps, int force_rescale, cudaStream_t st);
// Final update: wide matrices over the momentum pass's flat tiles
// (max_wide_tiles bounds ntiles), tall ones over units of one 64-column tile
// by up to four 64-row tiles (max_tall_units bounds
// final_update_tall_units over the tall matrices).
int64_t final_update_tall_units(int64_t rows, int64_t cols);
cudaError_t launch_final_update(const MatDesc* descs, int count, int max_wide_tiles, int64_t max_tall_units,
                                UpdateScalars s, cudaStream_t st);
cudaError_t launch_adamw(float* p, const float* g, float* m, float* v, int64_t n,
                         AdamwScalars s, int num_sms, cudaStream_t st);
// Multi-tensor AdamW (adamw_multi.cu): every tensor of the host array updated
// exactly as launch_adamw would, one launch per 448 tensors.
cudaError_t launch_adamw_multi(const adamw_tensor_t* tensors, int64_t count, AdamwScalars s, int num_sms,
                               cudaStream_t st);
// Gradient guard: per-tile sums of G^2 into the partials and a count of
// non-finite elements into the header; then, per chunk, the partials summed
// in order into header->sumsq; finally the clip factor and skip flag.
cudaError_t launch_grad_stats(const MatDesc* descs, int count, int max_tiles, WsHeader* header,
                              cudaStream_t st);
cudaError_t launch_grad_stats_reduce(MatDesc* descs, int count, WsHeader* header, cudaStream_t st);
cudaError_t launch_grad_decide(WsHeader* header, float max_grad_norm, int32_t skip_nonfinite,
                               cudaStream_t st);

// ---- step statistics (stats.cu) ------------------------------------------
// For every matrix with a stats entry: the RMS of scale * O over row tiles
// into o_partials (kStatsTiles floats per matrix), then ||u||_F from the
// norm partials and the update RMS into the entry (NaN when the guard's
// skip flag is set in `header`; header may be null).
cudaError_t launch_step_stats(const MatDesc* descs, int count, float* o_partials, const WsHeader* header,
                              cudaStream_t st);

// ---- Newton-Schulz GEMMs (ns_gemm.cu) -------------------------------------
// One shape group of wide bf16 matrices in the workspace: `count` matrices,
// each X buffer [mp][ldx], each Gram buffer [mp][lda]; consecutive matrices
// are `x_stride` / `g_stride` bytes apart.
struct NsGroup {
    uint16_t* X[2];
    uint16_t* A;
    uint16_t* B;
    int64_t mp, np, ldx, lda;
    int64_t x_stride, g_stride;  // bytes
    int64_t count;
    // Per-matrix factor the first step applies to X (X0 holds the scaled
    // input divided by it): matrix k's factor at scale[k * scale_stride];
    // null when X0 is the input as is.
    const float* scale;
    int64_t scale_stride;
};

constexpr int kNsMaxGroups = 4;

// Runs `steps` Newton-Schulz steps on every group; the result of each
// group ends in X[steps % 2].  `status` is a device int the kernels set on a
// bounded-wait timeout.  Returns a CUDA error or cudaSuccess; a tensor-map
// encoding failure returns cudaErrorInvalidValue.
// `coeffs` is host memory of 3 * steps floats, step s using coeffs[3s..3s+2].
// Launches the failure-detection self-check: a bounded wait that runs out
// after limit_ns and records MUON_ERR_TIMEOUT in *status.
cudaError_t launch_wait_probe(int* status, long long limit_ns, cudaStream_t st);

cudaError_t ns_run(const NsGroup* groups, int ngroups, int steps, const float* coeffs,
                   int* status, int num_sms, cudaStream_t st);
// Sets the NS kernels' attributes and queries the pair occupancy for the
// current device now (ns_run otherwise does it on first use), e.g. before a
// stream capture.
cudaError_t ns_prepare_device();

}  // namespace muon
