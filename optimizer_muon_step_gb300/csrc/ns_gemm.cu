// Newton-Schulz orthogonalisation on Blackwell tensor cores (sm_103a).
//
// One step of the odd matrix polynomial on a batch of wide bf16 matrices X
// (m' x n', m' <= n'), as three grouped GEMM launches:
//
//   SYRK    A = X X^T            tiles of the upper block band only
//   POLY    B = b A + c (A A)    tiles of the upper block band only
//   UPDATE  X' = a X + B X       all tiles
//
// The iteration is the one "LLM training series, part 2: optimizers"
// (mhpq.cn, section 4.2) describes: it pushes the singular values of X
// towards 1 without an SVD.  The cubic member there is (a, b, c) =
// (1.5, -0.5, 0); the library's default is the quintic (3.4445, -4.7750,
// 2.0315).  A and B are symmetric, so SYRK and POLY compute and store only
// the upper block band: with row blocks of S rows (S = 128 on single CTAs,
// 256 on CTA pairs), block (p, q) is stored when q >= p, diagonal blocks in
// full.  A consumer reading rows of block p along k takes the k-blocks of
// blocks q >= p as stored (K-major) and those of q < p from the transposed
// position (block (q, p), read MN-major): A[r][k] = A[k][r].  Nothing is
// stored twice and nothing below the band is ever read.
//
// Two kernels share the epilogue: a single-CTA kernel on 128x256 tiles and
// a CTA-pair kernel (tcgen05 cta_group::2) on 256x256 pair tiles, chosen per
// shape group (see use_pairs).
//
// Single-CTA kernel design (one persistent CTA per SM, 6 warps):
//   warp 0       TMA producer: 128B-swizzled tiles of both operands into a
//                4-stage shared-memory ring (mbarrier complete_tx)
//   warp 1       TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//                M=128 N=256 K=16, fp32 accumulators in TMEM, two 256-column
//                accumulator buffers so the epilogue of one tile overlaps the
//                main loop of the next
//   warps 2..5   epilogue, one warp per TMEM lane quarter: tcgen05.ld 32
//                lanes x 32 columns, fused polynomial / update arithmetic
//                in fp32, 32x64 bf16 blocks in and out through TMA
// X is read K-major by SYRK and MN-major by UPDATE (its B operand); A and B
// are read K-major or MN-major per k-block as above.  The instruction
// descriptor's per-operand major bits select the layout per MMA, so no
// matrix is ever transposed in memory.  Every wait is bounded: after
// ~2 seconds a CTA records MUON_ERR_TIMEOUT, drains what it issued, frees
// its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace muon {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
// A ring stage holds KPS consecutive 64-deep k-blocks: the MMA thread waits
// on one barrier per stage, and fewer, larger stages cut that per-k-block
// round trip (a wait on the full barrier and the tcgen05 fence after it).
// Measured on CTA pairs: two k-blocks per stage took 8-9% fewer MMA-thread
// cycles than one; three (two stages in the ring) starved the MMA.
#ifndef MUON_KPS_SINGLE
#define MUON_KPS_SINGLE 1
#endif
constexpr int KPS = MUON_KPS_SINGLE;             // single-CTA kernel: k-blocks per stage
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int SUB_BYTES = A_BYTES + B_BYTES;     // one k-block
constexpr int STAGES = 4 / KPS;
constexpr int STAGE_BYTES = KPS * SUB_BYTES;
#ifndef MUON_EPI_WARPS
#define MUON_EPI_WARPS 4
#endif
constexpr int EPI_WARPS = MUON_EPI_WARPS;  // 4 or 8; two warps per TMEM lane quarter when 8
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;  // two BN-column fp32 accumulators
#ifndef MUON_EPI_COLS
#define MUON_EPI_COLS 64
#endif
constexpr int EPI_COLS = MUON_EPI_COLS;                    // columns of one epilogue block: 32 or 64
constexpr int EROW_BYTES = EPI_COLS * 2;                   // one block row, bf16; also its swizzle span
constexpr int EBUF_BYTES = 32 * EROW_BYTES;                // one 32-row bf16 block
constexpr int NSLOT = 32768 / (EPI_WARPS * EBUF_BYTES);    // block buffers per epilogue warp (32 KB in all)
constexpr int MN_CHUNK_BYTES = 64 * BK * 2;                // one 64-row chunk of an MN-major operand
constexpr int EBUFS_BYTES = EPI_WARPS * NSLOT * EBUF_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EBUFS_BYTES + 256;
constexpr unsigned long long kDrainNs = 500000000ull;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

enum Mode { MODE_SYRK = 0, MODE_POLY = 1, MODE_UPDATE = 2 };

// MN-major operands (64-row chunks of the M or N dimension, each 64 k-rows
// of 128 bytes, 8 KB apart) are loaded one of two ways.  A "chunked" map
// views a row-major matrix whose width is a multiple of 64 as
// [matrix][chunk][row][64 elements] (chunk stride 128 bytes), so a single
// box {64, 64, C} brings C chunks in one copy; other widths take one
// {64, 64} box per chunk from a plain 3-D map.  Fewer, larger copies keep
// the TMA unit ahead of the tensor core.
struct GroupParams {
    CUtensorMap tm_a;      // A operand: rows of the left factor, K-major, box {64, 128}
    CUtensorMap tm_b;      // B operand: K-major box {64, 256} (pairs {64, 128}); UPDATE: X MN-major
    CUtensorMap tm_t;      // symmetric factor read MN-major (transposed position), 2 chunks per copy
    CUtensorMap tm_e;      // epilogue addend, box {EPI_COLS, 32}, swizzled over the row
    CUtensorMap tm_d;      // output block store, box {EPI_COLS, 32}, swizzled over the row
    const float* scale;    // first step of SYRK/UPDATE: X = scale * X0 per matrix, else null
    int64_t scale_stride;  // floats between consecutive matrices' scales
    int32_t M, N, K;
    int32_t count;
    int32_t tiles_n;
    int32_t tiles_per_mat;
    int32_t tile_begin;
    int32_t chunked;       // MN-major maps are chunked (4-D); else plain 3-D {64, 64} boxes
};

struct NsParams {
    GroupParams g[kNsMaxGroups];
    int32_t num_groups;
    int32_t total_tiles;
    float alpha;  // multiplies the addend E
    float beta;   // multiplies the accumulator
    int* status;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (another role timed out) or this wait itself ran past the limit, in which
// case the abort flag and the global status word are set.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int* status, unsigned long long limit_ns = kTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(status, 0, static_cast<int>(MUON_ERR_TIMEOUT));
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: used to let copies and MMAs this
// CTA issued land before it releases TMEM and exits.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kDrainNs) return;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 consecutive fp32 columns; the wait is in the same asm block
// so no use of the registers can be scheduled before the data has landed.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 family layout:
// start address, leading and stride byte offsets (all >> 4), fixed version
// bits 46..48 = 0b001, swizzle mode 2 (128B) in bits 61..63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), A and B major-ness (bits 15, 16), N >> 3
// (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t instr_desc(int m, int n, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Descriptor of the k-th 16-deep slice of an operand staged by one k-block
// load.  K-major: 128-byte rows of 64 k, 8-row groups 1024 bytes apart.
// MN-major: 64-element chunks of rows 8 KB apart, each 64 k-rows of 128
// bytes.  In both layouts row r of the operand starts r * 128 bytes in
// (for r a multiple of 64), which the caller adds to `base`.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k, bool mn_major) {
    return mn_major ? smem_desc(base + static_cast<uint32_t>(k) * 16 * 128, MN_CHUNK_BYTES, 1024)
                    : smem_desc(base + static_cast<uint32_t>(k) * 32, 16, 1024);
}

// Whether rows of row block `row_block` read k-block kb (64 wide) of a
// symmetric factor from the transposed position: blocks of 2^shift k-blocks.
__device__ __forceinline__ bool read_transposed(int kb, int row_block, int shift) {
    return (kb >> shift) < row_block;
}

// Copies of an MN-major operand covering rows [r0, r0 + 64 * nchunks) at
// k-block kb, chunk c landing at dst + c * 8 KB: `per_copy` chunks per copy
// from a chunked map (r0 a multiple of 64), or one {64, 64} box per chunk.
// LOAD3/LOAD4 issue a 3-D / 4-D tensor copy.
template <typename Load3, typename Load4>
__device__ __forceinline__ void load_mn(uint32_t dst, const CUtensorMap* map, bool chunked, int per_copy, int r0,
                                        int nchunks, int kb, int mat, Load3 load3, Load4 load4) {
    if (chunked) {
        for (int c = 0; c < nchunks; c += per_copy)
            load4(dst + static_cast<uint32_t>(c) * MN_CHUNK_BYTES, map, 0, kb * BK, (r0 >> 6) + c, mat);
    } else {
        for (int c = 0; c < nchunks; ++c)
            load3(dst + static_cast<uint32_t>(c) * MN_CHUNK_BYTES, map, r0 + 64 * c, kb * BK, mat);
    }
}

struct Tile {
    int group, mat, ti, tj;
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const NsParams& p, int t) {
    Tile out;
    int gi = 0;
    while (gi + 1 < p.num_groups && t >= p.g[gi + 1].tile_begin) ++gi;
    const GroupParams& g = p.g[gi];
    int local = t - g.tile_begin;
    out.group = gi;
    out.mat = local / g.tiles_per_mat;
    int r = local - out.mat * g.tiles_per_mat;
    if (MODE == MODE_UPDATE) {
        out.ti = r / g.tiles_n;
        out.tj = r - out.ti * g.tiles_n;
    } else {
        // upper-triangle band: row tile ti keeps column tiles tj >= ti / 2
        int ti = 0;
        for (;;) {
            const int cnt = g.tiles_n - (ti >> 1);
            if (r < cnt) break;
            r -= cnt;
            ++ti;
        }
        out.ti = ti;
        out.tj = (ti >> 1) + r;
    }
    return out;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Epilogue of one tile, run by one warp over its 32 TMEM lanes (rows) and
// the tile's 8 chunks of 32 columns.
// ---------------------------------------------------------------------------

// Chunk values packed as bf16 pairs, w[i] = columns (2i, 2i+1):
//   SYRK  beta*acc;   POLY, UPDATE  alpha*E + beta*acc
// (beta = 1 for SYRK and UPDATE except on the first step, where the
// per-matrix input scale s gives SYRK beta = s^2 and UPDATE alpha = a s,
// beta = s; multiplying by 1 is exact.)
template <int MODE>
__device__ __forceinline__ void chunk_values(const float (&v)[32], const uint4 (&e)[4], float alpha, float beta,
                                             uint32_t (&w)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t ew[4] = {e[q].x, e[q].y, e[q].z, e[q].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int i = q * 4 + h;
            float lo = v[2 * i], hi = v[2 * i + 1];
            if (MODE == MODE_SYRK) {
                lo = __fmul_rn(beta, lo);
                hi = __fmul_rn(beta, hi);
            } else {
                lo = __fadd_rn(__fmul_rn(alpha, bf16_lo(ew[h])), __fmul_rn(beta, lo));
                hi = __fadd_rn(__fmul_rn(alpha, bf16_hi(ew[h])), __fmul_rn(beta, hi));
            }
            w[i] = pack_bf16x2(lo, hi);
        }
    }
}

// Per-warp state of the epilogue's bulk copies; lives across tiles.  Each
// epilogue warp owns a ring of NSLOT block buffers (32 rows x EPI_COLS,
// swizzled over the row length: 64 or 128 bytes); a slot takes a block's
// addend in and the finished block out.
struct EpiBufs {
    uint32_t buf[NSLOT];    // shared::cta addresses
    uint8_t* ptr[NSLOT];    // the same buffers as generic pointers
    uint32_t bar[NSLOT];    // mbarriers of addend loads into the slots
    uint32_t phase;         // bit b: parity of the next completion of bar[b]
    uint32_t pending;       // bit b: an addend load into slot b is in flight
    uint32_t seq;           // blocks this warp has written so far (all tiles)
};

// How many blocks ahead of its use a block's addend is requested.  A slot
// is reused once the bulk group NSLOT - AHEAD blocks back has been read.
#ifndef MUON_EPI_AHEAD
#define MUON_EPI_AHEAD NSLOT
#endif
constexpr int EPI_AHEAD = MUON_EPI_AHEAD;
static_assert(EPI_AHEAD >= 1 && EPI_AHEAD <= NSLOT, "addend distance must fit the ring");

// Waits for the accumulator, then writes the warp's share of the tile,
// blocks of 32 rows x EPI_COLS columns at a time:
//   addend (POLY: A, UPDATE: X): bulk tensor load into a ring slot,
//     requested EPI_AHEAD blocks ahead; the first ones before the
//     accumulator wait so they overlap the main loop;
//   output: each lane writes its row of the finished block into the same
//     slot (same swizzle) and one lane issues a bulk tensor store.  Rows or
//     columns past the matrix are clipped by the tensor store.
// Blocks left of `col_min` (SYRK/POLY: the first column of the tile's row
// block) lie below the stored band and are neither computed nor written.
// Returns false when the CTA is aborting.
template <int MODE>
__device__ __forceinline__ bool epilogue_tile(const NsParams& p, const GroupParams& g, const Tile& tile,
                                              int col_min, uint32_t t_acc, int quarter, int half, int lane,
                                              uint32_t tfull, uint32_t acc_phase, volatile int* abort_flag,
                                              EpiBufs& eb) {
    constexpr int CH = BN / EPI_COLS / (EPI_WARPS / 4);  // blocks of EPI_COLS columns this warp writes
    const int row_base = tile.ti * BM + quarter * 32;
    const int col_base = tile.tj * BN + half * CH * EPI_COLS;
    const int N = g.N;
    float alpha = p.alpha, beta = p.beta;
    if (MODE != MODE_POLY && g.scale != nullptr) {
        const float sc = g.scale[static_cast<int64_t>(tile.mat) * g.scale_stride];
        if (MODE == MODE_SYRK) {
            beta = __fmul_rn(sc, sc);
        } else {
            alpha = __fmul_rn(alpha, sc);
            beta = sc;
        }
    }

    // blocks this warp writes: [c_lo, c_hi), the same for all lanes
    int c_hi = CH;
    while (c_hi > 0 && col_base + EPI_COLS * (c_hi - 1) >= N) --c_hi;
    if (row_base >= g.M) c_hi = 0;  // every row of this warp is past the matrix
    int c_lo = 0;
    while (c_lo < c_hi && col_base + EPI_COLS * c_lo < col_min) ++c_lo;
    const int nblocks = c_hi - c_lo;

    // Blocks are numbered across tiles (eb.seq) and block n uses slot
    // n % NSLOT.  Every block commits exactly one bulk group, so after block
    // n's "at most NSLOT - AHEAD groups still reading" every slot of blocks
    // <= n - (NSLOT - AHEAD) is free -- in particular the slot the addend
    // load for block n + AHEAD overwrites, in this tile or the next one.
    const uint32_t s0 = eb.seq;
    auto issue = [&](int k) {  // addend of the k-th written block of this tile
        if (MODE == MODE_SYRK) return;
        const int b = static_cast<int>((s0 + k) % NSLOT);
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(eb.bar[b], EBUF_BYTES);
            tma_load_3d(eb.buf[b], &g.tm_e, col_base + EPI_COLS * (c_lo + k), row_base, tile.mat, eb.bar[b]);
        }
        eb.pending |= 1u << b;
    };
#pragma unroll
    for (int k = 0; k < EPI_AHEAD; ++k)
        if (k < nblocks) issue(k);

    if (!wait_bounded(tfull, acc_phase, abort_flag, p.status)) return false;
    tc_fence_after();
    const uint32_t t_addr = t_acc + (static_cast<uint32_t>(quarter * 32) << 16);
    // swizzle of this lane's row: 16-byte chunk q sits at q ^ sw
    const int sw = EROW_BYTES == 64 ? (lane >> 1) & 3 : lane & 7;

    for (int k = 0; k < nblocks; ++k) {
        const int c = c_lo + k;
        const int b = static_cast<int>((s0 + k) % NSLOT);
        __syncwarp();
        uint8_t* brow = eb.ptr[b] + lane * EROW_BYTES;
        if (MODE != MODE_SYRK) {
            if (!wait_bounded(eb.bar[b], (eb.phase >> b) & 1u, abort_flag, p.status)) return false;
            eb.phase ^= 1u << b;
            eb.pending &= ~(1u << b);
        }
#pragma unroll
        for (int h = 0; h < EPI_COLS / 32; ++h) {
            float v[32];
            tmem_load_32cols(t_addr + static_cast<uint32_t>((half * CH + c) * EPI_COLS + 32 * h), v);
            uint4 e[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                          make_uint4(0u, 0u, 0u, 0u)};
            if (MODE != MODE_SYRK) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    e[q] = *reinterpret_cast<const uint4*>(brow + (((4 * h + q) ^ sw) << 4));
            }
            uint32_t w[16];
            chunk_values<MODE>(v, e, alpha, beta, w);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(brow + (((4 * h + q) ^ sw) << 4)) =
                    make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(&g.tm_d, eb.buf[b], col_base + EPI_COLS * c, row_base, tile.mat);
            bulk_commit();
            bulk_wait_read<NSLOT - EPI_AHEAD>();
        }
        __syncwarp();
        if (k + EPI_AHEAD < nblocks) issue(k + EPI_AHEAD);
    }
    eb.seq = s0 + static_cast<uint32_t>(nblocks);
    return true;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) ns_gemm_kernel(const __grid_constant__ NsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;
    uint8_t* ebufs = smem + STAGES * STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ebufs + EBUFS_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tfull_bar = bars + 2 * STAGES;
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    uint64_t* ebar = bars + 2 * STAGES + 5;  // NSLOT per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ebar + NSLOT * EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), EPI_WARPS);
        }
        mbar_init(smem_u32(drain_bar), 1);
        for (int i = 0; i < NSLOT * EPI_WARPS; ++i) mbar_init(smem_u32(&ebar[i]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        for (int gi = 0; gi < p.num_groups; ++gi) {
            tma_prefetch_desc(&p.g[gi].tm_a);
            tma_prefetch_desc(&p.g[gi].tm_b);
            if (MODE != MODE_SYRK) tma_prefetch_desc(&p.g[gi].tm_e);
            tma_prefetch_desc(&p.g[gi].tm_d);
            if (MODE != MODE_SYRK) tma_prefetch_desc(&p.g[gi].tm_t);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above touched only shared memory, TMEM and parameters
    pdl_wait_then_release();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int last_parity[STAGES];
        for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
            const Tile tile = decode_tile<MODE>(p, t);
            const GroupParams& g = p.g[tile.group];
            const int nk = (g.K + BK - 1) / BK;
            for (int kb0 = 0; kb0 < nk; kb0 += KPS) {
                if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full_bar[stage]);
                const int nsub = nk - kb0 < KPS ? nk - kb0 : KPS;
                mbar_expect_tx(fb, SUB_BYTES * nsub);
                auto load3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
                    tma_load_3d(dst, map, c0, c1, c2, fb);
                };
                auto load4 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3) {
                    tma_load_4d(dst, map, c0, c1, c2, c3, fb);
                };
                const bool chunked = g.chunked != 0;
                for (int q = 0; q < nsub; ++q) {
                    const int kb = kb0 + q;
                    const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES + q * SUB_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    // A operand: 128 rows of row block ti (POLY/UPDATE read the
                    // symmetric factor transposed left of the diagonal block)
                    if (MODE != MODE_SYRK && read_transposed(kb, tile.ti, 1))
                        load_mn(sa, &g.tm_t, chunked, 2, tile.ti * BM, BM / 64, kb, tile.mat, load3, load4);
                    else
                        tma_load_3d(sa, &g.tm_a, kb * BK, tile.ti * BM, tile.mat, fb);
                    // B operand: 256 rows = row blocks 2tj and 2tj+1; UPDATE reads X
                    // MN-major (4 chunks per copy), POLY each half per its own block
                    const int n0 = tile.tj * BN;
                    const bool t0 = MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, 2 * tile.tj, 1));
                    const bool t1 = MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, 2 * tile.tj + 1, 1));
                    if (MODE == MODE_UPDATE)
                        load_mn(sb, &g.tm_b, chunked, 4, n0, BN / 64, kb, tile.mat, load3, load4);
                    else if (t0)
                        load_mn(sb, &g.tm_t, chunked, 2, n0, BN / 64, kb, tile.mat, load3, load4);
                    else if (t1) {
                        tma_load_3d(sb, &g.tm_a, kb * BK, n0, tile.mat, fb);  // 128 K-major rows
                        load_mn(sb + A_BYTES, &g.tm_t, chunked, 2, n0 + BM, BM / 64, kb, tile.mat, load3, load4);
                    } else {
                        tma_load_3d(sb, &g.tm_b, kb * BK, n0, tile.mat, fb);
                    }
                }
                last_parity[stage] = static_cast<int>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // drain: every issued copy must land before the CTA may exit
        for (int s = 0; s < STAGES; ++s) {
            if (last_parity[s] >= 0) wait_drain(smem_u32(&full_bar[s]), static_cast<uint32_t>(last_parity[s]));
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++local) {
            const Tile tile = decode_tile<MODE>(p, t);
            const GroupParams& g = p.g[tile.group];
            const int nk = (g.K + BK - 1) / BK;
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            if (!wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, p.status)) break;
            tc_fence_after();
            // Columns of the tile the MMAs compute, [n_lo, n_hi): an odd row
            // tile on the diagonal of SYRK/POLY needs only its right half (the
            // left half lies below the diagonal), and the last column tile of
            // a ragged matrix only up to the next multiple of 16 past N.
            int n_lo = 0, n_hi = BN;
            if (MODE != MODE_UPDATE && (tile.ti & 1) && tile.tj == (tile.ti >> 1)) n_lo = BN / 2;
            const int rem = g.N - tile.tj * BN;
            if (rem < BN) n_hi = (rem + 15) & ~15;
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb0 = 0; kb0 < nk; kb0 += KPS) {
                if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nsub = nk - kb0 < KPS ? nk - kb0 : KPS;
                for (int q = 0; q < nsub; ++q) {
                    const int kb = kb0 + q;
                    const uint32_t sa = smem_u32(tiles + stage * STAGE_BYTES + q * SUB_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    // the same layout choices as the producer's
                    const bool ta = MODE != MODE_SYRK && read_transposed(kb, tile.ti, 1);
                    const bool t0 = MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, 2 * tile.tj, 1));
                    const bool t1 = MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, 2 * tile.tj + 1, 1));
                    // one MMA over [n_lo, n_hi), or one per half when the halves'
                    // layouts differ and both are computed
                    const bool split = t0 != t1 && n_lo < BN / 2 && n_hi > BN / 2;
                    const int seg_lo[2] = {n_lo, BN / 2};
                    const int seg_hi[2] = {split ? BN / 2 : n_hi, n_hi};
                    const bool seg_t[2] = {n_lo >= BN / 2 ? t1 : t0, t1};
#pragma unroll
                    for (int sg = 0; sg < 2; ++sg) {
                        if (sg == 1 && !split) break;
                        const uint32_t idesc = instr_desc(BM, seg_hi[sg] - seg_lo[sg], ta, seg_t[sg]);
                        const uint32_t b_base = sb + static_cast<uint32_t>(seg_lo[sg]) * 128;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            tc_mma(d_tmem + static_cast<uint32_t>(seg_lo[sg]), operand_desc(sa, k, ta),
                                   operand_desc(b_base, k, seg_t[sg]), idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                }
                tc_commit(smem_u32(&empty_bar[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit(smem_u32(&tfull_bar[acc]));
        }
        // drain: all issued MMAs complete before TMEM is released
        tc_commit(smem_u32(drain_bar));
        wait_drain(smem_u32(drain_bar), 0);
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
        const int half = (warp - 2) >> 2;    // column half when two warps share a quarter
        const int ew = warp - 2;
        EpiBufs eb;
        for (int b = 0; b < NSLOT; ++b) {
            eb.ptr[b] = ebufs + (NSLOT * ew + b) * EBUF_BYTES;
            eb.buf[b] = smem_u32(eb.ptr[b]);
            eb.bar[b] = smem_u32(&ebar[NSLOT * ew + b]);
        }
        eb.phase = 0;
        eb.pending = 0;
        eb.seq = 0;
        int local = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
            const Tile tile = decode_tile<MODE>(p, t);
            const GroupParams& g = p.g[tile.group];
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            const int col_min = MODE == MODE_UPDATE ? 0 : tile.ti * BM;
            if (!epilogue_tile<MODE>(p, g, tile, col_min, tmem_base + static_cast<uint32_t>(acc * BN), quarter, half,
                                     lane, smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, eb))
                break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
        // drain: addend loads still in flight land, and the output stores
        // complete, before the CTA exits
        for (int b = 0; b < NSLOT; ++b)
            if (eb.pending & (1u << b)) wait_drain(eb.bar[b], (eb.phase >> b) & 1u);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant: tcgen05.mma.cta_group::2 on 256x256 pair tiles.  Each
// CTA of a 2-CTA cluster stages its own 128 rows of A and its own half (128
// rows) of B, 32 KB per 64-deep k-block, in three stages of two k-blocks
// each; the even CTA issues the MMAs,
// which read both CTAs' shared memory and write each CTA's 128 accumulator
// rows into that CTA's TMEM.  Both CTAs' operand loads complete on the even
// CTA's full barrier; its MMA commits arrive on both CTAs' empty and
// accumulator-full barriers; both CTAs' epilogue warps arrive on the even
// CTA's accumulator-empty barrier.  The epilogue is the single-CTA one.
// ---------------------------------------------------------------------------
constexpr int PKPS = 2;                          // k-blocks per stage (see KPS)
constexpr int PSTAGES = 6 / PKPS;
constexpr int PA_BYTES = BM * BK * 2;            // this CTA's 128 rows of A
constexpr int PB_BYTES = (BN / 2) * BK * 2;      // this CTA's half of B
constexpr int PSUB_BYTES = PA_BYTES + PB_BYTES;  // one k-block
constexpr int PSTAGE_BYTES = PKPS * PSUB_BYTES;
constexpr int PBAR_BYTES = 512;
constexpr int PSMEM_BYTES = 1024 + PSTAGES * PSTAGE_BYTES + EBUFS_BYTES + PBAR_BYTES;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Tensor load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the barrier at this offset in every CTA of `mask` once all
// prior MMAs of the pair have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Columns of a pair tile the MMA computes: 256, or for the last column tile
// of a ragged matrix the next multiple of 32 past the edge (of 128 with
// chunked maps, so each CTA's half starts on a 64-row chunk).  CTA r of the
// pair holds B columns [r * n / 2, (r + 1) * n / 2) of the tile.
__device__ __forceinline__ int pair_tile_n(const GroupParams& g, int tj) {
    const int rem = g.N - tj * BN;
    const int q = g.chunked ? 127 : 31;
    return rem < BN ? ((rem + q) & ~q) : BN;
}

template <int MODE>
__device__ __forceinline__ Tile decode_pair_tile(const NsParams& p, int t, int rank) {
    Tile out;
    int gi = 0;
    while (gi + 1 < p.num_groups && t >= p.g[gi + 1].tile_begin) ++gi;
    const GroupParams& g = p.g[gi];
    const int local = t - g.tile_begin;
    out.group = gi;
    out.mat = local / g.tiles_per_mat;
    int r = local - out.mat * g.tiles_per_mat;
    int I, J;
    if (MODE == MODE_UPDATE) {
        I = r / g.tiles_n;
        J = r - I * g.tiles_n;
    } else {
        // upper triangle of square 256x256 pair tiles: J >= I
        I = 0;
        for (;;) {
            const int cnt = g.tiles_n - I;
            if (r < cnt) break;
            r -= cnt;
            ++I;
        }
        J = I + r;
    }
    out.ti = 2 * I + rank;  // this CTA's 128-row tile
    out.tj = J;
    return out;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_gemm_pair_kernel(const __grid_constant__ NsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = smem;
    uint8_t* ebufs = smem + PSTAGES * PSTAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ebufs + EBUFS_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + PSTAGES;
    uint64_t* tfull_bar = bars + 2 * PSTAGES;
    uint64_t* tempty_bar = bars + 2 * PSTAGES + 2;
    uint64_t* drain_bar = bars + 2 * PSTAGES + 4;
    uint64_t* ebar = bars + 2 * PSTAGES + 5;  // NSLOT per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ebar + NSLOT * EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(drain_bar), 1);
        for (int i = 0; i < NSLOT * EPI_WARPS; ++i) mbar_init(smem_u32(&ebar[i]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        for (int gi = 0; gi < p.num_groups; ++gi) {
            tma_prefetch_desc(&p.g[gi].tm_a);
            tma_prefetch_desc(&p.g[gi].tm_b);
            if (MODE != MODE_SYRK) tma_prefetch_desc(&p.g[gi].tm_e);
            tma_prefetch_desc(&p.g[gi].tm_d);
            if (MODE != MODE_SYRK) tma_prefetch_desc(&p.g[gi].tm_t);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above touched only shared memory, TMEM and parameters
    pdl_wait_then_release();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int last_parity[PSTAGES];
        for (int s = 0; s < PSTAGES; ++s) last_parity[s] = -1;
        bool ok = true;
        for (int t = pair; ok && t < p.total_tiles; t += npairs) {
            const Tile tile = decode_pair_tile<MODE>(p, t, static_cast<int>(rank));
            const GroupParams& g = p.g[tile.group];
            const int nk = (g.K + BK - 1) / BK;
            for (int kb0 = 0; kb0 < nk; kb0 += PKPS) {
                if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full_bar[stage]);
                const uint32_t fb_leader = mapa_shared(fb, 0);
                const int b0 = tile.tj * BN + static_cast<int>(rank) * (pair_tile_n(g, tile.tj) / 2);
                const int nsub = nk - kb0 < PKPS ? nk - kb0 : PKPS;
                if (rank == 0) mbar_expect_tx(fb, 2 * PSUB_BYTES * nsub);
                auto load3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
                    tma_load_3d_pair(dst, map, c0, c1, c2, fb_leader);
                };
                auto load4 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3) {
                    tma_load_4d_pair(dst, map, c0, c1, c2, c3, fb_leader);
                };
                const bool chunked = g.chunked != 0;
                for (int q = 0; q < nsub; ++q) {
                    const int kb = kb0 + q;
                    const uint32_t sa = smem_u32(tiles + stage * PSTAGE_BYTES + q * PSUB_BYTES);
                    const uint32_t sb = sa + PA_BYTES;
                    // row blocks of 256 (the pair tile): both CTAs make the same choices
                    if (MODE != MODE_SYRK && read_transposed(kb, tile.ti >> 1, 2))
                        load_mn(sa, &g.tm_t, chunked, 2, tile.ti * BM, BM / 64, kb, tile.mat, load3, load4);
                    else
                        tma_load_3d_pair(sa, &g.tm_a, kb * BK, tile.ti * BM, tile.mat, fb_leader);
                    if (MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, tile.tj, 2)))
                        load_mn(sb, MODE == MODE_UPDATE ? &g.tm_b : &g.tm_t, chunked, 2, b0, BN / 2 / 64, kb, tile.mat,
                                load3, load4);
                    else
                        tma_load_3d_pair(sb, &g.tm_b, kb * BK, b0, tile.mat, fb_leader);
                }
                last_parity[stage] = static_cast<int>(phase);
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // drain: the even CTA's full barriers count both CTAs' copies
        if (rank == 0)
            for (int s = 0; s < PSTAGES; ++s)
                if (last_parity[s] >= 0) wait_drain(smem_u32(&full_bar[s]), static_cast<uint32_t>(last_parity[s]));
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------- MMA issuer (even CTA) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = pair; ok && t < p.total_tiles; t += npairs, ++local) {
            const Tile tile = decode_pair_tile<MODE>(p, t, 0);
            const GroupParams& g = p.g[tile.group];
            const int nk = (g.K + BK - 1) / BK;
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            if (!wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, abort_flag, p.status)) break;
            tc_fence_after();
            const int n = pair_tile_n(g, tile.tj);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb0 = 0; kb0 < nk; kb0 += PKPS) {
                if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nsub = nk - kb0 < PKPS ? nk - kb0 : PKPS;
                for (int q = 0; q < nsub; ++q) {
                    const int kb = kb0 + q;
                    const uint32_t sa = smem_u32(tiles + stage * PSTAGE_BYTES + q * PSUB_BYTES);
                    const uint32_t sb = sa + PA_BYTES;
                    const bool ta = MODE != MODE_SYRK && read_transposed(kb, tile.ti >> 1, 2);
                    const bool tb = MODE == MODE_UPDATE || (MODE == MODE_POLY && read_transposed(kb, tile.tj, 2));
                    const uint32_t idesc = instr_desc(2 * BM, n, ta, tb);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc_mma_pair(d_tmem, operand_desc(sa, k, ta), operand_desc(sb, k, tb), idesc,
                                    (kb | k) != 0 ? 1u : 0u);
                }
                tc_commit_pair_mc(smem_u32(&empty_bar[stage]), 0x3);
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit_pair_mc(smem_u32(&tfull_bar[acc]), 0x3);
        }
        // drain: every MMA of the pair completes before either CTA frees TMEM
        tc_commit_pair_mc(smem_u32(drain_bar), 0x1);
        wait_drain(smem_u32(drain_bar), 0);
    } else if (warp >= 2) {
        // ---------------- epilogue (both CTAs) ----------------
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int ew = warp - 2;
        EpiBufs eb;
        for (int b = 0; b < NSLOT; ++b) {
            eb.ptr[b] = ebufs + (NSLOT * ew + b) * EBUF_BYTES;
            eb.buf[b] = smem_u32(eb.ptr[b]);
            eb.bar[b] = smem_u32(&ebar[NSLOT * ew + b]);
        }
        eb.phase = 0;
        eb.pending = 0;
        eb.seq = 0;
        int local = 0;
        for (int t = pair; t < p.total_tiles; t += npairs, ++local) {
            const Tile tile = decode_pair_tile<MODE>(p, t, static_cast<int>(rank));
            const GroupParams& g = p.g[tile.group];
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            // SYRK/POLY store the pair tile whole: its row block is 256 rows
            const int col_min = MODE == MODE_UPDATE ? 0 : (tile.ti >> 1) * 2 * BM;
            if (!epilogue_tile<MODE>(p, g, tile, col_min, tmem_base + static_cast<uint32_t>(acc * BN), quarter, half,
                                     lane, smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, eb))
                break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
        }
        for (int b = 0; b < NSLOT; ++b)
            if (eb.pending & (1u << b)) wait_drain(eb.bar[b], (eb.phase >> b) & 1u);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncwarp();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Failure-detection self-check: one thread waits, through the kernels' own
// bounded wait, on an mbarrier nothing ever arrives on.  After limit_ns the
// wait records MUON_ERR_TIMEOUT in *status and the kernel returns.
// ---------------------------------------------------------------------------
__global__ void bounded_wait_probe_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    wait_bounded(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D bf16 tensor map over [count][rows][inner] with row stride ld elements
// and matrix stride `mat_stride` bytes.
bool make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t count, int64_t ld,
              int64_t mat_stride, uint32_t box_inner, uint32_t box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(count)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(mat_stride)};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D chunked view of the same matrices for MN-major reads: dims {64,
// rows, inner / 64, count} with strides {ld, 64 elements, matrix}, box {64,
// box_rows, box_chunks}.  `inner` must be a multiple of 64 so no chunk
// reaches past a row.
bool make_map_chunked(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t count, int64_t ld,
                      int64_t mat_stride, uint32_t box_rows, uint32_t box_chunks) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || inner % 64 != 0) return false;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(inner / 64),
                          static_cast<cuuint64_t>(count)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld * 2), 128, static_cast<cuuint64_t>(mat_stride)};
    cuuint32_t box[4] = {64, box_rows, box_chunks, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MN-major maps for a symmetric factor (2 chunks per copy) or X (UPDATE's
// B operand, `x_chunks` per copy): chunked when the width allows it.
bool make_mn_map(CUtensorMap* map, bool chunked, const void* base, int64_t inner, int64_t rows, int64_t count,
                 int64_t ld, int64_t mat_stride, uint32_t chunks) {
    return chunked ? make_map_chunked(map, base, inner, rows, count, ld, mat_stride, BK, chunks)
                   : make_map(map, base, inner, rows, count, ld, mat_stride, 64, BK);
}

constexpr CUtensorMapSwizzle kEpiSwizzle = EROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;

int triangle_tiles(int tiles_m, int tiles_n) {
    int n = 0;
    for (int ti = 0; ti < tiles_m; ++ti) n += tiles_n - (ti >> 1);
    return n;
}

int triangle_pair_tiles(int tiles_n) { return tiles_n * (tiles_n + 1) / 2; }

// Kernel attributes and the pair occupancy of one stage kernel, set up once
// per device (with that device current) and remembered.
template <int MODE, bool kPair>
cudaError_t stage_setup(int* max_pairs) {
    constexpr int kMaxDevices = 64;
    static std::mutex setup_mu;
    static bool setup_done[kMaxDevices] = {};
    static cudaError_t setup_err[kMaxDevices] = {};
    static int setup_pairs[kMaxDevices] = {};
    int dev = 0;
    const cudaError_t dev_err = cudaGetDevice(&dev);
    if (dev_err != cudaSuccess) return dev_err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(setup_mu);
    if (!setup_done[dev]) {
        cudaError_t e;
        int n = 0;
        if (kPair) {
            e = cudaFuncSetAttribute(ns_gemm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PSMEM_BYTES);
            if (e == cudaSuccess) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(2, 1, 1);
                cfg.blockDim = dim3(NUM_THREADS, 1, 1);
                cfg.dynamicSmemBytes = PSMEM_BYTES;
                e = cudaOccupancyMaxActiveClusters(&n, ns_gemm_pair_kernel<MODE>, &cfg);
            }
        } else {
            e = cudaFuncSetAttribute(ns_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMEM_BYTES);
        }
        setup_err[dev] = e;
        setup_pairs[dev] = n;
        setup_done[dev] = true;
    }
    *max_pairs = setup_pairs[dev];
    return setup_err[dev];
}

template <int MODE, bool kPair>
cudaError_t launch_stage(const NsGroup* groups, int ngroups, int cur, bool first, float a, float b, float c,
                         int* status, int num_sms, cudaStream_t st) {
    int max_pairs = 0;
    const cudaError_t attr_err = stage_setup<MODE, kPair>(&max_pairs);
    if (attr_err != cudaSuccess) return attr_err;

    NsParams prm;
    memset(&prm, 0, sizeof prm);
    int tiles = 0;
    for (int i = 0; i < ngroups; ++i) {
        const NsGroup& G = groups[i];
        GroupParams& g = prm.g[i];
        const uint16_t* X = G.X[cur];
        bool ok = true;
        const bool chunked = G.mp % 64 == 0 && G.np % 64 == 0;
        g.chunked = chunked ? 1 : 0;
        if (MODE == MODE_SYRK) {
            ok &= make_map(&g.tm_a, X, G.np, G.mp, G.count, G.ldx, G.x_stride, BK, BM);
            ok &= make_map(&g.tm_b, X, G.np, G.mp, G.count, G.ldx, G.x_stride, BK, kPair ? BN / 2 : BN);
            ok &= make_map(&g.tm_d, G.A, G.mp, G.mp, G.count, G.lda, G.g_stride, EPI_COLS, 32, kEpiSwizzle);
            g.M = static_cast<int32_t>(G.mp);
            g.N = static_cast<int32_t>(G.mp);
            g.K = static_cast<int32_t>(G.np);
        } else if (MODE == MODE_POLY) {
            ok &= make_map(&g.tm_a, G.A, G.mp, G.mp, G.count, G.lda, G.g_stride, BK, BM);
            ok &= make_map(&g.tm_b, G.A, G.mp, G.mp, G.count, G.lda, G.g_stride, BK, kPair ? BN / 2 : BN);
            ok &= make_mn_map(&g.tm_t, chunked, G.A, G.mp, G.mp, G.count, G.lda, G.g_stride, 2);
            ok &= make_map(&g.tm_e, G.A, G.mp, G.mp, G.count, G.lda, G.g_stride, EPI_COLS, 32, kEpiSwizzle);
            ok &= make_map(&g.tm_d, G.B, G.mp, G.mp, G.count, G.lda, G.g_stride, EPI_COLS, 32, kEpiSwizzle);
            g.M = static_cast<int32_t>(G.mp);
            g.N = static_cast<int32_t>(G.mp);
            g.K = static_cast<int32_t>(G.mp);
        } else {
            ok &= make_map(&g.tm_a, G.B, G.mp, G.mp, G.count, G.lda, G.g_stride, BK, BM);
            ok &= make_mn_map(&g.tm_t, chunked, G.B, G.mp, G.mp, G.count, G.lda, G.g_stride, 2);
            ok &= make_mn_map(&g.tm_b, chunked, X, G.np, G.mp, G.count, G.ldx, G.x_stride, kPair ? 2 : 4);
            ok &= make_map(&g.tm_e, X, G.np, G.mp, G.count, G.ldx, G.x_stride, EPI_COLS, 32, kEpiSwizzle);
            ok &= make_map(&g.tm_d, G.X[cur ^ 1], G.np, G.mp, G.count, G.ldx, G.x_stride, EPI_COLS, 32, kEpiSwizzle);
            g.M = static_cast<int32_t>(G.mp);
            g.N = static_cast<int32_t>(G.np);
            g.K = static_cast<int32_t>(G.mp);
        }
        if (!ok) return cudaErrorInvalidValue;
        g.scale = (first && MODE != MODE_POLY) ? G.scale : nullptr;
        g.scale_stride = G.scale_stride;
        g.count = static_cast<int32_t>(G.count);
        g.tiles_n = (g.N + BN - 1) / BN;
        if (kPair) {
            const int pairs_m = (g.M + 2 * BM - 1) / (2 * BM);
            g.tiles_per_mat = (MODE == MODE_UPDATE) ? pairs_m * g.tiles_n : triangle_pair_tiles(g.tiles_n);
        } else {
            const int tiles_m = (g.M + BM - 1) / BM;
            g.tiles_per_mat = (MODE == MODE_UPDATE) ? tiles_m * g.tiles_n : triangle_tiles(tiles_m, g.tiles_n);
        }
        g.tile_begin = tiles;
        tiles += g.tiles_per_mat * g.count;
    }
    prm.num_groups = ngroups;
    prm.total_tiles = tiles;
    prm.status = status;
    if (MODE == MODE_POLY) {
        prm.alpha = b;
        prm.beta = c;
    } else if (MODE == MODE_UPDATE) {
        prm.alpha = a;
        prm.beta = 1.f;
    } else {
        prm.alpha = 0.f;
        prm.beta = 1.f;
    }
    if (tiles == 0) return cudaSuccess;
    constexpr int kind = MODE == MODE_SYRK ? MUON_KERNEL_NS_SYRK
                         : MODE == MODE_POLY ? MUON_KERNEL_NS_POLY : MUON_KERNEL_NS_UPDATE;
    launch_begin(kind, st);
    cudaError_t e;
    if (kPair) {
        int pairs = max_pairs > 0 ? max_pairs : num_sms / 2;
        if (tiles < pairs) pairs = tiles;
        e = launch_pdl(ns_gemm_pair_kernel<MODE>, dim3(2 * pairs), dim3(NUM_THREADS), PSMEM_BYTES, st, prm);
    } else {
        const int grid = tiles < num_sms ? tiles : num_sms;
        e = launch_pdl(ns_gemm_kernel<MODE>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, prm);
    }
    launch_end(kind, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

// Whether a shape group runs on CTA pairs (all three stages).  Pairs halve
// each SM's operand traffic and deepen the pipeline (measured 2% faster on
// 2048-row matrices, 11% on 7168-row ones), but compute the padded rows of
// a part-empty last pair row.  A group takes pairs when those are at most
// 1/8 of its rows.  With two k-blocks per pair-ring stage this includes
// the 1408-row MoE experts (9% padded rows) in every stage: their UPDATE
// on pairs measured 1.7% faster than on single CTAs.  Up to 512 rows single
// CTAs win (NS on 1200 matrices of 512 x 1024 14% faster, a lone 256 x 512
// step 11% faster: no cluster launch or cross-CTA handshakes for one or two
// row tiles); at 768 rows the two are level, at 1024 pairs lead by 6%.
bool use_pairs(const NsGroup& g) {
    if (g.mp <= 4 * BM) return false;
    const int64_t padded = (g.mp + 2 * BM - 1) / (2 * BM) * (2 * BM);
    return (padded - g.mp) * 8 <= g.mp;
}

template <int MODE>
cudaError_t run_stage(const NsGroup* pair_groups, int npair, const NsGroup* single_groups, int nsingle, int cur,
                      bool first, float a, float b, float c, int* status, int num_sms, cudaStream_t st) {
    for (int off = 0; off < npair; off += kNsMaxGroups) {
        const int n = npair - off < kNsMaxGroups ? npair - off : kNsMaxGroups;
        cudaError_t e = launch_stage<MODE, true>(pair_groups + off, n, cur, first, a, b, c, status, num_sms, st);
        if (e != cudaSuccess) return e;
    }
    for (int off = 0; off < nsingle; off += kNsMaxGroups) {
        const int n = nsingle - off < kNsMaxGroups ? nsingle - off : kNsMaxGroups;
        cudaError_t e = launch_stage<MODE, false>(single_groups + off, n, cur, first, a, b, c, status, num_sms, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_wait_probe(int* status, long long limit_ns, cudaStream_t st) {
    bounded_wait_probe_kernel<<<1, 32, 0, st>>>(status, static_cast<unsigned long long>(limit_ns));
    return cudaGetLastError();
}

cudaError_t ns_run(const NsGroup* groups, int ngroups, int steps, const float* coeffs, int* status, int num_sms,
                   cudaStream_t st) {
    std::vector<NsGroup> pairs, singles;
    for (int i = 0; i < ngroups; ++i) (use_pairs(groups[i]) ? pairs : singles).push_back(groups[i]);
    const int np = static_cast<int>(pairs.size()), ns = static_cast<int>(singles.size());
    for (int s = 0; s < steps; ++s) {
        const int cur = s & 1;
        const float a = coeffs[3 * s], b = coeffs[3 * s + 1], c = coeffs[3 * s + 2];
        const bool first = s == 0;
        cudaError_t e =
            run_stage<MODE_SYRK>(pairs.data(), np, singles.data(), ns, cur, first, a, b, c, status, num_sms, st);
        if (e == cudaSuccess)
            e = run_stage<MODE_POLY>(pairs.data(), np, singles.data(), ns, cur, first, a, b, c, status, num_sms, st);
        if (e == cudaSuccess)
            e = run_stage<MODE_UPDATE>(pairs.data(), np, singles.data(), ns, cur, first, a, b, c, status, num_sms,
                                       st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t ns_prepare_device() {
    int n = 0;
    cudaError_t e = stage_setup<MODE_SYRK, true>(&n);
    if (e == cudaSuccess) e = stage_setup<MODE_POLY, true>(&n);
    if (e == cudaSuccess) e = stage_setup<MODE_UPDATE, true>(&n);
    if (e == cudaSuccess) e = stage_setup<MODE_SYRK, false>(&n);
    if (e == cudaSuccess) e = stage_setup<MODE_POLY, false>(&n);
    if (e == cudaSuccess) e = stage_setup<MODE_UPDATE, false>(&n);
    return e;
}

}  // namespace muon
