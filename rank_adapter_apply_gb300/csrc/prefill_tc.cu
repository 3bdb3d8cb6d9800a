// Segmented prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// A prefill batch holds long runs of consecutive tokens that all use one slot
// (a sequence's prompt under one adapter; per-batch slots as on the
// "Multi-LoRA 适配器缓存生产实战" page, section 核心原理). For such a run the
// delta is a real dense contraction,
//
//   V = X_tile · A_s^T            (128 tokens x d_in) x (d_in x R)  -> fp32
//   Y_tile += scale_s · V · B_s^T  (128 x R) x (R x d_out),
//
// with scale_s = lora_alpha / r (the PEFT fields r and lora_alpha, "vLLM
// LoRA Resolver 插件详解" page, section 3.2). Slot pools are zero-padded to
// R = max_lora_rank, so the padded ranks contribute exact zeros.
//
// Two kernels per call, both HBM-bound:
//
// prefill_shrink_kernel  one CTA per (tile, input group, d_in chunk). An input
//   group is the set of layers of the call that read the same x (q/k/v, or
//   gate/up), so each x tile crosses HBM once for all of them. A TMA producer
//   warp streams 64-column k-blocks of x and of every A_s of the group through
//   a shared-memory ring; one thread issues tcgen05.mma (M 128, N R, K 16) into
//   one TMEM accumulator per layer; four epilogue warps write the fp32 partial
//   V of their rows to the workspace (chunk c of layer l at rows c*T + t).
//
// prefill_expand_kernel  persistent, one CTA per SM. The work items are
//   (layer, tile, 256-column block of d_out), split into contiguous ranges.
//   The V-loader warps sum the partials of V in a fixed order and write V as
//   bf16 high + low parts (double-buffered across tiles) into swizzled
//   shared memory, or at rank 64 into tensor memory (which leaves the shared
//   memory for one more ring stage), the producer streams y and B_s n-blocks
//   through the ring, one thread issues the expand MMAs (M 128, N 128, K R,
//   twice: high and low parts) into rotating TMEM accumulators, and the
//   epilogue computes
//   y = round(y + scale * D) in place in the ring and stores full tiles back
//   with a TMA store (ragged tiles with plain row stores, so that no row of a
//   neighbouring run is touched).
//
// Every mbarrier wait is bounded; a wait that gives up sets the workspace
// error word, the CTA stops issuing work, drains the copies and MMAs it has in
// flight, frees its TMEM and returns.
#include "device_util.cuh"
#include "kernels.cuh"
#include "tc_util.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_bf16.h>

namespace lora {
namespace {

constexpr int kThreads = 192;              // shrink: warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kExpandThreads = 448;        // expand: warp 0 TMA, 1 MMA, 2..5 V loaders, 6..13 epilogue
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kVThreads = 128;
constexpr int kTileBytes = 16384;          // 128 rows x 64 bf16: one x k-block or one y n-block
constexpr int kColBlock = 256;             // d_out columns per expand work item
constexpr int kNB = 128;                   // d_out columns per expand n-block (two 64-column y boxes)
constexpr int kAcc = 2;                    // expand accumulators (kNB TMEM columns each)
constexpr int kMaxStages = 8;
constexpr int kMaxJobs = 64;
constexpr uint32_t kWaitLimit = 1u << 22;

// Wait for a phase unless an earlier wait of this CTA already gave up.
__device__ __forceinline__ bool wait_ok(uint64_t *bar, uint32_t parity, volatile int *flag) {
    if (*flag) return false;
    if (mbar_wait_bounded(bar, parity, kWaitLimit)) return true;
    *flag = 1;
    return false;
}

__host__ __device__ inline uint32_t tmem_cols_for(int cols) {
    uint32_t c = 32;
    while ((int)c < cols) c <<= 1;
    return c;
}

// Where the expand keeps V. In tensor memory its 32 KB of shared memory at
// rank 64 become a fourth ring stage (3 -> 4: mixed-rank step 316 -> 300 us);
// at rank 32 the fifth stage that it would allow was measured slower than
// four (346 against 335 us per prefill step) and an MMA reading A from tensor
// memory slightly slower than one reading shared memory (337 us at four
// stages), so lower ranks keep V in shared memory.
__host__ __device__ constexpr bool expand_v_in_tmem(int R) { return R == 64; }

// Shared-memory descriptor of the B operand for 16-rank K step kk of a stage
// whose B part (at ba) holds the pool's rank blocks of kBK ranks, each a box
// of 128 rows x kBK bf16 with the swizzle of its row width.
template <int R>
__device__ __forceinline__ uint64_t bdesc(uint32_t ba, int kk) {
    constexpr int kBK = b_block(R);
    constexpr uint32_t kBBox = 128 * kBK * 2;
    constexpr uint32_t kSwzB = kBK == 32 ? tc::kSwz64 : tc::kSwz32;
    return tc::smem_desc(ba + (uint32_t)(kk / (kBK / 16)) * kBBox + (uint32_t)(kk % (kBK / 16)) * 32, 2 * kBK, kSwzB);
}

// Row i of a K-major operand of R bf16 per row, in the swizzle the TMA and
// the MMA descriptors use for that row width: 16-byte chunk c of the row goes
// to chunk c ^ f(i).
template <int R>
__device__ __forceinline__ int swz_chunk(int c, int i) {
    if constexpr (R == 64) return c ^ (i & 7);
    else if constexpr (R == 32) return c ^ ((i >> 1) & 3);
    else return c ^ ((i >> 2) & 1);
}

template <int R>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[R]) {
    if constexpr (R == 16) {
        uint32_t r[16];
        tc::tmem_ld16_sync(taddr, r);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
    } else {
#pragma unroll
        for (int c = 0; c < R / 32; ++c) {
            uint32_t r[32];
            tc::tmem_ld32_sync(taddr + 32 * c, r);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[32 * c + k] = __uint_as_float(r[k]);
        }
    }
}

// ============================================================================
// Shrink
// ============================================================================

struct ShrinkJob {
    int group, chunk, kb0, kb1;               // k-blocks [kb0, kb1) of d_in
};

struct ShrinkArgs {
    CUtensorMap mx[kMaxLayersPerCall];        // per group: x [T][d_in], box 64 x 128
    CUtensorMap mx32[kMaxLayersPerCall];      // the same x, box 64 x 32 (ragged tiles)
    CUtensorMap ma[kMaxLayersPerCall];        // per member (group order): A pool [S*R][d_in], box 64 x R
    float *part[kMaxLayersPerCall];           // per member
    int g_first[kMaxLayersPerCall], g_count[kMaxLayersPerCall];
    ShrinkJob jobs[kMaxJobs];
    const int4 *ptiles;
    int *hdr;
    int T, ring_bytes, tmem_cols;             // ring_bytes: this launch's shared ring (every group fits two stages)
};

// Sum of the d_in chunks of V, in chunk order, left in chunk 0: one CTA per
// (layer of the call, block of 256 / (R/4) rows of a tile), one 16-byte column
// of one row per thread.
struct ReduceArgs {
    float *part[kMaxLayersPerCall];
    int nch[kMaxLayersPerCall];
    const int4 *ptiles;
    const int *hdr;
    int T, R;
};

__global__ void __launch_bounds__(256)
prefill_reduce_kernel(const __grid_constant__ ReduceArgs a) {
    grid_dependency_wait();                 // the shrink's partials
    grid_launch_dependents();
    const int R4 = a.R / 4, rows_per_cta = 256 / R4, blocks = kPrefillRows / rows_per_cta;
    const int p = blockIdx.x / blocks, rb = blockIdx.x % blocks, l = blockIdx.y;
    if (p >= a.hdr[kHdrPrefillTiles] || a.nch[l] < 2) return;
    const int4 pt = a.ptiles[p];
    const int nch = a.nch[l];
    float4 *base = reinterpret_cast<float4 *>(a.part[l]) + (size_t)pt.y * R4;
    const size_t cs = (size_t)a.T * R4;
    const int e = rb * rows_per_cta * R4 + threadIdx.x;
    if (e < pt.z * R4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int c = 0;
        for (; c + 4 <= nch; c += 4) {
            float4 f[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) f[u] = __ldcg(base + (c + u) * cs + e);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc.x += f[u].x;
                acc.y += f[u].y;
                acc.z += f[u].z;
                acc.w += f[u].w;
            }
        }
        for (; c < nch; ++c) {
            const float4 f = __ldcg(base + c * cs + e);
            acc.x += f.x;
            acc.y += f.y;
            acc.z += f.z;
            acc.w += f.w;
        }
        base[e] = acc;
    }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 3)
prefill_shrink_kernel(const __grid_constant__ ShrinkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kMaxStages], empty[kMaxStages], acc_full, drained;
    __shared__ uint32_t tmem_base;
    __shared__ int error;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dependency_wait();                 // the tile list of the grouping kernel
    grid_launch_dependents();
    if ((int)blockIdx.x >= a.hdr[kHdrPrefillTiles]) return;
    const int4 pt = a.ptiles[blockIdx.x];
    const int s = pt.x, row0 = pt.y, rows = pt.z;
    const ShrinkJob job = a.jobs[blockIdx.y];
    const int g = job.group, nl = a.g_count[g], m0 = a.g_first[g];
    const uint32_t stage_bytes = kTileBytes + (uint32_t)nl * R * 128;
    // As many stages as this group's stage size fits in the ring (a group with
    // fewer layers has smaller stages and keeps more loads in flight).
    int stages = (int)((uint32_t)a.ring_bytes / stage_bytes);
    stages = stages > kMaxStages ? kMaxStages : stages;

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&drained, 1);
        error = 0;
        fence_mbar_init();
        tc::prefetch_tensormap(&a.mx[g]);
        tc::prefetch_tensormap(&a.mx32[g]);
        for (int l = 0; l < nl; ++l) tc::prefetch_tensormap(&a.ma[m0 + l]);
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_base, (uint32_t)a.tmem_cols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    volatile int *err = &error;
    const int nkb = job.kb1 - job.kb0;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer ----------------
            // A ragged tile (the last of a run) reads only the 32-row boxes
            // that hold its rows; the MMA rows past them are never stored.
            const int nx = rows >= kPrefillRows ? 0 : (rows + 31) >> 5;
            const uint32_t xbytes = nx ? (uint32_t)nx * 4096u : (uint32_t)kTileBytes;
            int issued = 0;
            for (int j = 0; j < nkb; ++j) {
                const int st = j % stages;
                if (!wait_ok(&empty[st], ((uint32_t)(j / stages) & 1u) ^ 1u, err)) break;
                uint8_t *tile = base + (size_t)st * stage_bytes;
                const int col = (job.kb0 + j) * 64;
                mbar_arrive_expect_tx(&full[st], stage_bytes - kTileBytes + xbytes);
                if (nx)
                    for (int q = 0; q < nx; ++q) tc::tma_load_2d(tile + q * 4096, &a.mx32[g], col, row0 + 32 * q, &full[st]);
                else
                    tc::tma_load_2d(tile, &a.mx[g], col, row0, &full[st]);
                for (int l = 0; l < nl; ++l)
                    tc::tma_load_2d(tile + kTileBytes + l * R * 128, &a.ma[m0 + l], col, s * R, &full[st]);
                issued = j + 1;
            }
            // Drain: the last loads issued must have landed before the CTA exits.
            for (int j = issued - stages < 0 ? 0 : issued - stages; j < issued; ++j)
                mbar_wait_bounded(&full[j % stages], (uint32_t)(j / stages) & 1u, kWaitLimit);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = tc::idesc_bf16(128, R);
            for (int j = 0; j < nkb; ++j) {
                const int st = j % stages;
                if (!wait_ok(&full[st], (uint32_t)(j / stages) & 1u, err)) break;
                tc::fence_after_sync();
                const uint32_t xa = smem_u32(base + (size_t)st * stage_bytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    for (int l = 0; l < nl; ++l)
                        tc::mma_bf16(tmem + (uint32_t)(l * R),
                                     tc::smem_desc(xa + k * 32, 128, tc::kSwz128),
                                     tc::smem_desc(xa + kTileBytes + l * R * 128 + k * 32, 128, tc::kSwz128),
                                     idesc, (j | k) != 0);
                tc::mma_commit(&empty[st]);
            }
            tc::mma_commit(&acc_full);
            tc::mma_commit(&drained);
            mbar_wait_bounded(&drained, 0, kWaitLimit);      // every MMA done before TMEM is freed
        }
    } else {
        // ---------------- epilogue: row i of the tile ----------------
        const int q = warp & 3;
        const int i = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const bool ok = wait_ok(&acc_full, 0, err);
        __syncwarp();
        tc::fence_after_sync();
        if (__all_sync(0xffffffffu, ok)) {
            for (int l = 0; l < nl; ++l) {
                float v[R];
                tmem_ld_row<R>(tmem + lane_addr + (uint32_t)(l * R), v);
                if (i < rows) {
                    float4 *dst = reinterpret_cast<float4 *>(a.part[m0 + l] +
                                                             ((size_t)job.chunk * a.T + row0 + i) * R);
#pragma unroll
                    for (int k = 0; k < R / 4; ++k)
                        dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (error && tid == 0) atomicExch(a.hdr + kHdrError, 1);
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
    }
}

// ============================================================================
// Expand
// ============================================================================

struct ExpandArgs {
    CUtensorMap my[kMaxLayersPerCall];        // y [T][d_out], box 64 x 128, 128-byte swizzle (loads)
    CUtensorMap ms[kMaxLayersPerCall];        // the same y, box 64 x 32 (one row quarter's store)
    CUtensorMap mb[kMaxLayersPerCall];        // B pool as [S*(R/kb)*d_out][kb] (rank blocks), box kb x 128
    const float *part[kMaxLayersPerCall];
    uint16_t *y[kMaxLayersPerCall];
    int d_out[kMaxLayersPerCall], ncb[kMaxLayersPerCall], nch[kMaxLayersPerCall];
    const int4 *ptiles;
    int *hdr;
    const float *scale;
    int n, T, stages, sum_ncb, S;
};

struct Item {
    int l, p, cb;
};

// Work item k: layers one after another, within a layer tiles, within a tile
// column blocks (so consecutive items of one CTA share the tile's V).
__device__ __forceinline__ Item item_at(const ExpandArgs &a, int k, int np) {
    int l = 0;
    while (l < a.n - 1 && k >= np * a.ncb[l]) {
        k -= np * a.ncb[l];
        ++l;
    }
    return Item{l, k / a.ncb[l], k % a.ncb[l]};
}

__device__ __forceinline__ int n_blocks(const ExpandArgs &a, const Item &it) {
    const int left = (a.d_out[it.l] - it.cb * kColBlock + kNB - 1) / kNB;
    return left < kColBlock / kNB ? left : kColBlock / kNB;
}

template <int R>
__global__ void __launch_bounds__(kExpandThreads, 1)
prefill_expand_kernel(const __grid_constant__ ExpandArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ uint64_t acc_full[kAcc], acc_empty[kAcc], v_full[2], v_empty[2], drained;
    __shared__ float sscale[kMaxSlots];
    __shared__ uint32_t tmem_base;
    __shared__ int error;

    constexpr int W = R * 2;                                   // bytes per V / B row
    constexpr uint32_t kSwzRank = R == 64 ? tc::kSwz128 : (R == 32 ? tc::kSwz64 : tc::kSwz32);
    constexpr uint32_t kStage = 2 * kTileBytes + kNB * W;       // y boxes [2][128][64], B [R / kBK][128][kBK]
    constexpr int kBK = b_block(R);                             // ranks per B block of the pool
    constexpr uint32_t kBBox = kNB * kBK * 2;                   // one block's box: 128 rows
    constexpr uint32_t kVBytes = 128 * W;
    // V in tensor memory (rank 64): after the kAcc accumulators of kNB
    // columns, [2 buffers][hi, lo] of R / 2 columns each (two bf16 per column)
    constexpr bool kVTmem = expand_v_in_tmem(R);
    constexpr uint32_t kVCol = kNB * kAcc, kTmemCols = kVTmem ? 512 : kNB * kAcc;
    static_assert(!kVTmem || kVCol + 2 * R <= kTmemCols, "V fits in the allocation");
    const int stages = a.stages;
    uint8_t *ring = base;
    uint8_t *vbuf = base + (size_t)stages * kStage;            // [2][hi, lo] (V in shared memory)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dependency_wait();                 // the partials of V (shrink, chunk sums)
    grid_launch_dependents();
    const int np = a.hdr[kHdrPrefillTiles];
    const long long total = (long long)np * a.sum_ncb;
    const int k0 = (int)(total * blockIdx.x / gridDim.x);
    const int k1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
    if (k0 >= k1) return;

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kEpiWarps);     // every epilogue warp, once its rows are stored
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&v_full[i], kVThreads);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(&drained, 1);
        error = 0;
        fence_mbar_init();
        for (int l = 0; l < a.n; ++l) {
            tc::prefetch_tensormap(&a.my[l]);
            tc::prefetch_tensormap(&a.ms[l]);
            tc::prefetch_tensormap(&a.mb[l]);
        }
    }
    for (int x = tid; x < a.S; x += kExpandThreads) sscale[x] = a.scale[x];
    if (warp == 1) {
        tc::tmem_alloc(&tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    volatile int *err = &error;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: y and B n-blocks ----------------
            int j = 0;
            for (int k = k0; k < k1 && !*err; ++k) {
                const Item it = item_at(a, k, np);
                const int4 pt = a.ptiles[it.p];
                const int nb = n_blocks(a, it), d_out = a.d_out[it.l];
                // a ragged tile reads only the 32-row boxes of y that hold its rows
                const int ny = pt.z >= kPrefillRows ? 0 : (pt.z + 31) >> 5;
                const uint32_t ybytes = ny ? 2u * (uint32_t)ny * 4096u : 2u * (uint32_t)kTileBytes;
                for (int b = 0; b < nb; ++b) {
                    const int st = j % stages;
                    if (!wait_ok(&empty[st], ((uint32_t)(j / stages) & 1u) ^ 1u, err)) break;
                    uint8_t *tile = ring + (size_t)st * kStage;
                    const int col = it.cb * kColBlock + b * kNB;
                    // B: the rank blocks the tile's slot has (the pool holds B in
                    // blocks of kBK ranks, each [d_out][kBK])
                    const int nblk = kBK == R ? 1 : (pt.w + kBK - 1) / kBK;
                    mbar_arrive_expect_tx(&full[st], (uint32_t)nblk * kBBox + ybytes);
                    if (ny) {
                        for (int q = 0; q < ny; ++q) {
                            tc::tma_load_2d(tile + q * 4096, &a.ms[it.l], col, pt.y + 32 * q, &full[st]);
                            tc::tma_load_2d(tile + kTileBytes + q * 4096, &a.ms[it.l], col + 64, pt.y + 32 * q,
                                            &full[st]);
                        }
                    } else {
                        tc::tma_load_2d(tile, &a.my[it.l], col, pt.y, &full[st]);
                        tc::tma_load_2d(tile + kTileBytes, &a.my[it.l], col + 64, pt.y, &full[st]);
                    }
                    for (int kb = 0; kb < nblk; ++kb)
                        tc::tma_load_2d(tile + 2 * kTileBytes + kb * kBBox, &a.mb[it.l], 0,
                                        (pt.x * (R / kBK) + kb) * d_out + col, &full[st]);
                    ++j;
                }
            }
            for (int i = j - stages < 0 ? 0 : j - stages; i < j; ++i)
                mbar_wait_bounded(&full[i % stages], (uint32_t)(i / stages) & 1u, kWaitLimit);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = tc::idesc_bf16(128, kNB);
            int j = 0, gen = -1, pl = -1, pp = -1, nkb = R / 16;
            for (int k = k0; k < k1 && !*err; ++k) {
                const Item it = item_at(a, k, np);
                if (it.l != pl || it.p != pp) {
                    ++gen;
                    pl = it.l;
                    // the slot's 16-rank MMA steps (its rank from the tile
                    // list, loaded while the wait for this tile's V runs)
                    // (up to rank 32 the pool's one block holds every rank: all steps)
                    if (kBK < R && it.p != pp) nkb = (a.ptiles[it.p].w + 15) >> 4;
                    pp = it.p;
                    if (!wait_ok(&v_full[gen & 1], (uint32_t)(gen >> 1) & 1u, err)) break;
                    tc::fence_after_sync();
                }
                // V: tensor-memory columns, or shared-memory addresses
                const uint32_t vh = kVTmem ? tmem + kVCol + (uint32_t)(gen & 1) * R
                                           : smem_u32(vbuf + (size_t)(gen & 1) * 2 * kVBytes);
                const uint32_t vl = kVTmem ? vh + R / 2 : vh + kVBytes;
                const int nb = n_blocks(a, it);
                for (int b = 0; b < nb; ++b) {
                    const int st = j % stages, ac = j % kAcc;
                    if (!wait_ok(&full[st], (uint32_t)(j / stages) & 1u, err)) break;
                    if (!wait_ok(&acc_empty[ac], ((uint32_t)(j / kAcc) & 1u) ^ 1u, err)) break;
                    tc::fence_after_sync();
                    const uint32_t ba = smem_u32(ring + (size_t)st * kStage + 2 * kTileBytes);
                    const uint32_t d = tmem + (uint32_t)kNB * ac;
                    // B for K step kk: block kk / (kBK / 16) of [128 rows][kBK ranks]
                    // (rows of 2 kBK bytes, swizzled across them), 32 bytes in; V
                    // columns past the slot's rank are zero, so steps past nkb
                    // (their blocks possibly not loaded) are skipped
                    if constexpr (kVTmem) {
#pragma unroll
                        for (int kk = 0; kk < R / 16; ++kk)
                            if (kk < nkb)
                                tc::mma_bf16_tmem_a(d, vh + kk * 8, bdesc<R>(ba, kk),
                                                    idesc, kk != 0);
#pragma unroll
                        for (int kk = 0; kk < R / 16; ++kk)
                            if (kk < nkb)
                                tc::mma_bf16_tmem_a(d, vl + kk * 8, bdesc<R>(ba, kk),
                                                    idesc, 1);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < R / 16; ++kk)
                            if (kk < nkb)
                                tc::mma_bf16(d, tc::smem_desc(vh + kk * 32, W, kSwzRank),
                                             bdesc<R>(ba, kk), idesc, kk != 0);
#pragma unroll
                        for (int kk = 0; kk < R / 16; ++kk)
                            if (kk < nkb)
                                tc::mma_bf16(d, tc::smem_desc(vl + kk * 32, W, kSwzRank),
                                             bdesc<R>(ba, kk), idesc, 1);
                    }
                    tc::mma_commit(&acc_full[ac]);
                    ++j;
                }
                bool last_use = k + 1 >= k1;
                if (!last_use) {
                    const Item nx = item_at(a, k + 1, np);
                    last_use = nx.l != it.l || nx.p != it.p;
                }
                if (last_use) tc::mma_commit(&v_empty[gen & 1]);
            }
            tc::mma_commit(&drained);
            mbar_wait_bounded(&drained, 0, kWaitLimit);
        }
    } else if (warp < 6) {
        // ---------------- V loaders: row i of the tile ----------------
        // (V in tensor memory: a warp reaches the lanes 32 (warp % 4) ..
        // 32 (warp % 4) + 31)
        const int i = kVTmem ? (warp & 3) * 32 + lane : tid - 64;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        int gen = -1, pl = -1, pp = -1;
        for (int k = k0; k < k1; ++k) {
            const Item it = item_at(a, k, np);
            if (it.l == pl && it.p == pp) continue;
            ++gen;
            pl = it.l;
            pp = it.p;
            const int vb = gen & 1;
            if constexpr (kVTmem) {
                // (warp-uniform: the TMEM stores below are issued by whole warps)
                if (!__all_sync(0xffffffffu, wait_ok(&v_empty[vb], ((uint32_t)(gen >> 1) & 1u) ^ 1u, err))) break;
                tc::fence_after_sync();
            } else {
                if (!wait_ok(&v_empty[vb], ((uint32_t)(gen >> 1) & 1u) ^ 1u, err)) break;
            }
            const int4 pt = a.ptiles[it.p];
            const uint32_t vth = tmem + lane_addr + kVCol + (uint32_t)vb * R, vtl = vth + R / 2;
            uint8_t *vh = vbuf + (size_t)vb * 2 * kVBytes;
            uint8_t *vl = vh + kVBytes;
            float v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = 0.f;
            if (i < pt.z) {
                // Partials in chunk order (fixed summation order); two chunks'
                // loads are in flight together where registers allow.
                constexpr int kPair = R <= 32 ? 2 : 1;
                const int nch = a.nch[it.l];
                const float4 *src = reinterpret_cast<const float4 *>(a.part[it.l] + ((size_t)pt.y + i) * R);
                const size_t cstride = (size_t)a.T * R / 4;
                int c = 0;
                for (; c + kPair <= nch; c += kPair) {
                    float4 f[kPair][R / 4];
#pragma unroll
                    for (int u = 0; u < kPair; ++u)
#pragma unroll
                        for (int r = 0; r < R / 4; ++r) f[u][r] = src[(c + u) * cstride + r];
#pragma unroll
                    for (int u = 0; u < kPair; ++u)
#pragma unroll
                        for (int r = 0; r < R / 4; ++r) {
                            v[4 * r] += f[u][r].x;
                            v[4 * r + 1] += f[u][r].y;
                            v[4 * r + 2] += f[u][r].z;
                            v[4 * r + 3] += f[u][r].w;
                        }
                }
                for (; c < nch; ++c) {
#pragma unroll
                    for (int r = 0; r < R / 4; ++r) {
                        const float4 f = src[c * cstride + r];
                        v[4 * r] += f.x;
                        v[4 * r + 1] += f.y;
                        v[4 * r + 2] += f.z;
                        v[4 * r + 3] += f.w;
                    }
                }
            }
            if constexpr (kVTmem) {
                // 16 ranks (eight tensor-memory columns) of each part at a time
#pragma unroll
                for (int c = 0; c < R / 16; ++c) {
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x0 = v[16 * c + 2 * e], x1 = v[16 * c + 2 * e + 1];
                        const float h0 = round_bf16(x0), h1 = round_bf16(x1);
                        hw[e] = pack_bf16(h0, h1);
                        lw[e] = pack_bf16(x0 - h0, x1 - h1);
                    }
                    tc::tmem_st8(vth + 8 * c, hw);
                    tc::tmem_st8(vtl + 8 * c, lw);
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();
            } else {
                // one swizzled 16-byte chunk (8 ranks) of each part at a time
#pragma unroll
                for (int c = 0; c < R / 8; ++c) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x0 = v[8 * c + 2 * e], x1 = v[8 * c + 2 * e + 1];
                        const float h0 = round_bf16(x0), h1 = round_bf16(x1);
                        hw[e] = pack_bf16(h0, h1);
                        lw[e] = pack_bf16(x0 - h0, x1 - h1);
                    }
                    const int pc = swz_chunk<R>(c, i);
                    *reinterpret_cast<uint4 *>(vh + i * W + pc * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(vl + i * W + pc * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
                tc::fence_proxy_async_smem();
            }
            tc::mbar_arrive(&v_full[vb]);
        }
    } else {
        // ---------------- epilogue: row i, columns 64h .. 64h + 63 of each n-block ----------------
        // Each warp updates its 32 rows x 64 columns of the stage in place and
        // stores them with its own TMA store (full tiles) or row stores
        // (ragged tiles); the stage goes back to the producer once all eight
        // warps' stores have read it.
        const int q = warp & 3, h = (warp - 6) >> 2;
        const int i = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int j = 0, pend = -1;
        // item metadata one item ahead, so its global load leaves the chain
        Item it = item_at(a, k0, np);
        int4 pt = a.ptiles[it.p];
        for (int k = k0; k < k1; ++k) {
            Item nit = it;
            int4 npt = pt;
            if (k + 1 < k1) {
                nit = item_at(a, k + 1, np);
                npt = a.ptiles[nit.p];
            }
            const int row0 = pt.y, rows = pt.z;
            const float scale = sscale[pt.x];
            const int nb = n_blocks(a, it), d_out = a.d_out[it.l];
            for (int b = 0; b < nb; ++b) {
                const int st = j % stages, ac = j % kAcc;
                const int col = it.cb * kColBlock + b * kNB + 64 * h;    // this warp's first column
                const bool live = col < d_out;
                bool ok = wait_ok(&acc_full[ac], (uint32_t)(j / kAcc) & 1u, err);
                ok = ok && wait_ok(&full[st], (uint32_t)(j / stages) & 1u, err);
                ok = __all_sync(0xffffffffu, ok);
                uint8_t *ybox = ring + (size_t)st * kStage + h * kTileBytes;
                uint8_t *yt = ybox + i * 128;                             // row i, 128-byte swizzle
                if (ok) {
                    tc::fence_after_sync();
                    uint32_t d[64];
                    tc::tmem_ld64_sync(tmem + lane_addr + (uint32_t)kNB * ac + 64u * h, d);
                    tc::fence_before_sync();
                    tc::mbar_arrive(&acc_empty[ac]);
                    if (live) {
                        // four 16-byte chunks of the row at a time: their loads
                        // go out together, then the arithmetic, then the
                        // stores (a store may not pass a later load of the same
                        // buffer, so one chunk at a time would chain them)
#pragma unroll
                        for (int c0 = 0; c0 < 8; c0 += 4) {
                            uint4 yv[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                yv[q] = *reinterpret_cast<const uint4 *>(yt + (((c0 + q) ^ (i & 7)) * 16));
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int c = c0 + q;
                                uint32_t w[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    w[e] = pack_bf16(fmaf(scale, __uint_as_float(d[8 * c + 2 * e]), bf_lo(w[e])),
                                                     fmaf(scale, __uint_as_float(d[8 * c + 2 * e + 1]), bf_hi(w[e])));
                                yv[q] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int c = c0 + q;
                                *reinterpret_cast<uint4 *>(yt + ((c ^ (i & 7)) * 16)) = yv[q];
                                if (rows < 128 && i < rows)
                                    reinterpret_cast<uint4 *>(a.y[it.l] + (size_t)(row0 + i) * d_out + col)[c] = yv[q];
                            }
                        }
                    }
                }
                // Generic writes to the stage become visible to the TMA store.
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (rows == 128 && live && !*err) {
                        tc::tma_store_2d(&a.ms[it.l], ybox + q * 32 * 128, col, row0 + 32 * q);
                        tc::bulk_commit_group();
                        tc::bulk_wait_group_read<1>();
                        if (pend >= 0) tc::mbar_arrive(&empty[pend]);
                        pend = st;
                    } else {
                        // No store of this block: hand back the one still pending too,
                        // so that the producer never waits on a stage nobody releases.
                        if (pend >= 0) {
                            tc::bulk_wait_group_read<0>();
                            tc::mbar_arrive(&empty[pend]);
                            pend = -1;
                        }
                        tc::mbar_arrive(&empty[st]);
                    }
                }
                ++j;
            }
            it = nit;
            pt = npt;
        }
        if (lane == 0) {
            tc::bulk_wait_group_all();
            if (pend >= 0) tc::mbar_arrive(&empty[pend]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (error && tid == 0) atomicExch(a.hdr + kHdrError, 1);
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ============================================================================
// Host side
// ============================================================================

// Shrink ring per CTA: three CTAs per SM below rank 64 (70 KB each: the q/k/v
// group keeps two stages, a single-layer group three; measured 335.6 ->
// 328.9 us per rank-32 prefill step against two CTAs of 108 KB), two at rank
// 64, whose four-layer groups need 48 KB stages and 256 TMEM columns.
constexpr size_t shrink_ring_budget(int R) { return R == 64 ? 108 * 1024 : 70 * 1024; }
constexpr size_t kExpandSmemBudget = 216 * 1024;   // one expand CTA per SM

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool encode_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int R>
size_t expand_smem(int stages) {
    return 1024 + (size_t)stages * (2 * kTileBytes + kNB * R * 2) +
           (expand_v_in_tmem(R) ? 0 : 4 * (size_t)128 * R * 2);
}

template <int R>
cudaError_t launch_r(const ShrinkArgs &sa, int grid_tiles, int n_jobs, size_t shrink_smem,
                     const ReduceArgs *ra, const ExpandArgs &ea, int expand_grid, cudaStream_t st,
                     int *kernels) {
    static std::atomic<uint64_t> attr{0};
    if (!device_bit(attr)) {
        cudaError_t e = cudaFuncSetAttribute(prefill_shrink_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(1024 + shrink_ring_budget(R)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(prefill_expand_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kExpandSmemBudget);
        if (e != cudaSuccess) return e;
        set_device_bit(attr);
    }
    int queued = 0;
    cudaError_t e = launch_pdl(prefill_shrink_kernel<R>, dim3(grid_tiles, n_jobs, 1), dim3(kThreads), shrink_smem,
                               st, sa);
    if (e == cudaSuccess) ++queued;
    if (e == cudaSuccess && ra) {
        e = launch_pdl(prefill_reduce_kernel, dim3(grid_tiles * (kPrefillRows / (256 / (R / 4))), ea.n, 1),
                       dim3(256), 0, st, *ra);
        if (e == cudaSuccess) ++queued;
    }
    if (e == cudaSuccess) {
        e = launch_pdl(prefill_expand_kernel<R>, dim3(expand_grid), dim3(kExpandThreads), expand_smem<R>(ea.stages),
                       st, ea);
        if (e == cudaSuccess) ++queued;
    }
    if (kernels) *kernels += queued;
    return e;
}

}  // namespace

bool prefill_tc_supported(int R) { return R == 16 || R == 32 || R == 64; }

cudaError_t launch_prefill_tc(const PrefillLayer *L, int n, int T, int S, int R, const float *scale,
                              int *hdr, const int4 *ptiles, int grid_tiles, int part_rows, int num_sms,
                              cudaStream_t st, int *kernels) {
    if (!prefill_tc_supported(R) || n < 1 || n > kMaxLayersPerCall || T < 1) return cudaErrorInvalidValue;
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }

    // Input groups: layers reading the same x, at most 256 TMEM columns each.
    const int max_members = 256 / R;
    int grp[kMaxLayersPerCall], ng = 0, gcount[kMaxLayersPerCall] = {0};
    int glead[kMaxLayersPerCall];
    for (int i = 0; i < n; ++i) {
        int g = -1;
        for (int h = 0; h < ng && g < 0; ++h)
            if (L[glead[h]].x == L[i].x && L[glead[h]].d_in == L[i].d_in && gcount[h] < max_members) g = h;
        if (g < 0) {
            g = ng++;
            glead[g] = i;
        }
        grp[i] = g;
        ++gcount[g];
    }

    ShrinkArgs sa{};
    ExpandArgs ea{};
    int m = 0;
    for (int g = 0; g < ng; ++g) {
        sa.g_first[g] = m;
        sa.g_count[g] = gcount[g];
        const PrefillLayer &x = L[glead[g]];
        if (!encode_2d(&sa.mx[g], x.x, (uint64_t)x.d_in, (uint64_t)T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&sa.mx32[g], x.x, (uint64_t)x.d_in, (uint64_t)T, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        for (int i = 0; i < n; ++i) {
            if (grp[i] != g) continue;
            if (!encode_2d(&sa.ma[m], L[i].A, (uint64_t)L[i].d_in, (uint64_t)S * R, 64, (uint32_t)R,
                           CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
            sa.part[m] = L[i].part;
            ++m;
        }
    }

    // d_in chunks: about one and a half waves of two shrink CTAs per SM,
    // each group's share proportional to its d_in; partial rows bound the
    // chunk count. (Measured: a target of 3 x SMs CTAs equals 4 x on the
    // rank-32 prefill step and beats it by 2 us on the rank-64 mixed step;
    // 2 x and 6-12 x are slower.)
    int max_ch = part_rows / T;
    if (max_ch > 16) max_ch = 16;
    if (max_ch < 1) return cudaErrorInvalidValue;
    const int est_tiles = T / kPrefillRows + 1;
    int kb[kMaxLayersPerCall], nch[kMaxLayersPerCall], kb_total = 0;
    for (int g = 0; g < ng; ++g) {
        kb[g] = (L[glead[g]].d_in + 63) / 64;
        kb_total += kb[g];
    }
    const int want = (3 * num_sms + est_tiles - 1) / est_tiles;    // jobs per tile
    int n_jobs = 0;
    for (int g = 0; g < ng; ++g) {
        int c = (int)(((long long)want * kb[g] + kb_total - 1) / kb_total);
        if (c < 1) c = 1;
        if (c > max_ch) c = max_ch;
        if (c > kb[g]) c = kb[g];
        nch[g] = c;
        n_jobs += c;
    }
    while (n_jobs > kMaxJobs) {
        int gm = 0;
        for (int g = 1; g < ng; ++g)
            if (nch[g] > nch[gm]) gm = g;
        --nch[gm];
        --n_jobs;
    }
    int jb = 0;
    size_t max_stage = 0;
    for (int g = 0; g < ng; ++g) {
        const size_t sb = kTileBytes + (size_t)gcount[g] * R * 128;
        if (sb > max_stage) max_stage = sb;
        for (int c = 0; c < nch[g]; ++c) {
            sa.jobs[jb].group = g;
            sa.jobs[jb].chunk = c;
            sa.jobs[jb].kb0 = (int)((long long)kb[g] * c / nch[g]);
            sa.jobs[jb].kb1 = (int)((long long)kb[g] * (c + 1) / nch[g]);
            ++jb;
        }
    }
    // One ring for the launch; each CTA cuts it into as many stages of its
    // group's size as fit (at least two for the largest stage).
    const size_t ring_budget = shrink_ring_budget(R);
    if (ring_budget / max_stage < 2) return cudaErrorInvalidValue;
    sa.ring_bytes = (int)ring_budget;
    const size_t shrink_smem = 1024 + ring_budget;
    int max_cols = 0;
    for (int g = 0; g < ng; ++g)
        if (gcount[g] * R > max_cols) max_cols = gcount[g] * R;
    sa.tmem_cols = (int)tmem_cols_for(max_cols);
    sa.ptiles = ptiles;
    sa.hdr = hdr;
    sa.T = T;
    // The expand's V loaders add the chunks themselves when that takes them
    // at most two rounds of loads (two chunks per round up to rank 32, one at
    // rank 64); otherwise a separate pass adds them once per (layer, tile)
    // with thousands of loads in flight.
    int max_nch = 1;
    for (int g = 0; g < ng; ++g) max_nch = nch[g] > max_nch ? nch[g] : max_nch;
    const int per_round = R <= 32 ? 2 : 1;
    const bool reduce_pass = (max_nch + per_round - 1) / per_round > 2;
    ReduceArgs ra{};
    ra.ptiles = ptiles;
    ra.hdr = hdr;
    ra.T = T;
    ra.R = R;

    ea.n = n;
    ea.sum_ncb = 0;
    for (int i = 0; i < n; ++i) {
        if (L[i].d_out % 64 != 0) return cudaErrorInvalidValue;
        if (!encode_2d(&ea.my[i], L[i].y, (uint64_t)L[i].d_out, (uint64_t)T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&ea.ms[i], L[i].y, (uint64_t)L[i].d_out, (uint64_t)T, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&ea.mb[i], L[i].B, (uint64_t)b_block(R), (uint64_t)S * (R / b_block(R)) * L[i].d_out,
                       (uint32_t)b_block(R), kNB,
                       b_block(R) == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B))
            return cudaErrorInvalidValue;
        ea.part[i] = L[i].part;
        ea.y[i] = static_cast<uint16_t *>(L[i].y);
        ea.d_out[i] = L[i].d_out;
        ea.ncb[i] = (L[i].d_out + kColBlock - 1) / kColBlock;
        ea.nch[i] = reduce_pass ? 1 : nch[grp[i]];
        ra.part[i] = L[i].part;
        ra.nch[i] = nch[grp[i]];
        ea.sum_ncb += ea.ncb[i];
    }
    const size_t vbytes = expand_v_in_tmem(R) ? 0 : 4 * (size_t)128 * R * 2;
    const size_t stage = 2 * kTileBytes + kNB * (size_t)R * 2;
    ea.stages = (int)((kExpandSmemBudget - 1024 - vbytes) / stage);
    if (ea.stages > kMaxStages) ea.stages = kMaxStages;
    ea.ptiles = ptiles;
    ea.hdr = hdr;
    ea.scale = scale;
    ea.S = S;
    ea.T = T;
    long long items = (long long)grid_tiles * ea.sum_ncb;
    const int expand_grid = (int)(items < num_sms ? items : num_sms);

    switch (R) {
    case 16: return launch_r<16>(sa, grid_tiles, n_jobs, shrink_smem, reduce_pass ? &ra : nullptr, ea, expand_grid, st,
                             kernels);
    case 32: return launch_r<32>(sa, grid_tiles, n_jobs, shrink_smem, reduce_pass ? &ra : nullptr, ea, expand_grid, st,
                             kernels);
    case 64: return launch_r<64>(sa, grid_tiles, n_jobs, shrink_smem, reduce_pass ? &ra : nullptr, ea, expand_grid, st,
                             kernels);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace lora
