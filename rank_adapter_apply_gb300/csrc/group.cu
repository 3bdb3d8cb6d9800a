// Token grouping: turns token_slot_idx into
//  * prefill tiles: runs (maximal stretches of consecutive tokens with the
//    same effective slot) of >= min_run tokens, cut into tiles of
//    kPrefillRows rows (slot, first row, rows), in token order;
//  * decode tiles: every other adapter token, grouped by slot (a counting
//    sort into `perm`), cut into tiles of kTileTokens (slot, perm offset,
//    count, the slot's rank), slots in increasing order.
// Base-only tokens (-1), out-of-range indices and empty slots (rank 0) are
// dropped; out-of-range indices are added to the header's invalid counter.
// Multiple slots per batch come from the "Multi-LoRA 适配器缓存生产实战" page,
// section 核心原理 (max_loras: adapters usable in one batch).
//
// Work split: every token is handled on its own. A CTA of 1024 threads owns a
// block of up to kGBlock tokens (16 contiguous tokens per thread) held in
// shared memory: a block-wide max scan gives each token the start of its run,
// a min scan the start of the next run, so each token knows its run's length
// and slot without walking it. Batches of up to kGBlock tokens take one CTA;
// larger ones one CTA per block, which exchange per-block figures (first and
// last run start, prefill tile heads, decode tokens per slot) through the
// workspace at two grid barriers. The grid never exceeds what fits on the
// GPU at once, every barrier wait is bounded, and a wait that gives up sets
// the error word and leaves the batch with no tiles at all (every row of y
// unchanged). The position of a decode token inside its slot's list comes
// from shared-memory atomics, so the order of tokens of one slot is not fixed;
// every token's result is computed from its own row only, so no output
// depends on it.
#include "kernels.cuh"
#include "device_util.cuh"

namespace lora {
namespace {

constexpr int kGT = 1024;                  // threads per CTA
constexpr int kGPer = 16;                  // contiguous tokens per thread
constexpr int kGBlock = kGT * kGPer;       // tokens per CTA
constexpr int kGW = kGT / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kBarrierLimit = 1u << 22;
constexpr int kNoStart = 0x7fffffff;

struct GroupArgs {
    const int32_t *idx;
    const int *rank;
    int T, S, min_run, G;
    int *hdr, *perm;
    int4 *tiles, *ptiles;
    int *gx;        // exchange between CTAs: [G] first start, [G] last start, [G] tile heads, [G][S] decode counts
};

struct GroupSmem {
    int eff[kGBlock];               // effective slot of each token of the block (-1: none)
    int rank[kMaxSlots];
    int cnt[kMaxSlots];             // decode tokens of this block per slot, then the fill counters
    int base[kMaxSlots];            // where this block's decode tokens of each slot start in perm
    int wpart[kGW];
    int red;
    int invalid;
    int prev_eff;                   // effective slot of the token before the block (-2: none)
    int fail;
    int n_tiles, n_ptiles, n_dec;
    int up[kGT], from[kGT];         // per-thread last / first run start (block positions)
};

// Block-wide scans over one value per thread (all threads call). `op` 0: sum,
// exclusive (returns the sum of lower threads, *total = the sum of all);
// 1: max, inclusive; 2: min over this and higher threads (inclusive suffix).
template <int OP>
__device__ int block_scan(int v, GroupSmem &sm, int *total = nullptr) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    auto f = [](int a, int b) { return OP == 0 ? a + b : (OP == 1 ? max(a, b) : min(a, b)); };
    const int ident = OP == 0 ? 0 : (OP == 1 ? -1 : kNoStart);
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = OP == 2 ? __shfl_down_sync(kFull, x, o) : __shfl_up_sync(kFull, x, o);
        if (OP == 2 ? lane + o < 32 : lane >= o) x = f(x, y);
    }
    if (OP == 2 ? lane == 0 : lane == 31) sm.wpart[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = sm.wpart[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = OP == 2 ? __shfl_down_sync(kFull, s, o) : __shfl_up_sync(kFull, s, o);
            if (OP == 2 ? lane + o < 32 : lane >= o) s = f(s, y);
        }
        sm.wpart[lane] = s;         // inclusive over warps (prefix, or suffix for OP 2)
        if (lane == (OP == 2 ? 0 : 31)) sm.red = s;
    }
    __syncthreads();
    int res;
    if (OP == 0) res = x - v + (w > 0 ? sm.wpart[w - 1] : 0);
    else if (OP == 1) res = f(x, w > 0 ? sm.wpart[w - 1] : ident);
    else res = f(x, w < kGW - 1 ? sm.wpart[w + 1] : ident);
    if (total) *total = sm.red;
    __syncthreads();
    return res;
}

__device__ __forceinline__ int eff_of(int raw, const int *rank_s, int S) {
    return (raw >= 0 && raw < S && rank_s[raw] > 0) ? raw : -1;
}

// Grid barrier k (1, 2) over the G CTAs, bounded. Counters start at zero in
// every call (the last CTA to finish resets them).
__device__ bool grid_barrier(int *ctr, int k, int G) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1);
        uint32_t n = 0;
        int v;
        do {
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= k * G) break;
            __nanosleep(64);
        } while (++n < kBarrierLimit);
        __threadfence();
        ok = v >= k * G;
    }
    __syncthreads();
    return ok;
}

__global__ void __launch_bounds__(kGT, 1) group_tokens_kernel(const __grid_constant__ GroupArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GroupSmem &sm = *reinterpret_cast<GroupSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x, G = a.G, S = a.S;
    // Launched early (programmatic dependent launch): the slot ids and ranks
    // may come from the kernel before, and the previous apply's kernels still
    // read the lists rewritten here, so everything waits for it.
    grid_dependency_wait();
    grid_launch_dependents();
    const int b0 = (int)((long long)a.T * c / G), b1 = (int)((long long)a.T * (c + 1) / G);
    const int n = b1 - b0;

    // ---- phase 1: slot ids of the block into shared memory ---------------
    if (tid == 0) {
        sm.invalid = 0;
        sm.fail = 0;
        sm.n_tiles = sm.n_ptiles = sm.n_dec = 0;
    }
    for (int s = tid; s < S; s += kGT) {
        sm.rank[s] = a.rank[s];
        sm.cnt[s] = 0;
    }
    int inval = 0;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int i = j * kGT + tid;
        const int raw = i < n ? a.idx[b0 + i] : -1;
        inval += (i < n) && (raw < -1 || raw >= S);
        sm.eff[i] = raw;
    }
    const int raw_prev = (tid == 0 && b0 > 0) ? a.idx[b0 - 1] : -1;
    __syncthreads();
    if (tid == 0) sm.prev_eff = b0 > 0 ? eff_of(raw_prev, sm.rank, S) : -2;
    const int p0 = tid * kGPer;                 // this thread's tokens: block positions [p0, p0 + 16)
    int e[kGPer];
#pragma unroll
    for (int j = 0; j < kGPer; ++j) e[j] = p0 + j < n ? eff_of(sm.eff[p0 + j], sm.rank, S) : -1;
    if (inval) atomicAdd(&sm.invalid, inval);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kGPer; ++j) sm.eff[p0 + j] = e[j];
    __syncthreads();

    // ---- phase 2: each token's run [start, end) ---------------------------
    // Run starts (block positions); the last one at or before each token by a
    // max scan, the first one after each token by a suffix min scan.
    int last_start = -1, first_start = kNoStart;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int p = p0 + j;
        const bool st = p < n && e[j] != (p == 0 ? sm.prev_eff : sm.eff[p - 1]);
        if (st) {
            last_start = p;
            if (first_start == kNoStart) first_start = p;
        }
    }
    const int upto = block_scan<1>(last_start, sm);      // last start at or before my last token
    const int from = block_scan<2>(first_start, sm);     // first start at or after my first token
    bool good = true;
    if (G > 1) {
        // the block's first and last run start, for the neighbouring blocks
        if (tid == 0) a.gx[c] = from == kNoStart ? kNoStart : b0 + from;
        if (tid == kGT - 1) a.gx[G + c] = upto < 0 ? -1 : b0 + upto;
        good = grid_barrier(a.hdr + kHdrGroupBar, 1, G);
    }
    // Runs that cross the block's edges: the last start before the block and
    // the first start after it (global positions; block 0 starts a run at 0).
    int before = 0, after = a.T;
    if (G > 1 && good) {
        for (int q = 0; q < c; ++q) before = max(before, a.gx[G + q]);
        for (int q = G - 1; q > c; --q) after = a.gx[q] != kNoStart ? a.gx[q] : after;
    }
    // The last start among lower threads and the first among higher threads
    // bound the runs of this thread's first and last tokens; the tokens in
    // between are walked.
    sm.up[tid] = upto;
    sm.from[tid] = from;
    __syncthreads();
    const int lo_start = tid > 0 ? sm.up[tid - 1] : -1;
    const int hi_start = tid < kGT - 1 ? sm.from[tid + 1] : kNoStart;

    int heads = 0;
    int run_s[kGPer], run_e[kGPer];
    {
        int cur = lo_start >= 0 ? b0 + lo_start : before;
        for (int j = 0; j < kGPer; ++j) {
            const int p = p0 + j;
            if (p < n && e[j] != (p == 0 ? sm.prev_eff : sm.eff[p - 1])) cur = b0 + p;
            run_s[j] = cur;
        }
        int nxt = hi_start != kNoStart ? b0 + hi_start : after;
        for (int j = kGPer - 1; j >= 0; --j) {
            const int p = p0 + j;
            run_e[j] = nxt;
            if (p < n && e[j] != (p == 0 ? sm.prev_eff : sm.eff[p - 1])) nxt = b0 + p;
        }
    }
    // Classify: prefill tile heads and decode tokens (per-slot counts).
    unsigned dec_mask = 0;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int p = p0 + j;
        if (p >= n || e[j] < 0) continue;
        const int len = run_e[j] - run_s[j];
        if (a.min_run > 0 && len >= a.min_run) {
            heads += ((b0 + p - run_s[j]) % kPrefillRows) == 0;
        } else {
            dec_mask |= 1u << j;
        }
    }
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int s = (dec_mask >> j) & 1u ? e[j] : -1 - lane;
        const unsigned peers = __match_any_sync(kFull, s);
        if (s >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sm.cnt[s], __popc(peers));
    }
    int n_heads_blk;
    const int head_pos = block_scan<0>(heads, sm, &n_heads_blk);
    if (G > 1) {
        if (tid == 0) a.gx[2 * G + c] = n_heads_blk;
        for (int s = tid; s < S; s += kGT) a.gx[3 * G + c * S + s] = sm.cnt[s];
        good = grid_barrier(a.hdr + kHdrGroupBar, 2, G) && good;
    }
    if (!good) {
        // A barrier gave up: this CTA writes no list (the header will hold no tiles).
        if (tid == 0) sm.fail = 1;
        goto header;
    }

    // ---- phase 3: offsets, then every list ---------------------------------
    {
    int head0 = 0, n_ptiles = n_heads_blk;
    if (G > 1) {
        n_ptiles = 0;
        for (int q = 0; q < G; ++q) {
            const int h = a.gx[2 * G + q];
            head0 += q < c ? h : 0;
            n_ptiles += h;
        }
    }
    // decode tokens per slot over the batch, and this block's share before it
    int tot = 0, mine_before = 0;
    if (tid < S) {
        if (G > 1) {
            for (int q = 0; q < G; ++q) {
                const int v = a.gx[3 * G + q * S + tid];
                tot += v;
                mine_before += q < c ? v : 0;
            }
        } else {
            tot = sm.cnt[tid];
        }
    }
    int n_dec;
    const int slot_off = block_scan<0>(tid < S ? tot : 0, sm, &n_dec);
    const int nt = (tot + kTileTokens - 1) / kTileTokens;
    int n_tiles;
    const int tile_off = block_scan<0>(tid < S ? nt : 0, sm, &n_tiles);
    if (tid < S) {
        sm.base[tid] = slot_off + mine_before;
        sm.cnt[tid] = 0;                        // now the fill counter of this block
        if (c == 0)
            for (int i = 0; i < nt; ++i) {
                const int k = tot - i * kTileTokens;
                a.tiles[tile_off + i] = make_int4(tid, slot_off + i * kTileTokens, k < kTileTokens ? k : kTileTokens,
                                                  sm.rank[tid]);
            }
    }
    __syncthreads();
    // prefill tiles, in token order
    int hp = head0 + head_pos;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int p = p0 + j;
        if (p >= n || e[j] < 0 || ((dec_mask >> j) & 1u)) continue;
        if (((b0 + p - run_s[j]) % kPrefillRows) != 0) continue;
        const int rows = run_e[j] - (b0 + p);
        a.ptiles[hp++] = make_int4(e[j], b0 + p, rows < kPrefillRows ? rows : kPrefillRows, 0);
    }
    // decode tokens: a place in their slot's list
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int s = (dec_mask >> j) & 1u ? e[j] : -1 - lane;
        const unsigned peers = __match_any_sync(kFull, s);
        const int leader = __ffs(peers) - 1;
        int at = 0;
        if (s >= 0 && lane == leader) at = atomicAdd(&sm.cnt[s], __popc(peers));
        at = __shfl_sync(kFull, at, leader);
        if (s >= 0) a.perm[sm.base[s] + at + __popc(peers & ((1u << lane) - 1u))] = b0 + p0 + j;
    }
    if (tid == 0) {
        sm.n_tiles = n_tiles;
        sm.n_ptiles = n_ptiles;
        sm.n_dec = n_dec;
    }
    }

    // ---- the header: written by the last CTA to finish ---------------------
header:
    __syncthreads();
    if (tid == 0) {
        const int n_tiles = sm.n_tiles, n_ptiles = sm.n_ptiles, n_dec = sm.n_dec;
        if (sm.invalid) atomicAdd(a.hdr + kHdrInvalid, sm.invalid);
        if (sm.fail) {
            atomicExch(a.hdr + kHdrError, 1);
            atomicExch(a.hdr + kHdrGroupFail, 1);
        }
        __threadfence();
        const int done = G > 1 ? atomicAdd(a.hdr + kHdrGroupDone, 1) : 0;
        if (done == G - 1) {
            __threadfence();
            const bool failed = sm.fail || (G > 1 && atomicAdd(a.hdr + kHdrGroupFail, 0) != 0);
            // A failed barrier leaves the lists incomplete: no tiles at all.
            a.hdr[kHdrTiles] = failed ? 0 : n_tiles;
            a.hdr[kHdrPrefillTiles] = failed ? 0 : n_ptiles;
            a.hdr[kHdrDecodeTokens] = failed ? 0 : n_dec;
            if (G > 1) {
                a.hdr[kHdrGroupBar] = 0;
                a.hdr[kHdrGroupDone] = 0;
                a.hdr[kHdrGroupFail] = 0;
            }
        }
    }
}

}  // namespace

int group_ctas(int T) {
    const int G = (T + kGBlock - 1) / kGBlock;
    return G < 1 ? 1 : G;
}

int group_max_tokens(int num_sms) { return (num_sms > 0 ? num_sms : 1) * kGBlock; }

cudaError_t launch_group_tokens(const int32_t *idx, int T, const int *rank_dev, int S,
                                int min_run, char *ws, const WsLayout &lay, int num_sms, cudaStream_t st) {
    static std::atomic<uint64_t> attr_set{0};
    const size_t smem = sizeof(GroupSmem);
    if (!device_bit(attr_set)) {
        cudaError_t e = cudaFuncSetAttribute(group_tokens_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set_device_bit(attr_set);
    }
    GroupArgs a{};
    a.idx = idx;
    a.rank = rank_dev;
    a.T = T;
    a.S = S;
    a.min_run = min_run;
    // One CTA per block of kGBlock tokens; the barriers need every CTA
    // resident at once (one per SM at most), so larger batches are refused.
    a.G = group_ctas(T);
    if (a.G > num_sms || (a.G > 1 && (size_t)a.G * (3 + S) > lay.gx_ints)) return cudaErrorInvalidValue;
    a.hdr = reinterpret_cast<int *>(ws + lay.hdr);
    a.perm = reinterpret_cast<int *>(ws + lay.perm);
    a.tiles = reinterpret_cast<int4 *>(ws + lay.tiles);
    a.ptiles = reinterpret_cast<int4 *>(ws + lay.ptiles);
    a.gx = reinterpret_cast<int *>(ws + lay.gx);
    return launch_pdl(group_tokens_kernel, dim3(a.G), dim3(kGT), smem, st, a);
}

}  // namespace lora
