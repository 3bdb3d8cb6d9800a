// Token grouping: turns token_slot_idx into
//  * prefill tiles: runs (maximal stretches of consecutive tokens with the
//    same effective slot) of >= min_run tokens, cut into tiles of
//    kPrefillRows rows (slot, first row, rows, the slot's rank), in token order;
//  * decode tiles: every other adapter token, grouped by slot (a counting
//    sort into `perm`), cut into tiles of kTileTokens (slot, perm offset,
//    count, the slot's rank), slots in increasing order.
// Base-only tokens (-1), out-of-range indices and empty slots (rank 0) are
// dropped; out-of-range indices are added to the header's invalid counter.
// Multiple slots per batch come from the "Multi-LoRA 适配器缓存生产实战" page,
// section 核心原理 (max_loras: adapters usable in one batch).
//
// Work split: a CTA of 256 threads owns a block of up to kGBlock = 4096
// tokens, 16 contiguous tokens per thread, held in shared memory. Each thread
// marks the run starts among its tokens in a 16-bit mask; a suffix min scan
// gives it the first run start after its tokens, so every run's length is
// known to the thread holding its start, which classifies it (prefill tiles
// or decode tokens) and emits its prefill tiles; a max scan hands the class
// of the run entering each thread's tokens to that thread. Scans are warp
// shuffles plus one exchange of warp totals through shared memory. Batches of
// up to kGBlock tokens take one CTA; larger ones one CTA per block, which
// exchange per-block figures (first and last run start, prefill tiles,
// decode tokens per slot) at two barriers. Up to kGCluster blocks form one
// thread-block cluster: the figures go to CTA 0's shared memory and the
// barriers are the cluster's hardware barriers (every CTA of a cluster is
// resident at once and reaches each of them on every path). Larger batches
// exchange through the workspace at two grid barriers; that grid never
// exceeds what fits on the GPU at once, every barrier wait is bounded, and a
// wait that gives up sets the error word and leaves the batch with no tiles
// at all (every row of y unchanged). The position of a decode token inside
// its slot's list comes from one shared-memory atomic per stretch of
// same-slot tokens of a thread (which also counts them), so the order of
// tokens of one slot is not fixed; every token's result is computed from its
// own row only, so no output depends on it.
#include "kernels.cuh"
#include "device_util.cuh"

#include <cooperative_groups.h>

namespace lora {
namespace {

constexpr int kGT = 256;                   // threads per CTA
constexpr int kGPer = 16;                  // contiguous tokens per thread
constexpr int kGBlock = kGT * kGPer;       // tokens per CTA
constexpr int kGW = kGT / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kBarrierLimit = 1u << 22;
constexpr int kNoStart = 0x7fffffff;
constexpr int kGCluster = 8;               // blocks that exchange through a cluster's shared memory
static_assert(kMaxSlots <= kGT, "one thread per slot in the per-slot scans");
static_assert(kPrefillRows == 128, "prefill tile count by shift");

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
    int cnt[kMaxSlots];             // decode tokens of this block per slot
    int base[kMaxSlots];            // where this block's decode tokens of each slot start in perm
    int toff[kMaxSlots + 1];        // first decode tile of each slot; [S]: all decode tiles
    int soff[kMaxSlots + 1];        // first place of each slot in perm; [S]: all decode tokens
    int gx[kGCluster * (3 + kMaxSlots)];   // a cluster's exchange area (CTA 0's copy is used)
    int w0[3][kGW], w1[3][kGW];     // warp totals of the three scan passes
    int invalid;
    int prev_eff;                   // effective slot of the token before the block (-2: none)
    int fail;
    int blk_last;                   // the block's last run start (block position, -1: none)
    int n_tiles, n_ptiles, n_dec;
};

// Warp-level inclusive scans.
__device__ __forceinline__ int warp_sum(int x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    return x;
}
__device__ __forceinline__ int warp_max(int x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x = max(x, y);
    }
    return x;
}
__device__ __forceinline__ int warp_suffix_min(int x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(kFull, x, o);
        if (lane + o < 32) x = min(x, y);
    }
    return x;
}

// Reduce a[q * stride] over q < G (op 0: sum, 1: max, 2: sum over q < lim
// only), eight loads in flight at a time.
template <int OP>
__device__ __forceinline__ int gx_reduce(const int *a, int stride, int G, int lim = 0) {
    int acc = OP == 1 ? -1 : 0;
    for (int q0 = 0; q0 < G; q0 += 8) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = q0 + i < G ? a[(size_t)(q0 + i) * stride] : (OP == 1 ? -1 : 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (OP == 1) acc = max(acc, v[i]);
            else if (OP == 0 || q0 + i < lim) acc += v[i];
        }
    }
    return acc;
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
            __nanosleep(32);
        } while (++n < kBarrierLimit);
        __threadfence();
        ok = v >= k * G;
    }
    __syncthreads();
    return ok;
}

// The two exchanges between the blocks of a batch: with a cluster, the
// cluster's barrier (release the figures written into CTA 0, acquire every
// block's); otherwise the bounded grid barrier.
template <bool kCl>
__device__ __forceinline__ bool exchange(int *hdr, int k, int G) {
    if constexpr (kCl) {
        cluster_arrive_release();
        cluster_wait_acquire();
        return true;
    } else {
        return grid_barrier(hdr + kHdrGroupBar, k, G);
    }
}

template <bool kCl>
__global__ void __launch_bounds__(kGT, 1) group_tokens_kernel(const __grid_constant__ GroupArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GroupSmem &sm = *reinterpret_cast<GroupSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x, G = a.G, S = a.S, T = a.T;
    // Exchange area: CTA 0's shared copy in a cluster, else the workspace's.
    int *gx = a.gx;
    if constexpr (kCl) {
        cluster_arrive_relaxed();             // this CTA has started: peers may write into it
        gx = cooperative_groups::this_cluster().map_shared_rank(sm.gx, 0);
    }
    // Launched early (programmatic dependent launch): the slot ids and ranks
    // may come from the kernel before, and the previous apply's kernels still
    // read the lists rewritten here, so everything waits for it.
    grid_dependency_wait();
    grid_launch_dependents();
    const int b0 = (int)((long long)T * c / G), b1 = (int)((long long)T * (c + 1) / G);
    const int n = b1 - b0;

    // ---- phase 1: slot ids of the block into shared memory ---------------
    // every load issued before any is used (one memory round trip)
    int raw[kGPer];
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        const int i = j * kGT + tid;
        raw[j] = -1;
        if (i < n) raw[j] = a.idx[b0 + i];
    }
    const int raw_prev = (tid == 0 && b0 > 0) ? a.idx[b0 - 1] : -1;
    const int my_rank = tid < S ? a.rank[tid] : 0;
    if (tid == 0) {
        sm.invalid = 0;
        sm.fail = 0;
        sm.n_tiles = sm.n_ptiles = sm.n_dec = 0;
        sm.blk_last = -1;
    }
    if (tid < S) {
        sm.rank[tid] = my_rank;
        sm.cnt[tid] = 0;
    }
    int inval = 0;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        inval += raw[j] < -1 || raw[j] >= S;
        sm.eff[j * kGT + tid] = raw[j];
    }
    __syncthreads();
    if (tid == 0) sm.prev_eff = b0 > 0 ? eff_of(raw_prev, sm.rank, S) : -2;
    if (inval) atomicAdd(&sm.invalid, inval);
    // this thread's tokens: block positions [p0, p0 + kGPer), read 16 bytes at a time
    const int p0 = tid * kGPer;
    int e[kGPer];
    {
        const int4 *src = reinterpret_cast<const int4 *>(sm.eff + p0);
#pragma unroll
        for (int q = 0; q < kGPer / 4; ++q) {
            const int4 v = src[q];
            e[4 * q] = v.x;
            e[4 * q + 1] = v.y;
            e[4 * q + 2] = v.z;
            e[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < kGPer; ++j) e[j] = p0 + j < n ? eff_of(e[j], sm.rank, S) : -1;
    }
    __syncthreads();
    {
        int4 *dst = reinterpret_cast<int4 *>(sm.eff + p0);
#pragma unroll
        for (int q = 0; q < kGPer / 4; ++q) dst[q] = make_int4(e[4 * q], e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
    }
    __syncthreads();

    // ---- phase 2: runs ----------------------------------------------------
    // Bit j of smask: token p0 + j starts a run (its slot differs from the
    // token before).
    unsigned smask = 0;
    {
        int prev = tid == 0 ? sm.prev_eff : sm.eff[p0 - 1];
#pragma unroll
        for (int j = 0; j < kGPer; ++j) {
            if (p0 + j < n && e[j] != prev) smask |= 1u << j;
            prev = e[j];
        }
    }
    // First run start after this thread's tokens (block position): suffix min
    // over higher lanes, then over higher warps.
    int hi_start, blk_first;
    {
        const int first_start = smask ? p0 + __ffs(smask) - 1 : kNoStart;
        const int inc = warp_suffix_min(first_start, lane);
        int exc = __shfl_down_sync(kFull, inc, 1);
        if (lane == 31) exc = kNoStart;
        if (lane == 0) sm.w0[0][w] = inc;
        if (smask) atomicMax(&sm.blk_last, p0 + 31 - __clz(smask));
        __syncthreads();
        int higher = kNoStart, all = kNoStart;
#pragma unroll
        for (int q = 0; q < kGW; ++q) {
            const int v = sm.w0[0][q];
            if (q > w) higher = min(higher, v);
            all = min(all, v);
        }
        hi_start = min(exc, higher);
        blk_first = all;
    }
    bool good = true;
    if (G > 1) {
        if constexpr (kCl) cluster_wait_acquire();   // every CTA of the cluster has started
        if (tid == 0) {
            gx[c] = blk_first == kNoStart ? kNoStart : b0 + blk_first;
            gx[G + c] = sm.blk_last < 0 ? -1 : b0 + sm.blk_last;
        }
        good = exchange<kCl>(a.hdr, 1, G);
    }
    // The last start before the block and the first one after it (global
    // positions; block 0 starts a run at token 0).
    int before = 0, after = T;
    if (G > 1 && good) {
        if (c > 0) before = max(0, gx_reduce<1>(gx + G, 1, c));
        for (int q0 = c + 1; q0 < G; q0 += 8) {     // the nearest later block with a start
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = q0 + i < G ? gx[q0 + i] : kNoStart;
            int f = kNoStart;
#pragma unroll
            for (int i = 7; i >= 0; --i) f = v[i] != kNoStart ? v[i] : f;
            if (f != kNoStart) {
                after = f;
                break;
            }
        }
    }
    // Class of a run: 0 none (base-only slot), 1 prefill tiles, 2 decode tokens.
    auto run_class = [&](int slot, int len) {
        return slot < 0 ? 0 : ((a.min_run > 0 && len >= a.min_run) ? 1 : 2);
    };
    // Runs starting in this thread's tokens: their prefill tiles, the class of
    // the last one (for the tokens of higher threads), 2 bits of class per start.
    // (last start first: each run ends where the next one starts)
    int heads = 0, last_key = -1;
    uint32_t cls_bits = 0;
    {
        int end = hi_start != kNoStart ? b0 + hi_start : after;
#pragma unroll
        for (int j = kGPer - 1; j >= 0; --j) {
            if ((smask >> j) & 1u) {
                const int s0 = b0 + p0 + j;
                const int cls = run_class(e[j], end - s0);
                if (cls == 1) heads += (end - s0 + kPrefillRows - 1) >> 7;
                cls_bits |= (uint32_t)cls << (2 * j);
                if (last_key < 0) last_key = (p0 + j + 1) * 4 + cls;
                end = s0;
            }
        }
    }
    // One pass: the last run key of lower threads (max) and the prefill tiles
    // of lower threads (sum).
    int key_lower, head_pos, n_heads_blk;
    {
        const int km = warp_max(last_key, lane), hs = warp_sum(heads, lane);
        int km_exc = __shfl_up_sync(kFull, km, 1), hs_exc = hs - heads;
        if (lane == 0) km_exc = -1;
        if (lane == 31) {
            sm.w0[1][w] = km;
            sm.w1[1][w] = hs;
        }
        __syncthreads();
        int kl = -1, hl = 0, ht = 0;
#pragma unroll
        for (int q = 0; q < kGW; ++q) {
            const int kv = sm.w0[1][q], hv = sm.w1[1][q];
            if (q < w) {
                kl = max(kl, kv);
                hl += hv;
            }
            ht += hv;
        }
        key_lower = max(km_exc, kl);
        head_pos = hs_exc + hl;
        n_heads_blk = ht;
    }
    // The class of the run entering this thread's tokens.
    int cls_cur;
    if (key_lower >= 0) {
        cls_cur = key_lower & 3;
    } else if (c == 0) {
        cls_cur = 0;                              // token 0 starts a run
    } else {
        const int end = blk_first != kNoStart ? b0 + blk_first : after;
        cls_cur = run_class(sm.prev_eff, end - before);
    }
    unsigned dec_mask = 0;
#pragma unroll
    for (int j = 0; j < kGPer; ++j) {
        if ((smask >> j) & 1u) cls_cur = (cls_bits >> (2 * j)) & 3u;
        if (p0 + j < n && e[j] >= 0 && cls_cur == 2) dec_mask |= 1u << j;
    }
    // Decode tokens per slot, and each token's place among this block's
    // tokens of its slot: one shared atomic per stretch of same-slot decode
    // tokens of this thread claims the whole stretch (its length from a
    // backward pass).
    int off[kGPer];
    {
        int len[kGPer];
        int n_len = 0, n_slot = -1;
#pragma unroll
        for (int j = kGPer - 1; j >= 0; --j) {
            const int s = (dec_mask >> j) & 1u ? e[j] : -1;
            n_len = (s >= 0 && s == n_slot) ? n_len + 1 : 1;
            len[j] = n_len;
            n_slot = s;
        }
        int ps = -1, o = 0;
#pragma unroll
        for (int j = 0; j < kGPer; ++j) {
            const int s = (dec_mask >> j) & 1u ? e[j] : -1;
            if (s >= 0) o = s == ps ? o + 1 : atomicAdd(&sm.cnt[s], len[j]);
            off[j] = o;
            ps = s;
        }
    }
    __syncthreads();
    if (G > 1) {
        if (tid == 0) gx[2 * G + c] = n_heads_blk;
        if (tid < S) gx[3 * G + c * S + tid] = sm.cnt[tid];
        good = exchange<kCl>(a.hdr, 2, G) && good;
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
            head0 = gx_reduce<2>(gx + 2 * G, 1, G, c);
            n_ptiles = gx_reduce<0>(gx + 2 * G, 1, G);
        }
        // decode tokens per slot over the batch (thread = slot), and the
        // blocks' share before this one
        int tot = 0, mine_before = 0;
        if (tid < S) {
            if (G > 1) {
                tot = gx_reduce<0>(gx + 3 * G + tid, S, G);
                mine_before = gx_reduce<2>(gx + 3 * G + tid, S, G, c);
            } else {
                tot = sm.cnt[tid];
            }
        }
        // One pass: each slot's first place in perm and first decode tile.
        const int nt = (tot + kTileTokens - 1) / kTileTokens;
        int slot_off, tile_off, n_dec, n_tiles;
        {
            const int ds = warp_sum(tot, lane), ts = warp_sum(nt, lane);
            if (lane == 31) {
                sm.w0[2][w] = ds;
                sm.w1[2][w] = ts;
            }
            __syncthreads();
            int dl = 0, tl = 0, dt = 0, tt = 0;
#pragma unroll
            for (int q = 0; q < kGW; ++q) {
                const int dv = sm.w0[2][q], tv = sm.w1[2][q];
                if (q < w) {
                    dl += dv;
                    tl += tv;
                }
                dt += dv;
                tt += tv;
            }
            slot_off = ds - tot + dl;
            tile_off = ts - nt + tl;
            n_dec = dt;
            n_tiles = tt;
        }
        if (tid < S) {
            sm.base[tid] = slot_off + mine_before;
            sm.toff[tid] = tile_off;
            sm.soff[tid] = slot_off;
        }
        if (tid == 0) {
            sm.toff[S] = n_tiles;
            sm.soff[S] = n_dec;
        }
        __syncthreads();
        // decode tiles, spread over every thread of the grid: tile i belongs
        // to the slot s with toff[s] <= i < toff[s + 1]
        for (int i = c * kGT + tid; i < n_tiles; i += G * kGT) {
            int lo = 0, hi = S;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sm.toff[mid] <= i) lo = mid;
                else hi = mid;
            }
            const int k = i - sm.toff[lo];
            const int left = sm.soff[lo + 1] - sm.soff[lo] - k * kTileTokens;
            a.tiles[i] = make_int4(lo, sm.soff[lo] + k * kTileTokens, left < kTileTokens ? left : kTileTokens,
                                   sm.rank[lo]);
        }
        // prefill tiles of the runs starting here, in token order
        int hp = head0 + head_pos;
        unsigned m = smask;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            if (((cls_bits >> (2 * j)) & 3u) != 1u) continue;
            const int s0 = b0 + p0 + j;
            const int end = m ? b0 + p0 + __ffs(m) - 1 : (hi_start != kNoStart ? b0 + hi_start : after);
            const int slot = sm.eff[p0 + j];
            for (int r = s0; r < end; r += kPrefillRows)
                a.ptiles[hp++] = make_int4(slot, r, end - r < kPrefillRows ? end - r : kPrefillRows, sm.rank[slot]);
        }
        // decode tokens at the places claimed above
#pragma unroll
        for (int j = 0; j < kGPer; ++j)
            if ((dec_mask >> j) & 1u) a.perm[sm.base[e[j]] + off[j]] = b0 + p0 + j;
        if (tid == 0) {
            sm.n_tiles = n_tiles;
            sm.n_ptiles = n_ptiles;
            sm.n_dec = n_dec;
        }
    }

    // ---- the header: written by the last CTA to finish ---------------------
header:
    __syncthreads();
    if constexpr (kCl) {
        // CTA 0 keeps its shared memory until every peer has read it
        if (G > 1) {
            cluster_arrive_release();
            cluster_wait_acquire();
        }
    }
    if (tid == 0) {
        const int n_tiles = sm.n_tiles, n_ptiles = sm.n_ptiles, n_dec = sm.n_dec;
        if (sm.invalid) atomicAdd(a.hdr + kHdrInvalid, sm.invalid);
        if (sm.fail) {
            atomicExch(a.hdr + kHdrError, 1);
            atomicExch(a.hdr + kHdrGroupFail, 1);
            __threadfence();                    // the flag before the count
        }
        // (the lists need no fence: the kernels that read them start after
        // this one has completed)
        const int done = kCl ? (c == 0 ? G - 1 : -1) : (G > 1 ? atomicAdd(a.hdr + kHdrGroupDone, 1) : 0);
        if (done == G - 1) {
            const bool failed = sm.fail || (G > 1 && atomicAdd(a.hdr + kHdrGroupFail, 0) != 0);
            // A failed barrier leaves the lists incomplete: no tiles at all.
            a.hdr[kHdrTiles] = failed ? 0 : n_tiles;
            a.hdr[kHdrPrefillTiles] = failed ? 0 : n_ptiles;
            a.hdr[kHdrDecodeTokens] = failed ? 0 : n_dec;
            if (!kCl && G > 1) {
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
        cudaError_t e = cudaFuncSetAttribute(group_tokens_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(group_tokens_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
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
    if (a.G == 1 || a.G > kGCluster)
        return launch_pdl(group_tokens_kernel<false>, dim3(a.G), dim3(kGT), smem, st, a);
    // 2..kGCluster blocks: one cluster of G CTAs
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.G);
    cfg.blockDim = dim3(kGT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.G;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, group_tokens_kernel<true>, a);
}

}  // namespace lora
