// Token grouping: one CTA turns token_slot_idx into
//  * runs: maximal stretches of consecutive tokens with the same effective slot;
//  * prefill tiles: runs of >= min_run tokens on one slot, cut into tiles of
//    kPrefillRows rows (slot, first row, rows);
//  * decode tiles: every other adapter token, grouped by slot (counting sort
//    into `perm`, one run at a time), cut into tiles of kTileTokens (slot, perm
//    offset, count, the slot's rank).
// Each thread owns a contiguous block of tokens and then a contiguous block of
// runs, so the whole batch takes a handful of block-wide scans. The order of
// tokens inside one slot's decode list is not fixed (runs claim their places
// with shared-memory atomics); every token's result is computed from its own
// row only, so the outputs do not depend on it.
// Base-only tokens (-1), out-of-range indices and empty slots (rank 0) are
// dropped; out-of-range indices are added to the header's invalid counter.
// Multiple slots per batch come from the "Multi-LoRA 适配器缓存生产实战" page,
// section 核心原理 (max_loras: adapters usable in one batch).
#include "kernels.cuh"

namespace lora {
namespace {

constexpr int kGroupThreads = 1024;
constexpr int kWarps = kGroupThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

struct GroupSmem {
    int warp_part[kWarps];
    int total;
    int invalid;
    int rank[kMaxSlots];
    int slot_cnt[kMaxSlots];
    int slot_off[kMaxSlots];
    int slot_fill[kMaxSlots];
};

// Exclusive prefix sum over the CTA; *total receives the sum. All threads call.
__device__ int block_excl_scan(int v, GroupSmem &sm, int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_part[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = sm.warp_part[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        sm.warp_part[lane] = s;          // inclusive per-warp totals
        if (lane == 31) sm.total = s;
    }
    __syncthreads();
    int res = x - v + (w > 0 ? sm.warp_part[w - 1] : 0);
    *total = sm.total;
    __syncthreads();
    return res;
}

__device__ __forceinline__ int eff_of(int raw, const int *rank_s, int S) {
    return (raw >= 0 && raw < S && rank_s[raw] > 0) ? raw : -1;
}

__global__ void __launch_bounds__(kGroupThreads, 1)
group_tokens_kernel(const int32_t *__restrict__ idx, int T, const int *__restrict__ rank, int S,
                    int min_run, int *hdr, int *perm, int *run_start, int4 *tiles,
                    int4 *ptiles) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GroupSmem &sm = *reinterpret_cast<GroupSmem *>(smem_raw);
    const int tid = threadIdx.x;
    if (tid == 0) sm.invalid = 0;
    for (int s = tid; s < S; s += kGroupThreads) {
        sm.rank[s] = rank[s];
        sm.slot_cnt[s] = 0;
        sm.slot_fill[s] = 0;
    }
    __syncthreads();

    // Pass 1: run starts over this thread's tokens [t0, t1).
    const int K = (T + kGroupThreads - 1) / kGroupThreads;
    const int t0 = min(T, tid * K), t1 = min(T, t0 + K);
    const int before = t0 > 0 ? eff_of(idx[t0 - 1], sm.rank, S) : -2;   // -2 never matches
    int starts = 0, inval = 0, p = before;
    for (int t = t0; t < t1; ++t) {
        const int raw = idx[t];
        inval += (raw < -1 || raw >= S);
        const int e = eff_of(raw, sm.rank, S);
        starts += (e != p);
        p = e;
    }
    if (inval) atomicAdd(&sm.invalid, inval);
    int n_runs;
    int r = block_excl_scan(starts, sm, &n_runs) - 1;
    p = before;
    for (int t = t0; t < t1; ++t) {
        const int e = eff_of(idx[t], sm.rank, S);
        if (e != p) run_start[++r] = t;
        p = e;
    }
    if (tid == 0) run_start[n_runs] = T;
    __syncthreads();

    // Pass 2: this thread's runs [r0, r1): prefill tiles, decode counts per slot.
    const int KR = (n_runs + kGroupThreads - 1) / kGroupThreads;
    const int r0 = min(n_runs, tid * KR), r1 = min(n_runs, r0 + KR);
    int my_ptiles = 0;
    for (int q = r0; q < r1; ++q) {
        const int st = run_start[q], len = run_start[q + 1] - st;
        const int e = eff_of(idx[st], sm.rank, S);
        if (e < 0) continue;
        if (min_run > 0 && len >= min_run) my_ptiles += (len + kPrefillRows - 1) / kPrefillRows;
        else atomicAdd(&sm.slot_cnt[e], len);
    }
    int n_ptiles;
    int pos = block_excl_scan(my_ptiles, sm, &n_ptiles);
    for (int q = r0; q < r1 && my_ptiles > 0; ++q) {
        const int st = run_start[q], len = run_start[q + 1] - st;
        const int e = eff_of(idx[st], sm.rank, S);
        if (e < 0 || !(min_run > 0 && len >= min_run)) continue;
        for (int i = 0; i * kPrefillRows < len; ++i) {
            const int rows = len - i * kPrefillRows;
            ptiles[pos++] = make_int4(e, st + i * kPrefillRows, rows < kPrefillRows ? rows : kPrefillRows, 0);
        }
    }

    // Pass 3: slot offsets and decode tiles (S <= kMaxSlots <= kGroupThreads).
    const int cnt = tid < S ? sm.slot_cnt[tid] : 0;
    int n_dec;
    const int off = block_excl_scan(cnt, sm, &n_dec);
    if (tid < S) sm.slot_off[tid] = off;
    const int nt = (cnt + kTileTokens - 1) / kTileTokens;
    int n_tiles;
    const int tpos = block_excl_scan(nt, sm, &n_tiles);
    for (int i = 0; i < nt; ++i) {
        const int c = cnt - i * kTileTokens;
        tiles[tpos + i] = make_int4(tid, off + i * kTileTokens, c < kTileTokens ? c : kTileTokens, sm.rank[tid]);
    }
    __syncthreads();

    // Pass 4: decode runs claim a contiguous stretch of their slot's list.
    for (int q = r0; q < r1; ++q) {
        const int st = run_start[q], len = run_start[q + 1] - st;
        const int e = eff_of(idx[st], sm.rank, S);
        if (e < 0 || (min_run > 0 && len >= min_run)) continue;
        const int at = sm.slot_off[e] + atomicAdd(&sm.slot_fill[e], len);
        for (int i = 0; i < len; ++i) perm[at + i] = st + i;
    }

    if (tid == 0) {
        hdr[kHdrTiles] = n_tiles;
        hdr[kHdrPrefillTiles] = n_ptiles;
        hdr[kHdrDecodeTokens] = n_dec;
        if (sm.invalid) atomicAdd(&hdr[kHdrInvalid], sm.invalid);
    }
}

}  // namespace

cudaError_t launch_group_tokens(const int32_t *idx, int T, const int *rank_dev, int S,
                                int min_run, char *ws, const WsLayout &lay, cudaStream_t st) {
    static std::atomic<uint64_t> attr_set{0};
    size_t smem = sizeof(GroupSmem);
    if (!device_bit(attr_set)) {
        cudaError_t e = cudaFuncSetAttribute(group_tokens_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set_device_bit(attr_set);
    }
    group_tokens_kernel<<<1, kGroupThreads, smem, st>>>(
        idx, T, rank_dev, S, min_run, reinterpret_cast<int *>(ws + lay.hdr),
        reinterpret_cast<int *>(ws + lay.perm), reinterpret_cast<int *>(ws + lay.run_start),
        reinterpret_cast<int4 *>(ws + lay.tiles),
        reinterpret_cast<int4 *>(ws + lay.ptiles));
    return cudaGetLastError();
}

}  // namespace lora
