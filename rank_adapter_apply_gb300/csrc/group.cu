// Token grouping: one CTA turns token_slot_idx into
//  * prefill tiles: contiguous runs of >= min_run tokens on one slot, cut into
//    tiles of kPrefillRows rows (slot, first row, rows);
//  * decode tiles: every other adapter token, grouped by slot with a stable
//    counting sort into `perm`, cut into tiles of kTileTokens (slot, perm
//    offset, count).
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
    int slot_cnt[kMaxSlots];
    int slot_off[kMaxSlots];
    int slot_carry[kMaxSlots];
    int wcnt[kWarps][kMaxSlots];
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

__device__ __forceinline__ int eff_slot(const int32_t *idx, const int *rank, int S, int t) {
    int s = idx[t];
    return (s >= 0 && s < S && rank[s] > 0) ? s : -1;
}

__global__ void __launch_bounds__(kGroupThreads, 1)
group_tokens_kernel(const int32_t *__restrict__ idx, int T, const int *__restrict__ rank, int S,
                    int min_run, int *hdr, int *perm, int *run_start, int *run_of,
                    int4 *tiles, int4 *ptiles) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    GroupSmem &sm = *reinterpret_cast<GroupSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) sm.invalid = 0;
    for (int s = tid; s < S; s += kGroupThreads) { sm.slot_cnt[s] = 0; sm.slot_carry[s] = 0; }
    __syncthreads();

    // Pass 1: runs of equal effective slot (only needed when the prefill path is on).
    int n_runs = 0;
    if (min_run > 0) {
        for (int base = 0; base < T; base += kGroupThreads) {
            int t = base + tid;
            int start = 0, e = -1;
            if (t < T) {
                int raw = idx[t];
                if (raw < -1 || raw >= S) atomicAdd(&sm.invalid, 1);
                e = eff_slot(idx, rank, S, t);
                start = (t == 0) || (eff_slot(idx, rank, S, t - 1) != e);
            }
            int tot;
            int pos = n_runs + block_excl_scan(start, sm, &tot);
            if (t < T) {
                if (start) run_start[pos] = t;
                run_of[t] = pos + start - 1;
            }
            n_runs += tot;
        }
        if (tid == 0) run_start[n_runs] = T;
    } else {
        for (int t = tid; t < T; t += kGroupThreads) {
            int raw = idx[t];
            if (raw < -1 || raw >= S) atomicAdd(&sm.invalid, 1);
        }
    }
    __syncthreads();

    // Pass 2: per-slot counts of decode tokens; prefill tiles from long runs.
    for (int t = tid; t < T; t += kGroupThreads) {
        int e = eff_slot(idx, rank, S, t);
        if (e < 0) continue;
        bool pre = false;
        if (min_run > 0) {
            int r = run_of[t];
            pre = (run_start[r + 1] - run_start[r]) >= min_run;
        }
        if (!pre) atomicAdd(&sm.slot_cnt[e], 1);
    }
    int n_ptiles = 0;
    if (min_run > 0) {
        for (int base = 0; base < n_runs; base += kGroupThreads) {
            int r = base + tid, nt = 0, st = 0, len = 0, e = -1;
            if (r < n_runs) {
                st = run_start[r];
                len = run_start[r + 1] - st;
                e = eff_slot(idx, rank, S, st);
                if (e >= 0 && len >= min_run) nt = (len + kPrefillRows - 1) / kPrefillRows;
            }
            int tot;
            int pos = n_ptiles + block_excl_scan(nt, sm, &tot);
            for (int i = 0; i < nt; ++i) {
                int rows = len - i * kPrefillRows;
                ptiles[pos + i] = make_int4(e, st + i * kPrefillRows,
                                            rows < kPrefillRows ? rows : kPrefillRows, 0);
            }
            n_ptiles += tot;
        }
    }
    __syncthreads();

    // Pass 3: slot offsets and decode tiles (S <= kMaxSlots <= kGroupThreads).
    int cnt = tid < S ? sm.slot_cnt[tid] : 0;
    int n_dec;
    int off = block_excl_scan(cnt, sm, &n_dec);
    if (tid < S) sm.slot_off[tid] = off;
    int nt = (cnt + kTileTokens - 1) / kTileTokens;
    int n_tiles;
    int tpos = block_excl_scan(nt, sm, &n_tiles);
    for (int i = 0; i < nt; ++i) {
        int c = cnt - i * kTileTokens;
        tiles[tpos + i] = make_int4(tid, off + i * kTileTokens, c < kTileTokens ? c : kTileTokens, 0);
    }
    __syncthreads();

    // Pass 4: stable scatter of decode tokens into perm, 1024 tokens at a time.
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < T; base += kGroupThreads) {
        for (int i = tid; i < kWarps * S; i += kGroupThreads) sm.wcnt[i / S][i % S] = 0;
        __syncthreads();
        int t = base + tid, e = -1;
        if (t < T) {
            e = eff_slot(idx, rank, S, t);
            if (e >= 0 && min_run > 0) {
                int r = run_of[t];
                if (run_start[r + 1] - run_start[r] >= min_run) e = -1;
            }
        }
        int key = e >= 0 ? e : (0x40000000 + lane);
        unsigned peers = __match_any_sync(kFull, key);
        int rank_in_warp = __popc(peers & lt_mask);
        if (e >= 0 && rank_in_warp == 0) sm.wcnt[w][e] = __popc(peers);
        __syncthreads();
        int chunk_total = 0;
        if (tid < S) {
            int run = 0;
            for (int ww = 0; ww < kWarps; ++ww) {
                int c = sm.wcnt[ww][tid];
                sm.wcnt[ww][tid] = run;
                run += c;
            }
            chunk_total = run;
        }
        __syncthreads();
        if (e >= 0) perm[sm.slot_off[e] + sm.slot_carry[e] + sm.wcnt[w][e] + rank_in_warp] = t;
        __syncthreads();
        if (tid < S) sm.slot_carry[tid] += chunk_total;
        __syncthreads();
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
    static bool attr_set = false;
    size_t smem = sizeof(GroupSmem);
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(group_tokens_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    group_tokens_kernel<<<1, kGroupThreads, smem, st>>>(
        idx, T, rank_dev, S, min_run, reinterpret_cast<int *>(ws + lay.hdr),
        reinterpret_cast<int *>(ws + lay.perm), reinterpret_cast<int *>(ws + lay.run_start),
        reinterpret_cast<int *>(ws + lay.run_of), reinterpret_cast<int4 *>(ws + lay.tiles),
        reinterpret_cast<int4 *>(ws + lay.ptiles));
    return cudaGetLastError();
}

}  // namespace lora
