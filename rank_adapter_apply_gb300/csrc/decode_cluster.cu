// Decode step on thread-block clusters: one launch applies every layer of a
// layer set to a batch of at most kFusedMaxTokens tokens.
//
//   v[t][k]  = sum_j A_s[k][j] x[t][j]                      (k < r_s)
//   y[t][i] += (lora_alpha_s / r_s) * sum_k B_s[i][k] v[t][k]
//
// (the LoRA delta with the PEFT fields r / lora_alpha, "vLLM LoRA Resolver
// 插件详解" page, section 3.2; several slots per batch, max_loras and
// max_lora_rank from the "Multi-LoRA 适配器缓存生产实战" page, section 核心原理.)
//
// Work split. Tokens are grouped by slot into tiles of <= 16 tokens. One
// cluster of kCl = 8 CTAs owns one (layer, tile): CTA c of the cluster
//   * copies its 1/8 slice of d_in -- the tile's x rows and the slot's A rows
//     -- and its 1/8 slice of d_out -- the tile's y rows and the slot's B rows
//     -- into shared memory with 16-byte cp.async issued by every thread
//     (completion tracked per stage on an mbarrier), all issued at once so the
//     whole working set is in flight. Rows are a few hundred bytes and
//     gathered by token, which one-row bulk copies serve poorly (each copy is
//     a separate TMA request); 128 threads issuing coalesced 16-byte copies
//     fill the rings in a few instructions per thread;
//   * computes its partial v over its d_in slice (mma m16n8k16, bf16 in, fp32
//     accumulate) and leaves it in its own shared memory;
//   * after a cluster barrier reads the 8 partials of the tile through
//     distributed shared memory, adds them in rank order (deterministic),
//     splits v into bf16 high and low parts and runs the expand MMAs for its
//     d_out slice, writing y once (fp32 add, one rounding). When the slice is
//     at most two stages (d_out <= 4096) the products B_s v are formed before
//     the wait on the previous kernel and parked in shared memory; after the
//     wait only the y rows (prefetched into L2) are loaded, updated and stored.
// No global flags; every wait for data is a bounded mbarrier wait (stage
// loads, and the exchange: each CTA arrives remotely on every peer's exchange
// barrier after pushing its partial), and a wait that gives up sets the error
// word and leaves the rows it guards unchanged. The two cluster barriers that
// remain only make sure that every CTA has started before a peer writes into
// it and has stopped writing into a peer before that peer exits; each CTA
// reaches both on every path, whatever its loads do.
// Each CTA also groups the batch itself (slot ids in shared memory, counts,
// prefix sums, warp ballots), so the step is a single launch; with
// programmatic dependent launch the next launch's CTAs are already resident
// when this one ends.
#include "device_util.cuh"
#include "kernels.cuh"

#include <cooperative_groups.h>

namespace lora {
namespace {

constexpr int kCl = 8;          // CTAs per cluster = slices of d_in and d_out
constexpr int kCT = 128;        // threads per CTA
constexpr int kCW = kCT / 32;
constexpr int kSW = 256;        // columns per pipeline stage (shrink and expand)
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr unsigned kFullMask = 0xffffffffu;

// Grouping scratch of the prologue. It lives in the partial-exchange buffer,
// which no peer writes before every CTA of the cluster has passed the
// prologue (the first cluster barrier).
struct GroupScratch {
    int cnt[kMaxSlots];
    int toff[kMaxSlots + 1];
    int rank[kMaxSlots];
    float scale[kMaxSlots];
    uint8_t eff[kFusedMaxTokens];          // slot of each token, 0xff = none
};

struct ClusterSmem {
    int tok[kTileTokens];
    int wcnt[kCW];                         // per-warp counts while collecting the tile's tokens
    uint64_t sbar[2], ebar[2];
    uint64_t xbar;                         // one remote arrival per CTA of the cluster once its partial is here
    int ntiles, invalid;
    float scale;                           // scale of this tile's slot
    uint32_t bad[kCl];                     // per source rank: its shrink data never arrived
};

// Dynamic shared memory of one CTA for a given number of 16-rank blocks.
// Region 1 holds the two shrink stages (x rows, A rows) and, once the shrink
// has consumed them, the two expand stages (y rows, B rows) in the same bytes.
__host__ __device__ constexpr size_t region1_bytes(int KB) {
    return 2 * (size_t)kTileTokens * kSW * 2 + 2 * (size_t)KB * 16 * kSW * 2;
}
__host__ __device__ constexpr size_t dyn_bytes(int KB) {
    return region1_bytes(KB)
           + (size_t)kCl * kTileTokens * KB * 16 * 4   // partials pushed by the 8 ranks
           + (size_t)kCW * KB * 8 * 32 * 4;             // cross-warp sums of the shrink, then v
}
static_assert(sizeof(GroupScratch) <= (size_t)kCl * kTileTokens * 16 * 4, "grouping scratch fits");

template <int KB>
struct Dyn {
    uint16_t *xs, *as, *ys, *bs;
    float *vpart;                            // [kCl][16][KB*16] partials pushed by each rank
    float *red;                              // [kCW][KB*8][32]
    float *vsum;                             // [16][KB*16], in `red` once the partials are pushed
    GroupScratch *g;                         // prologue only, aliases vpart
    __device__ Dyn(uint8_t *base) {
        xs = reinterpret_cast<uint16_t *>(base);
        as = xs + 2 * kTileTokens * kSW;
        ys = xs;                                             // after the shrink
        bs = xs + 2 * kTileTokens * kSW;                     // after the shrink
        vpart = reinterpret_cast<float *>(base + region1_bytes(KB));
        red = vpart + kCl * kTileTokens * KB * 16;
        vsum = red;
        g = reinterpret_cast<GroupScratch *>(vpart);
    }
};

__device__ __forceinline__ uint4 lds128(const uint16_t *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint2 lds64(const uint16_t *p) { return *reinterpret_cast<const uint2 *>(p); }

struct Tile {
    int s, cnt, r;
};

// Shared-memory offset of element (row, col) of a 256-column stage row: the
// 16-byte chunk index is XORed with 4 on odd rows, so the two rows read by one
// 8-lane phase of an MMA fragment load fall in disjoint bank groups.
__device__ __forceinline__ int swz(int row, int col) {
    return row * kSW + ((((col >> 3) ^ ((row & 1) << 2)) << 3) | (col & 7));
}

// Shared-memory offset of element (P, k) of a stage's B rows (R elements per
// row, k a multiple of 4). The mapping spreads the rows {P, P+1, P+8, P+9}
// that one 16-lane phase of the expand reads over distinct bank groups:
// R = 16 permutes rows inside each group of 16, R = 32 and R = 64 XOR the
// 16-byte chunk index with bits of P. Other ranks are stored unswizzled.
__device__ __forceinline__ int bsw(int P, int k, int R) {
    if (R == 16) return (P ^ (((P >> 3) & 1) << 1)) * 16 + k;
    int ch = k >> 3;
    if (R == 32) ch ^= ((P >> 3) & 1) << 1;
    else if (R == 64) ch ^= ((P & 1) | (((P >> 3) & 1) << 1)) << 1;
    return P * R + (ch << 3) + (k & 7);
}

// Products B_s v for one warp's 64 columns [c0, c0 + 64) of an expand stage:
// two 32-column groups of four 8-column MMA blocks. Every B fragment is read
// first; then, for each 16-rank block, the high-part MMAs of all eight column
// blocks are issued, and after them the low-part ones. Each accumulator still
// adds high before low, rank block by rank block, so the sums are those of a
// one-block-at-a-time loop, but eight independent MMAs go out back to back
// instead of each waiting on its dependent partner and on its own B load.
template <int KB>
__device__ __forceinline__ void expand_products(const uint16_t *bs, int c0, int w, int R, int r, int nmb,
                                                const uint32_t (&ahi)[KB][4], const uint32_t (&alo)[KB][4],
                                                int gq, int tq, float (&acc)[2][4][4]) {
    uint2 bfr[2][4][KB];
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) {
            const int P = c0 + grp * 32 + 8 * (gq >> 1) + 2 * jn + (gq & 1);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                const int k = kb * 16 + 4 * tq;
                uint2 bb = (kb < nmb && P < w && k < R) ? lds64(bs + bsw(P, k, R)) : make_uint2(0, 0);
                if (k + 4 > r) {               // ranks at or past r contribute nothing
                    if (k + 0 >= r) bb.x &= 0xffff0000u;
                    if (k + 1 >= r) bb.x &= 0x0000ffffu;
                    if (k + 2 >= r) bb.y &= 0xffff0000u;
                    if (k + 3 >= r) bb.y &= 0x0000ffffu;
                }
                bfr[grp][jn][kb] = bb;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[grp][jn][q] = 0.f;
        }
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
        if (kb >= nmb) break;
#pragma unroll
        for (int grp = 0; grp < 2; ++grp)
#pragma unroll
            for (int jn = 0; jn < 4; ++jn)
                mma_bf16(acc[grp][jn], ahi[kb][0], ahi[kb][1], ahi[kb][2], ahi[kb][3], bfr[grp][jn][kb].x,
                         bfr[grp][jn][kb].y);
#pragma unroll
        for (int grp = 0; grp < 2; ++grp)
#pragma unroll
            for (int jn = 0; jn < 4; ++jn)
                mma_bf16(acc[grp][jn], alo[kb][0], alo[kb][1], alo[kb][2], alo[kb][3], bfr[grp][jn][kb].x,
                         bfr[grp][jn][kb].y);
    }
}

// Shrink stage j: x rows of the tile and A rows of the slot, columns [ks, ks + w).
template <int KB>
__device__ void issue_shrink(const LayerArgs &L, const ClusterSmem &sm, Dyn<KB> &d, const Tile &t,
                             int R, int k0, int k1, int j, uint64_t *bar) {
    const int b = j & 1;
    const int ks = k0 + j * kSW, w = min(kSW, k1 - ks);
    const int cpr = w >> 3;                 // 16-byte chunks per row
    const uint16_t *x = static_cast<const uint16_t *>(L.x);
    const uint16_t *A = static_cast<const uint16_t *>(L.A) + (size_t)t.s * R * L.d_in;
    uint16_t *xs = d.xs + b * kTileTokens * kSW;
    uint16_t *as = d.as + b * KB * 16 * kSW;
    const int total = (t.cnt + t.r) * cpr;
    auto issue = [&](int row, int col) {
        if (row < t.cnt)
            cp_async16(xs + swz(row, col), x + (size_t)sm.tok[row] * L.d_in + ks + col);
        else
            cp_async16(as + swz(row - t.cnt, col), A + (size_t)(row - t.cnt) * L.d_in + ks + col);
    };
    if (cpr == kSW / 8) {                   // a full stage: row and column by shifts
        for (int e = threadIdx.x; e < total; e += kCT) issue(e >> 5, (e & 31) << 3);
    } else {
        for (int e = threadIdx.x; e < total; e += kCT) {
            const int row = e / cpr;
            issue(row, (e - row * cpr) * 8);
        }
    }
    cp_async_arrive_noinc(bar);
}

// Expand stage j: y rows of the tile and B rows [os, os + w) of the slot.
// parts: 1 = B rows only (no arrival yet), 2 = y rows and the stage arrival,
// 3 = both. Splitting lets B be fetched before the wait on the previous kernel.
template <int KB>
__device__ void issue_expand(const LayerArgs &L, const ClusterSmem &sm, Dyn<KB> &d, const Tile &t,
                             int R, int o0, int o1, int j, uint64_t *bar, int parts = 3) {
    const int b = j & 1;
    const int os = o0 + j * kSW, w = min(kSW, o1 - os);
    const int cpr = w >> 3;
    const uint16_t *y = static_cast<const uint16_t *>(L.y);
    const uint16_t *B = static_cast<const uint16_t *>(L.B) + (size_t)t.s * L.d_out * R;   // the slot's B
    uint16_t *ys = d.ys + b * kTileTokens * kSW;
    uint16_t *bs = d.bs + (size_t)b * kSW * KB * 16;
    if (parts & 1) {
        // rows os .. os + w - 1 of every rank block (blocks of kb ranks, each
        // [d_out][kb] contiguous): chunk e of a block is row e / (kb / 8),
        // ranks blk * kb + 8 (e % (kb / 8)) ..
        const int kb = b_block(R), cpr = kb >> 3, cs = kb == 32 ? 2 : (kb == 16 ? 1 : 0);
        for (int blk = 0; blk * kb < t.r; ++blk) {           // the slot's blocks (ranks past r: masked)
            const uint16_t *src = B + ((size_t)blk * L.d_out + os) * kb;
            for (int e = threadIdx.x; e < w * cpr; e += kCT) {
                const int P = e >> cs, k = blk * kb + ((e & (cpr - 1)) << 3);
                cp_async16(bs + bsw(P, k, R), src + (size_t)e * 8);
            }
        }
    }
    if (parts & 2) {
        if (cpr == kSW / 8) {
            for (int e = threadIdx.x; e < t.cnt * cpr; e += kCT) {
                const int row = e >> 5, col = (e & 31) << 3;
                cp_async16(ys + swz(row, col), y + (size_t)sm.tok[row] * L.d_out + os + col);
            }
        } else {
            for (int e = threadIdx.x; e < t.cnt * cpr; e += kCT) {
                const int row = e / cpr, col = (e - row * cpr) * 8;
                cp_async16(ys + swz(row, col), y + (size_t)sm.tok[row] * L.d_out + os + col);
            }
        }
        cp_async_arrive_noinc(bar);
    }
}

// Resident CTAs per SM the register budget must allow (the shared memory of
// one CTA permits that many): rank 16 fits five, so two consecutive decode
// steps' CTAs can be resident together under programmatic dependent launch.
constexpr int min_blocks(int KB) { return KB == 1 ? 5 : (KB == 2 ? 3 : 1); }

template <int KB>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kCT, min_blocks(KB))
decode_cluster_kernel(const __grid_constant__ FusedArgs fa) {
    __shared__ ClusterSmem sm;
    extern __shared__ __align__(128) uint8_t dyn_raw[];
    Dyn<KB> d(dyn_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, gq = lane >> 2, tq = lane & 3;
    const int T = fa.T, S = fa.S, R = fa.R;
    const int tile = blockIdx.x / kCl;
    const int crank = (int)cluster_ctarank();
    const LayerArgs &L = fa.l[blockIdx.y];

    // Inputs may come from the previous kernel in the stream: wait for it, then
    // let the next launch start filling free SMs. With fa.early the caller has
    // declared that only y can be written by that kernel: everything else is
    // read before the wait, y after it.
    if (!fa.early) grid_dependency_wait();
    grid_launch_dependents();

    // ---- group the batch by slot (every CTA, from shared memory) ----------
    constexpr int kPer = kFusedMaxTokens / kCT;
    int raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int t = tid + i * kCT;
        raw[i] = t < T ? __ldg(fa.idx + t) : -1;
    }
    for (int s = tid; s < S; s += kCT) {
        d.g->rank[s] = fa.rank[s];
        d.g->scale[s] = fa.scale[s];
        d.g->cnt[s] = 0;
    }
    if (tid == 0) {
        sm.invalid = 0;
        mbar_init(&sm.sbar[0], kCT);
        mbar_init(&sm.sbar[1], kCT);
        mbar_init(&sm.ebar[0], kCT);
        mbar_init(&sm.ebar[1], kCT);
        mbar_init(&sm.xbar, kCl);
        fence_mbar_init();
    }
    __syncthreads();
    int inv = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int t = tid + i * kCT;
        if (i * kCT >= T) break;            // uniform across the CTA
        const int r = raw[i];
        const bool ok = t < T && r >= 0 && r < S && d.g->rank[r] > 0;
        if (t < T) {
            inv += (r < -1 || r >= S);
            d.g->eff[t] = ok ? (uint8_t)r : (uint8_t)0xff;
        }
        // one shared atomic per distinct slot per warp
        const unsigned peers = __match_any_sync(kFullMask, ok ? r : -2 - lane);
        if (ok && lane == __ffs(peers) - 1) atomicAdd(&d.g->cnt[r], __popc(peers));
    }
    if (inv) atomicAdd(&sm.invalid, inv);
    __syncthreads();
    // Tiles per slot, their prefix, and this tile's slot. With at most 32 slots
    // every warp does this in registers (one lane per slot, no barrier);
    // beyond that warp 0 scans through shared memory.
    int ntiles, lo, toff_lo;
    if (S <= 32) {
        const int c = lane < S ? d.g->cnt[lane] : 0;
        const int nt = (c + kTileTokens - 1) / kTileTokens;
        int it = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a2 = __shfl_up_sync(kFullMask, it, o);
            if (lane >= o) it += a2;
        }
        ntiles = __shfl_sync(kFullMask, it, 31);
        const int tex = it - nt;            // first tile of slot `lane`
        // the slot whose tiles hold `tile`: the last one that has tiles and
        // starts at or before it
        const unsigned cand = __ballot_sync(kFullMask, nt > 0 && tex <= tile);
        lo = cand ? 31 - __clz(cand) : 0;
        toff_lo = __shfl_sync(kFullMask, tex, lo);
    } else {
        if (warp == 0) {
            int carry_t = 0;
            for (int base = 0; base < S; base += 32) {
                const int s = base + lane;
                const int c = s < S ? d.g->cnt[s] : 0;
                const int nt = (c + kTileTokens - 1) / kTileTokens;
                int it = nt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int a2 = __shfl_up_sync(kFullMask, it, o);
                    if (lane >= o) it += a2;
                }
                if (s < S) d.g->toff[s] = carry_t + it - nt;
                carry_t += __shfl_sync(kFullMask, it, 31);
            }
            if (lane == 0) {
                d.g->toff[S] = carry_t;
                sm.ntiles = carry_t;
            }
        }
        __syncthreads();
        ntiles = sm.ntiles;
        lo = 0;
        int hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (d.g->toff[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        toff_lo = d.g->toff[lo];
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0 && sm.invalid)
        atomicAdd(fa.hdr + kHdrInvalid, sm.invalid);
    if (tile >= ntiles) return;             // the whole cluster leaves together

    // ---- this tile: slot, tokens -----------------------------------------
    Tile t;
    {
        t.s = lo;
        const int first = (tile - toff_lo) * kTileTokens;
        t.cnt = min(kTileTokens, d.g->cnt[lo] - first);
        t.r = d.g->rank[lo];
        if (tid == 0) sm.scale = d.g->scale[lo];
        // The (first + i)-th token on slot lo, in original order: every warp
        // takes 32 tokens of a 128-token block (one ballot each), the warp
        // counts meet in shared memory, and a running count carries the
        // blocks before; the loop stops once the tile's tokens are found.
        {
            const unsigned lt = (1u << lane) - 1u;
            int seen = 0;                   // the same in every thread
            for (int base = 0; base < T && seen < first + kTileTokens; base += kCT) {
                const int tk = base + tid;
                const bool m = tk < T && d.g->eff[tk] == (uint8_t)lo;
                const unsigned bal = __ballot_sync(kFullMask, m);
                if (lane == 0) sm.wcnt[warp] = __popc(bal);
                __syncthreads();
                int before = seen + __popc(bal & lt), total = 0;
#pragma unroll
                for (int w2 = 0; w2 < kCW; ++w2) {
                    const int c = sm.wcnt[w2];
                    before += w2 < warp ? c : 0;
                    total += c;
                }
                if (m && before >= first && before < first + kTileTokens) sm.tok[before - first] = tk;
                seen += total;
                __syncthreads();            // wcnt is rewritten by the next block
            }
        }
    }
    __syncthreads();
    // The grouping scratch is dead from here on: let peers know this CTA runs
    // (distributed shared memory may be written only after that).
    cluster_arrive_relaxed();
    const int nmb = (t.r + 15) >> 4;
    const int k0 = crank * L.chunk_cols, k1 = min(L.d_in, k0 + L.chunk_cols);
    const int o0 = crank * L.out_cols, o1 = min(L.d_out, o0 + L.out_cols);
    const int nks = k1 > k0 ? (k1 - k0 + kSW - 1) / kSW : 0;
    const int nes = o1 > o0 ? (o1 - o0 + kSW - 1) / kSW : 0;

    // ---- issue everything that fits in the stage rings --------------------
    for (int j = 0; j < nks && j < 2; ++j) issue_shrink<KB>(L, sm, d, t, R, k0, k1, j, &sm.sbar[j]);
    // The slot's B rows of this slice and the tile's y rows are read only
    // after the shrink and the exchange: asking L2 for them now, behind the
    // shrink's loads, takes their DRAM latency out of the chain that follows.
    // A prefetch changes nothing a load observes (L2 is where every SM's
    // stores land), so y may still be written by the kernel before this one.
    if (nes > 0) {
        if (tid < t.cnt)
            prefetch_l2_bulk(static_cast<const uint16_t *>(L.y) + (size_t)sm.tok[tid] * L.d_out + o0,
                             (uint32_t)(o1 - o0) * 2u);
        // rows o0 .. o1 - 1 of each of the slot's rank blocks
        const int kb = b_block(R), pb = kCT - 1 - tid;
        if (pb * kb < t.r)
            prefetch_l2_bulk(static_cast<const uint16_t *>(L.B) + ((size_t)t.s * L.d_out * R +
                                                                   ((size_t)pb * L.d_out + o0) * kb),
                             (uint32_t)(o1 - o0) * (uint32_t)kb * 2u);
    }
    bool ok = true;

    // ---- shrink over this CTA's d_in slice ---------------------------------
    float acc[KB][2][4];
#pragma unroll
    for (int m = 0; m < KB; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][n][q] = 0.f;
    for (int j = 0; j < nks; ++j) {
        const int b = j & 1;
        ok = mbar_wait_bounded(&sm.sbar[b], (j >> 1) & 1, kWaitLimit) && ok;
        const int w = min(kSW, k1 - (k0 + j * kSW));
        const uint16_t *xs = d.xs + b * kTileTokens * kSW;
        const uint16_t *as = d.as + b * KB * 16 * kSW;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            // The MMAs are warp-wide, so the test that skips a step is too:
            // a lane whose 8 columns lie past the slice (its last step can end
            // inside the 32 columns, w being a multiple of 8 only) takes zeros.
            const int cb = warp * 64 + step * 32;
            if (cb < w) {
                const int cc = cb + 8 * tq;
                const bool in = cc < w;
                const uint4 z = make_uint4(0, 0, 0, 0);
                const uint4 xa = in ? lds128(xs + swz(gq, cc)) : z;
                const uint4 xb = in ? lds128(xs + swz(gq + 8, cc)) : z;
                // A fragments of every rank block first; then the first halves
                // of K for every accumulator and after them the second halves
                // (each accumulator adds in the same order, and no MMA waits on
                // the one issued just before it)
                uint4 a0[KB], a1[KB];
#pragma unroll
                for (int m = 0; m < KB; ++m) {
                    a0[m] = (in && m < nmb) ? lds128(as + swz(m * 16 + gq, cc)) : z;
                    a1[m] = (in && m < nmb) ? lds128(as + swz(m * 16 + gq + 8, cc)) : z;
                }
#pragma unroll
                for (int m = 0; m < KB; ++m) {
                    if (m < nmb) {
                        mma_bf16(acc[m][0], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xa.x, xa.y);
                        mma_bf16(acc[m][1], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xb.x, xb.y);
                    }
                }
#pragma unroll
                for (int m = 0; m < KB; ++m) {
                    if (m < nmb) {
                        mma_bf16(acc[m][0], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xa.z, xa.w);
                        mma_bf16(acc[m][1], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xb.z, xb.w);
                    }
                }
            }
        }
        __syncthreads();                    // stage buffer b free again
        if (j + 2 < nks) issue_shrink<KB>(L, sm, d, t, R, k0, k1, j + 2, &sm.sbar[b]);
    }

    // The shrink stages are consumed: the same bytes now receive the expand
    // stages. B never depends on the previous kernel; y may (fa.early waits
    // for it once the partials of v have been exchanged).
    __syncthreads();
    for (int j = 0; j < nes && j < 2; ++j) issue_expand<KB>(L, sm, d, t, R, o0, o1, j, &sm.ebar[j], 1);

    // Cross-warp sum into this CTA's partial v[token][k].
    float *red = d.red;
#pragma unroll
    for (int m = 0; m < KB; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) red[(warp * KB * 8 + (m * 2 + n) * 4 + q) * 32 + lane] = acc[m][n][q];
    __syncthreads();
    // Sum the 4 warps and push this CTA's partial (4 consecutive ranks per
    // store) into slot `crank` of every peer's shared memory.
    cluster_wait_acquire();                 // every peer has started and left its prologue
    {
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        constexpr int RK = KB * 16;
        for (int e = tid; e < kTileTokens * (RK / 4); e += kCT) {
            const int tk = e / (RK / 4), k4 = (e % (RK / 4)) * 4;
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = k4 + i, m = k >> 4, kk = k & 15;
                const int ln = (kk & 7) * 4 + ((tk & 7) >> 1);
                const int sj = (m * 2 + (tk >> 3)) * 4 + (kk >> 3) * 2 + (tk & 1);
                float a = 0.f;
#pragma unroll
                for (int ww = 0; ww < kCW; ++ww) a += red[(ww * KB * 8 + sj) * 32 + ln];
                v[i] = a;
            }
            const float4 v4 = make_float4(v[0], v[1], v[2], v[3]);
            float *slot = d.vpart + (crank * kTileTokens + tk) * RK + k4;
#pragma unroll
            for (int p = 0; p < kCl; ++p)
                *reinterpret_cast<float4 *>(cluster.map_shared_rank(slot, (unsigned)p)) = v4;
        }
        if (tid < kCl) *cluster.map_shared_rank(&sm.bad[crank], (unsigned)tid) = ok ? 0u : 1u;
    }
    // Every thread's stores into the peers are done; thread p then arrives on
    // peer p's exchange barrier (release at cluster scope), and each CTA waits
    // on its own barrier for the 8 arrivals with the usual iteration limit.
    // The cluster barrier arrived on here is waited on only before exit, so
    // that no CTA leaves while a peer may still write into it; it waits for
    // peers to reach this point, never for data.
    __syncthreads();
    if (tid < kCl) mbar_arrive_remote(map_peer(smem_u32(&sm.xbar), (uint32_t)tid));
    cluster_arrive_release();
    if (!mbar_wait_bounded_cluster(&sm.xbar, 0, kWaitLimit)) ok = false;

    // ---- v = sum of the 8 partials in rank order (deterministic) -----------
    for (int e = tid; e < kTileTokens * KB * 16; e += kCT) {
        float a = 0.f;
#pragma unroll
        for (int p = 0; p < kCl; ++p) a += d.vpart[p * kTileTokens * KB * 16 + e];
        d.vsum[e] = a;
    }
    __syncthreads();
    uint32_t ahi[KB][4], alo[KB][4];
    {
#pragma unroll
        for (int p = 0; p < kCl; ++p)
            if (sm.bad[p]) ok = false;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            float f[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const int k = kb * 16 + 4 * tq;
            if (kb < nmb) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 q = *reinterpret_cast<const float4 *>(d.vsum + (gq + 8 * h) * KB * 16 + k);
                    f[h][0] = q.x;
                    f[h][1] = q.y;
                    f[h][2] = q.z;
                    f[h][3] = q.w;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (k + i >= t.r || gq + 8 * h >= t.cnt) f[h][i] = 0.f;
            }
            float hi[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) hi[h][i] = round_bf16(f[h][i]);
            ahi[kb][0] = pack_bf16(hi[0][0], hi[0][1]);
            ahi[kb][1] = pack_bf16(hi[1][0], hi[1][1]);
            ahi[kb][2] = pack_bf16(hi[0][2], hi[0][3]);
            ahi[kb][3] = pack_bf16(hi[1][2], hi[1][3]);
            alo[kb][0] = pack_bf16(f[0][0] - hi[0][0], f[0][1] - hi[0][1]);
            alo[kb][1] = pack_bf16(f[1][0] - hi[1][0], f[1][1] - hi[1][1]);
            alo[kb][2] = pack_bf16(f[0][2] - hi[0][2], f[0][3] - hi[0][3]);
            alo[kb][3] = pack_bf16(f[1][2] - hi[1][2], f[1][3] - hi[1][3]);
        }
    }

    const float scale = sm.scale;
    const int tok0 = gq < t.cnt ? sm.tok[gq] : -1;
    const int tok1 = gq + 8 < t.cnt ? sm.tok[gq + 8] : -1;
    uint16_t *yg = static_cast<uint16_t *>(L.y);
    const int d_out = L.d_out;

    // ---- short path: this CTA's d_out slice is at most two stages ----------
    // The products B_s v do not depend on y, so they are formed here, before
    // the wait on the previous kernel, and parked as fp32 in region 1 (slots
    // private to each thread: float4 index (stage * 8 + i) * kCT + tid). After
    // the wait only the y rows are read, straight into registers, updated with
    // the same fma and rounding as below, and written back.
    if (nes <= 2) {
        cp_async_wait_all();                // this thread's B rows have landed
        __syncthreads();                    // and everyone else's
        float4 *dl = reinterpret_cast<float4 *>(d.xs);
        float4 keep[8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (j >= nes) break;
            const int w = min(kSW, o1 - (o0 + j * kSW));
            const uint16_t *bs = d.bs + (size_t)j * kSW * KB * 16;
            float acc2[2][4][4];
            expand_products<KB>(bs, warp * 64, w, R, t.r, nmb, ahi, alo, gq, tq, acc2);
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float(&a)[4][4] = acc2[grp];
                    const float4 f0 = make_float4(a[0][2 * h], a[0][2 * h + 1], a[1][2 * h], a[1][2 * h + 1]);
                    const float4 f1 = make_float4(a[2][2 * h], a[2][2 * h + 1], a[3][2 * h], a[3][2 * h + 1]);
                    const int i = grp * 4 + h * 2;
                    if (j == 0) {
                        dl[i * kCT + tid] = f0;
                        dl[(i + 1) * kCT + tid] = f1;
                    } else {
                        keep[i] = f0;
                        keep[i + 1] = f1;
                    }
                }
            }
        }
        __syncthreads();                    // every read of the B rows is done
        if (nes == 2) {
#pragma unroll
            for (int i = 0; i < 8; ++i) dl[(8 + i) * kCT + tid] = keep[i];
        }
        if (fa.early) grid_dependency_wait();
        uint4 yv[2][2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int grp = 0; grp < 2; ++grp)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int os = o0 + j * kSW, cc = warp * 64 + grp * 32 + 8 * tq;
                    const int tok = h ? tok1 : tok0;
                    yv[j][grp][h] = (j < nes && cc < o1 - os && tok >= 0)
                                        ? __ldcg(reinterpret_cast<const uint4 *>(yg + (size_t)tok * d_out + os + cc))
                                        : make_uint4(0, 0, 0, 0);
                }
        if (ok) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int grp = 0; grp < 2; ++grp)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int os = o0 + j * kSW, cc = warp * 64 + grp * 32 + 8 * tq;
                        const int tok = h ? tok1 : tok0;
                        if (j >= nes || cc >= o1 - os || tok < 0) continue;
                        const int i = j * 8 + grp * 4 + h * 2;
                        const float4 f0 = dl[i * kCT + tid], f1 = dl[(i + 1) * kCT + tid];
                        const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                        uint32_t wv[4] = {yv[j][grp][h].x, yv[j][grp][h].y, yv[j][grp][h].z, yv[j][grp][h].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            wv[q] = pack_bf16(fmaf(scale, f[2 * q], bf_lo(wv[q])), fmaf(scale, f[2 * q + 1], bf_hi(wv[q])));
                        *reinterpret_cast<uint4 *>(yg + (size_t)tok * d_out + os + cc) =
                            make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
        }
        if (!ok && tid == 0) atomicExch(fa.hdr + kHdrError, 1);
        cluster_wait_acquire();             // no peer writes into this CTA any more
        return;
    }

    // Everything so far depends only on inputs the caller declared ready
    // (fa.early): the partial exchange ran before the wait, so after it only
    // the y rows are fetched, updated and written.
    if (fa.early) grid_dependency_wait();
    for (int j = 0; j < nes && j < 2; ++j) issue_expand<KB>(L, sm, d, t, R, o0, o1, j, &sm.ebar[j], 2);

    // ---- expand over this CTA's d_out slice --------------------------------
    for (int j = 0; j < nes; ++j) {
        const int b = j & 1;
        const bool got = mbar_wait_bounded(&sm.ebar[b], (j >> 1) & 1, kWaitLimit);
        ok = got && ok;
        const int os = o0 + j * kSW, w = min(kSW, o1 - os);
        const uint16_t *ys = d.ys + b * kTileTokens * kSW;
        const uint16_t *bs = d.bs + (size_t)b * kSW * KB * 16;
        // y fragments first, then the products, then the stores
        uint4 yv[2][2];
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int cc = warp * 64 + grp * 32 + 8 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                yv[grp][h] = (cc < w && gq + 8 * h < t.cnt) ? lds128(ys + swz(gq + 8 * h, cc))
                                                             : make_uint4(0, 0, 0, 0);
        }
        float acc[2][4][4];
        expand_products<KB>(bs, warp * 64, w, R, t.r, nmb, ahi, alo, gq, tq, acc);
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int c = warp * 64 + grp * 32;          // stage-local first column
            const float(&acc2)[4][4] = acc[grp];
            const int cc = c + 8 * tq;
            if (cc >= w || !ok) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tok = h ? tok1 : tok0;
                if (tok < 0) continue;
                uint32_t wv[4] = {yv[grp][h].x, yv[grp][h].y, yv[grp][h].z, yv[grp][h].w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    wv[q] = pack_bf16(fmaf(scale, acc2[q][2 * h], bf_lo(wv[q])),
                                      fmaf(scale, acc2[q][2 * h + 1], bf_hi(wv[q])));
                *reinterpret_cast<uint4 *>(yg + (size_t)tok * d_out + os + cc) =
                    make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
        }
        __syncthreads();
        if (j + 2 < nes) issue_expand<KB>(L, sm, d, t, R, o0, o1, j + 2, &sm.ebar[b]);
    }
    if (!ok && tid == 0) atomicExch(fa.hdr + kHdrError, 1);
    cluster_wait_acquire();                 // no peer writes into this CTA any more
}

// The exchange wait of decode_cluster_kernel on a barrier that nothing
// arrives on: the same barrier setup, remote-arrival count, cluster-scope
// bounded wait and exit barrier, in a two-CTA cluster. Each CTA that gives up
// adds one to `gave_up` and sets the error word, then leaves normally.
__global__ void __cluster_dims__(2, 1, 1) selftest_cluster_wait_kernel(int *err_word, int *gave_up,
                                                                       uint32_t limit) {
    __shared__ uint64_t xbar;
    if (threadIdx.x == 0) {
        mbar_init(&xbar, kCl);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();
    cluster_wait_acquire();
    cluster_arrive_release();
    const bool done = mbar_wait_bounded_cluster(&xbar, 0, limit);
    if (!done && threadIdx.x == 0) {
        atomicAdd(gave_up, 1);
        atomicExch(err_word, 1);
    }
    cluster_wait_acquire();
}

}  // namespace

cudaError_t launch_selftest_cluster_wait(int *err_word, int *gave_up, uint32_t limit, cudaStream_t st) {
    selftest_cluster_wait_kernel<<<2, 32, 0, st>>>(err_word, gave_up, limit);
    return cudaGetLastError();
}

int cluster_decode_kb(int R) { return R <= 16 ? 1 : (R <= 32 ? 2 : 4); }

size_t cluster_decode_smem(int R) { return dyn_bytes(cluster_decode_kb(R)); }

template <int KB>
static cudaError_t launch_cluster_kb(const FusedArgs &fa, int tiles, cudaStream_t st, bool pdl) {
    static std::atomic<uint64_t> attr_done{0};
    const size_t smem = dyn_bytes(KB);
    if (!device_bit(attr_done)) {
        cudaError_t e = cudaFuncSetAttribute(decode_cluster_kernel<KB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        set_device_bit(attr_done);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(tiles * kCl), (unsigned)fa.n, 1);
    cfg.blockDim = dim3(kCT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_cluster_kernel<KB>, fa);
}

cudaError_t launch_cluster_decode(const FusedArgs &fa, int tiles, cudaStream_t st, bool pdl) {
    switch (cluster_decode_kb(fa.R)) {
    case 1: return launch_cluster_kb<1>(fa, tiles, st, pdl);
    case 2: return launch_cluster_kb<2>(fa, tiles, st, pdl);
    default: return launch_cluster_kb<4>(fa, tiles, st, pdl);
    }
}

}  // namespace lora
