// Fused decode step: token grouping, shrink and expand-add of every layer of a
// layer set in ONE launch, for batches of at most kFusedMaxTokens tokens.
//
//   v[t][k]  = sum_j A_s[k][j] x[t][j]                      (k < r_s)
//   y[t][i] += (lora_alpha_s / r_s) * sum_k B_s[i][k] v[t][k]
//
// (the LoRA delta with the PEFT fields r / lora_alpha, "vLLM LoRA Resolver
// 插件详解" page, section 3.2; several slots per batch, max_loras and
// max_lora_rank from the "Multi-LoRA 适配器缓存生产实战" page, section 核心原理.)
//
// A decode batch moves only a few MB per layer, so the cost of three dependent
// launches (group, shrink, expand) dominates. Here every CTA of a grid that is
// fully resident on the GPU:
//   1. loads the slot ids into shared memory and groups tokens by slot itself
//      (counts, prefix sums; each tile's token list by warp ballots);
//   2. issues the loads of its first expand item (y rows, B_s fragments) into
//      registers, so that the y stream overlaps the shrink;
//   3. runs its shrink items (tile of <= 16 same-slot tokens x one d_in chunk,
//      mma m16n8k16), writes the chunk partial and publishes a per-(tile,
//      chunk) flag with a release store;
//   4. for each expand item waits (bounded) for the flags of its tile, sums the
//      chunk partials in chunk order (deterministic), splits v into bf16 high
//      and low parts, runs the MMAs and writes y once (fp32 add, one rounding).
// Flags carry a per-context epoch (launch count) so they never need clearing.
// Every CTA finishes its shrink items before it waits, and all CTAs are
// resident, so every wait is for work that is running; waits still give up
// after kSpinLimit polls, set the error word and skip the affected rows.
#include "device_util.cuh"
#include "kernels.cuh"

namespace lora {
namespace {

constexpr int kFT = 128;
constexpr int kFW = kFT / 32;
constexpr int kECols = 256;
constexpr unsigned kSpinLimit = 1u << 20;
constexpr unsigned kFull = 0xffffffffu;

struct FusedSmem {
    int16_t eff[kFusedMaxTokens];
    int cnt[kMaxSlots];
    int off[kMaxSlots + 1];
    int toff[kMaxSlots + 1];
    int rank[kMaxSlots];
    float scale[kMaxSlots];
    int tok_s[kTileTokens];
    int tok_e[kTileTokens];
    float red[kFW][32][32];
    int ntiles, invalid, ok;
    unsigned epoch;
};

struct TileInfo {
    int s, pos0, cnt, r, first;
};

__device__ __forceinline__ TileInfo tile_info(const FusedSmem &sm, int S, int tile) {
    int lo = 0, hi = S - 1;                  // largest s with toff[s] <= tile
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (sm.toff[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    TileInfo ti;
    ti.s = lo;
    ti.first = (tile - sm.toff[lo]) * kTileTokens;
    ti.pos0 = sm.off[lo] + ti.first;
    ti.cnt = min(kTileTokens, sm.cnt[lo] - ti.first);
    ti.r = sm.rank[lo];
    return ti;
}

// Warp-wide: dst[i] = the (first + i)-th token (original order) on slot s.
__device__ __forceinline__ void find_tokens(const FusedSmem &sm, int T, int s, int first, int *dst,
                                            int lane) {
    const unsigned lt = (1u << lane) - 1u;
    int seen = 0;
    for (int base = 0; base < T && seen < first + kTileTokens; base += 32) {
        const int t = base + lane;
        const bool m = t < T && sm.eff[t] == s;
        const unsigned bal = __ballot_sync(kFull, m);
        const int before = seen + __popc(bal & lt);
        if (m && before >= first && before < first + kTileTokens) dst[before - first] = t;
        seen += __popc(bal);
    }
}

__device__ __forceinline__ void decode_item(const FusedArgs &fa, int ntiles, int item, bool expand,
                                            int &l, int &tile, int &sub) {
    for (l = 0; l < fa.n; ++l) {
        const int per = expand ? (fa.l[l].d_out + kECols - 1) / kECols : fa.l[l].n_chunks;
        const int n = ntiles * per;
        if (item < n) {
            tile = item % ntiles;
            sub = item / ntiles;
            return;
        }
        item -= n;
    }
    l = tile = sub = -1;
}

// --------------------------------------------------------------------------
// Shrink item: tokens of one tile x one d_in chunk -> chunk partial + flag.
// --------------------------------------------------------------------------
template <int KB>
__device__ void shrink_item(const FusedArgs &fa, FusedSmem &sm, int l, int tile, int chunk,
                            unsigned target) {
    const LayerArgs &L = fa.l[l];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, tq = lane & 3;
    const TileInfo ti = tile_info(sm, fa.S, tile);
    if (warp == 0) find_tokens(sm, fa.T, ti.s, ti.first, sm.tok_s, lane);
    __syncthreads();
    const int tok0 = gq < ti.cnt ? sm.tok_s[gq] : -1;
    const int tok1 = gq + 8 < ti.cnt ? sm.tok_s[gq + 8] : -1;
    const int d_in = L.d_in, R = fa.R, r = ti.r;
    const int nmb = (r + 15) >> 4;
    const uint16_t *x = static_cast<const uint16_t *>(L.x);
    const uint16_t *xr0 = x + (size_t)(tok0 < 0 ? 0 : tok0) * d_in;
    const uint16_t *xr1 = x + (size_t)(tok1 < 0 ? 0 : tok1) * d_in;
    const uint16_t *As = static_cast<const uint16_t *>(L.A) + (size_t)ti.s * R * d_in;

    float acc[KB][2][4];
#pragma unroll
    for (int m = 0; m < KB; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][n][j] = 0.f;

    constexpr int ITB = KB == 1 ? 4 : 2;      // 32-column steps whose loads are in flight together
    const int c0 = chunk * L.chunk_cols;
    const int c1 = min(d_in, c0 + L.chunk_cols);
    for (int colb = c0 + warp * 32; colb < c1; colb += ITB * kFW * 32) {
        uint4 xa[ITB], xb[ITB], a0[ITB][KB], a1[ITB][KB];
#pragma unroll
        for (int it = 0; it < ITB; ++it) {
            const int col = colb + it * kFW * 32;
            const bool in = col < c1;
            const int cc = col + 8 * tq;
            xa[it] = load8_bf16(xr0, cc, d_in, in && tok0 >= 0, 1);
            xb[it] = load8_bf16(xr1, cc, d_in, in && tok1 >= 0, 1);
#pragma unroll
            for (int m = 0; m < KB; ++m) {
                const int k0 = m * 16 + gq, k1 = k0 + 8;
                a0[it][m] = load8_bf16(As + (size_t)k0 * d_in, cc, d_in, in && m < nmb && k0 < r, 1);
                a1[it][m] = load8_bf16(As + (size_t)k1 * d_in, cc, d_in, in && m < nmb && k1 < r, 1);
            }
        }
#pragma unroll
        for (int it = 0; it < ITB; ++it)
#pragma unroll
            for (int m = 0; m < KB; ++m) {
                if (m < nmb) {
                    mma_bf16(acc[m][0], a0[it][m].x, a1[it][m].x, a0[it][m].y, a1[it][m].y, xa[it].x, xa[it].y);
                    mma_bf16(acc[m][0], a0[it][m].z, a1[it][m].z, a0[it][m].w, a1[it][m].w, xa[it].z, xa[it].w);
                    mma_bf16(acc[m][1], a0[it][m].x, a1[it][m].x, a0[it][m].y, a1[it][m].y, xb[it].x, xb[it].y);
                    mma_bf16(acc[m][1], a0[it][m].z, a1[it][m].z, a0[it][m].w, a1[it][m].w, xb[it].z, xb[it].w);
                }
            }
    }
#pragma unroll
    for (int m = 0; m < KB; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) sm.red[warp][(m * 2 + n) * 4 + j][lane] = acc[m][n][j];
    __syncthreads();
    float *dst = fa.part + (size_t)l * fa.part_layer_stride + (size_t)chunk * fa.T * R;
    for (int e = threadIdx.x; e < nmb * 256; e += kFT) {
        const int ln = e & 31, sj = e >> 5;
        const int j = sj & 3, n = (sj >> 2) & 1, m = sj >> 3;
        const float v = sm.red[0][sj][ln] + sm.red[1][sj][ln] + sm.red[2][sj][ln] + sm.red[3][sj][ln];
        const int k = m * 16 + (ln >> 2) + ((j & 2) ? 8 : 0);
        const int tk = n * 8 + 2 * (ln & 3) + (j & 1);
        if (tk < ti.cnt && k < r) dst[(size_t)(ti.pos0 + tk) * R + k] = v;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        st_release_gpu(fa.flags + ((size_t)l * fa.max_tiles + tile) * kMaxChunks + chunk, target);
}

// --------------------------------------------------------------------------
// Expand item: tokens of one tile x 256 output columns.
// --------------------------------------------------------------------------
template <int KB>
struct ExpandRegs {
    uint4 y[2][2];          // [column group][token row g / g+8]
    uint2 b[2][4][KB];      // [column group][n-permutation j][16-rank block]
    int tok[2];
    int l, tile, db;
    TileInfo ti;
};

template <int KB>
__device__ void expand_prefetch(const FusedArgs &fa, FusedSmem &sm, int l, int tile, int db,
                                ExpandRegs<KB> &er) {
    const LayerArgs &L = fa.l[l];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, tq = lane & 3;
    er.l = l;
    er.tile = tile;
    er.db = db;
    er.ti = tile_info(sm, fa.S, tile);
    __syncthreads();                        // tok_e free (previous item done with it)
    if (warp == 0) find_tokens(sm, fa.T, er.ti.s, er.ti.first, sm.tok_e, lane);
    __syncthreads();
    er.tok[0] = gq < er.ti.cnt ? sm.tok_e[gq] : -1;
    er.tok[1] = gq + 8 < er.ti.cnt ? sm.tok_e[gq + 8] : -1;
    const int d_out = L.d_out, R = fa.R, r = er.ti.r;
    const int nkb = (r + 15) >> 4;
    const uint16_t *Bs = static_cast<const uint16_t *>(L.B) + (size_t)er.ti.s * d_out * R;
    const uint16_t *y = static_cast<const uint16_t *>(L.y);
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
        const int c = db * kECols + warp * 64 + grp * 32;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int P = c + 8 * (gq >> 1) + 2 * j + (gq & 1);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                const int k = kb * 16 + 4 * tq;
                uint2 bb = make_uint2(0, 0);
                if (kb < nkb && P < d_out && k < R)
                    bb = __ldg(reinterpret_cast<const uint2 *>(Bs + (size_t)P * R + k));
                if (k + 4 > r) {
                    if (k + 0 >= r) bb.x &= 0xffff0000u;
                    if (k + 1 >= r) bb.x &= 0x0000ffffu;
                    if (k + 2 >= r) bb.y &= 0xffff0000u;
                    if (k + 3 >= r) bb.y &= 0x0000ffffu;
                }
                er.b[grp][j][kb] = bb;
            }
        }
        const int cc = c + 8 * tq;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int tok = er.tok[h];
            er.y[grp][h] = (tok >= 0 && cc < d_out)
                               ? *reinterpret_cast<const uint4 *>(y + (size_t)tok * d_out + cc)
                               : make_uint4(0, 0, 0, 0);
        }
    }
}

template <int KB>
__device__ void expand_finish(const FusedArgs &fa, FusedSmem &sm, ExpandRegs<KB> &er,
                              unsigned target) {
    const LayerArgs &L = fa.l[er.l];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, tq = lane & 3;
    const int nch = L.n_chunks;
    // Wait for every chunk partial of this tile (bounded).
    if (warp == 0) {
        const unsigned *fl = fa.flags + ((size_t)er.l * fa.max_tiles + er.tile) * kMaxChunks;
        bool done = false;
        for (unsigned it = 0; it < kSpinLimit; ++it) {
            const bool mine = lane >= nch || ld_acquire_gpu(fl + lane) == target;
            if (__all_sync(kFull, mine)) {
                done = true;
                break;
            }
            __nanosleep(64);
        }
        if (lane == 0) {
            sm.ok = done;
            if (!done) atomicExch(&fa.hdr[kHdrError], 1);
        }
    }
    __syncthreads();
    if (!sm.ok) return;

    const int R = fa.R, r = er.ti.r;
    const int nkb = (r + 15) >> 4;
    const float scale = sm.scale[er.ti.s];
    const float *part = fa.part + (size_t)er.l * fa.part_layer_stride;
    uint32_t ahi[KB][4], alo[KB][4];
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
        float f[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int k = kb * 16 + 4 * tq;
        if (kb < nkb && k < r) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = gq + 8 * h;
                if (row < er.ti.cnt) {
                    const float *p = part + (size_t)(er.ti.pos0 + row) * R + k;
                    for (int c = 0; c < nch; ++c) {
                        const float4 q = __ldcg(reinterpret_cast<const float4 *>(p + (size_t)c * fa.T * R));
                        f[h][0] += q.x;
                        f[h][1] += q.y;
                        f[h][2] += q.z;
                        f[h][3] += q.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (k + i >= r) f[0][i] = f[1][i] = 0.f;
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

    const int d_out = L.d_out;
    uint16_t *y = static_cast<uint16_t *>(L.y);
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
        const int c = er.db * kECols + warp * 64 + grp * 32;
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                if (kb < nkb) {
                    mma_bf16(acc[j], ahi[kb][0], ahi[kb][1], ahi[kb][2], ahi[kb][3],
                             er.b[grp][j][kb].x, er.b[grp][j][kb].y);
                    mma_bf16(acc[j], alo[kb][0], alo[kb][1], alo[kb][2], alo[kb][3],
                             er.b[grp][j][kb].x, er.b[grp][j][kb].y);
                }
            }
        }
        const int cc = c + 8 * tq;
        if (cc >= d_out) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int tok = er.tok[h];
            if (tok < 0) continue;
            const uint4 yv = er.y[grp][h];
            uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                w[q] = pack_bf16(fmaf(scale, acc[q][2 * h], bf_lo(w[q])),
                                 fmaf(scale, acc[q][2 * h + 1], bf_hi(w[q])));
            *reinterpret_cast<uint4 *>(y + (size_t)tok * d_out + cc) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int KB>
__global__ void __launch_bounds__(kFT)
fused_decode_kernel(const __grid_constant__ FusedArgs fa) {
    __shared__ FusedSmem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = fa.T, S = fa.S;

    // Slot ids into registers and slot parameters into shared memory, together.
    constexpr int kPer = kFusedMaxTokens / kFT;
    int raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int t = tid + i * kFT;
        raw[i] = t < T ? __ldg(fa.idx + t) : -1;
    }
    for (int s = tid; s < S; s += kFT) {
        sm.rank[s] = fa.rank[s];
        sm.scale[s] = fa.scale[s];
        sm.cnt[s] = 0;
    }
    if (tid == 0) {
        sm.invalid = 0;
        sm.epoch = *reinterpret_cast<volatile unsigned *>(fa.hdr + kHdrEpoch);
    }
    __syncthreads();
    int inv = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int t = tid + i * kFT;
        if (t < T) {
            const int r = raw[i];
            const int e = (r >= 0 && r < S && sm.rank[r] > 0) ? r : -1;
            inv += (r < -1 || r >= S);
            sm.eff[t] = (int16_t)e;
            if (e >= 0) atomicAdd(&sm.cnt[e], 1);
        }
    }
    if (inv) atomicAdd(&sm.invalid, inv);
    __syncthreads();
    if (warp == 0) {                         // grouped offsets and tile offsets per slot
        int carry_o = 0, carry_t = 0;
        for (int base = 0; base < S; base += 32) {
            const int s = base + lane;
            const int c = s < S ? sm.cnt[s] : 0;
            const int nt = (c + kTileTokens - 1) / kTileTokens;
            int ic = c, it = nt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(kFull, ic, o), b = __shfl_up_sync(kFull, it, o);
                if (lane >= o) { ic += a; it += b; }
            }
            if (s < S) {
                sm.off[s] = carry_o + ic - c;
                sm.toff[s] = carry_t + it - nt;
            }
            carry_o += __shfl_sync(kFull, ic, 31);
            carry_t += __shfl_sync(kFull, it, 31);
        }
        if (lane == 0) {
            sm.off[S] = carry_o;
            sm.toff[S] = carry_t;
            sm.ntiles = carry_t;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0 && sm.invalid) atomicAdd(fa.hdr + kHdrInvalid, sm.invalid);
    const int ntiles = sm.ntiles;
    const unsigned target = sm.epoch + 1u;
    int ns = 0, ne = 0;
    for (int l = 0; l < fa.n; ++l) {
        ns += ntiles * fa.l[l].n_chunks;
        ne += ntiles * ((fa.l[l].d_out + kECols - 1) / kECols);
    }
    const int G = gridDim.x;

    ExpandRegs<KB> er;
    const int e0 = blockIdx.x;
    if (e0 < ne) {
        int l, tile, db;
        decode_item(fa, ntiles, e0, true, l, tile, db);
        expand_prefetch<KB>(fa, sm, l, tile, db, er);
    }
    for (int it = blockIdx.x; it < ns; it += G) {
        int l, tile, chunk;
        decode_item(fa, ntiles, it, false, l, tile, chunk);
        shrink_item<KB>(fa, sm, l, tile, chunk, target);
    }
    for (int it = e0; it < ne; it += G) {
        if (it != e0) {
            int l, tile, db;
            decode_item(fa, ntiles, it, true, l, tile, db);
            expand_prefetch<KB>(fa, sm, l, tile, db, er);
        }
        expand_finish<KB>(fa, sm, er, target);
    }

    // The last CTA to finish advances the epoch for the next launch.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(fa.hdr + kHdrExit, 1);
        if (prev == G - 1) {
            fa.hdr[kHdrExit] = 0;
            atomicAdd(fa.hdr + kHdrEpoch, 1);
        }
    }
}

template <int KB>
int ctas_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_decode_kernel<KB>, kFT, 0) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

}  // namespace

int fused_decode_ctas_per_sm(int max_lora_rank) {
    if (max_lora_rank <= 16) return ctas_per_sm<1>();
    if (max_lora_rank <= 32) return ctas_per_sm<2>();
    return ctas_per_sm<4>();
}

cudaError_t launch_fused_decode(const FusedArgs &fa, int grid, cudaStream_t st) {
    if (fa.R <= 16)
        fused_decode_kernel<1><<<grid, kFT, 0, st>>>(fa);
    else if (fa.R <= 32)
        fused_decode_kernel<2><<<grid, kFT, 0, st>>>(fa);
    else
        fused_decode_kernel<4><<<grid, kFT, 0, st>>>(fa);
    return cudaGetLastError();
}

}  // namespace lora
