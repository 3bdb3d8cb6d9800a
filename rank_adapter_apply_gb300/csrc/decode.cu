// Decode path: grouped shrink and expand-add over tiles of <= 16 tokens that
// share one slot.
//
//   shrink:  v[t][k] = sum_j A_s[k][j] x[t][j]           (k < r_s, fp32)
//   expand:  y[t][i] = round(y[t][i] + scale_s * sum_k B_s[i][k] v[t][k])
//
// The delta itself is the LoRA update written with the PEFT adapter fields r
// and lora_alpha (the adapter_config.json example on the "vLLM LoRA Resolver
// 插件详解" page, section 3.2); scale_s = lora_alpha / r_s with the adapter's own
// rank, ranks zero-padded to max_lora_rank in the slot pools (the
// "Multi-LoRA 适配器缓存生产实战" page, section 核心原理, parameter table).
//
// bf16: both contractions run on the tensor cores with mma.m16n8k16 (bf16
// operands, fp32 accumulation). Operands go straight from global memory to
// registers with 128-bit loads: the order of the k index inside one MMA is a
// free choice as long as both operands use the same one, so every lane loads
// eight consecutive elements of a row at once. The expand splits v into a bf16
// high part and a bf16 remainder (two MMAs) so v keeps ~16 significant bits.
// fp32: plain CUDA-core loops (exact fp32 FMAs).
//
// The shrink splits d_in into n_chunks column chunks (one CTA each) so a
// decode batch fills the GPU; each CTA writes its partial sums, and the last
// CTA to arrive for a tile adds them in chunk order (deterministic) and writes v.
#include "kernels.cuh"
#include "device_util.cuh"

#include <cuda_bf16.h>

namespace lora {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kExpandCols = 256;          // output columns per expand CTA (bf16 and fp32)

// v of the bf16 path, kept in the order the expand's MMA fragments read it:
// row `pos` of VS = v_stride(R) floats holds, for every four ranks k0 .. k0 + 3 (k0 a
// multiple of 4), one 16-byte group: the bf16 high parts of the four ranks,
// then their bf16 low parts (value - high part), lower rank first. The
// expand then loads a fragment with one 16-byte load per row instead of
// splitting fp32 values for every 256-column block it covers.
__device__ __forceinline__ void store_vfrag(float *v, int VS, int pos, int k, float s) {
    const __nv_bfloat16 h = __float2bfloat16_rn(s);
    const __nv_bfloat16 l = __float2bfloat16_rn(s - __bfloat162float(h));
    __nv_bfloat16 *grp = reinterpret_cast<__nv_bfloat16 *>(v + (size_t)pos * VS) + (k >> 2) * 8;
    grp[k & 3] = h;
    grp[4 + (k & 3)] = l;
}

// Sum the chunk partials of one tile in chunk order and write v (last CTA
// only): ranks below `kr` of each row, as fp32 or (frag) in the bf16
// fragment order. A partial row is v_stride(R) floats long (whole 16-rank
// blocks, like the rows of v). Loads of eight chunks are issued before they
// are added (the sum keeps the chunk order), so a 14-way split costs two L2
// round trips, not fourteen.
__device__ void finish_split(const LayerArgs &L, const GroupView &g, int tile_i, int p0, int cnt,
                             int kr, bool frag) {
    __shared__ int last;
    // The CTA's partial stores are ordered before thread 0's count by the
    // barrier, and published at GPU scope by the count's release; the last
    // CTA's acquire (the same atomic) and the barrier after it order every
    // thread's reads of the other chunks' partials after their counts.
    __syncthreads();
    if (threadIdx.x == 0) {
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(prev) : "l"(L.counters + tile_i) : "memory");
        last = (prev == L.n_chunks - 1);
    }
    __syncthreads();
    if (!last) return;
    const int R = g.R, T = g.T, PS = v_stride(R);
    const size_t cs = (size_t)T * PS;
    for (int e = threadIdx.x; e < cnt * kr; e += kThreads) {
        const int pos = p0 + e / kr, k = e % kr;
        const float *src = L.part + (size_t)pos * PS + k;
        float s = 0.f;
        int ch = 0;
        for (; ch + 8 <= L.n_chunks; ch += 8) {
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldcg(src + (size_t)(ch + u) * cs);
#pragma unroll
            for (int u = 0; u < 8; ++u) s += a[u];
        }
        for (; ch < L.n_chunks; ++ch) s += __ldcg(src + (size_t)ch * cs);
        if (frag) store_vfrag(L.v, v_stride(R), pos, k, s);
        else L.v[(size_t)pos * R + k] = s;
    }
    if (threadIdx.x == 0) L.counters[tile_i] = 0;
}

// ---------------------------------------------------------------------------
// bf16 shrink. CTA = (d_in chunk, tile, layer); 4 warps stride the chunk in
// 32-column steps. Per warp and step: m16n8k16 with M = 16 ranks (per 16-rank
// block), N = 8 tokens (two token blocks), K = 16 (two MMAs per 32 columns).
// ---------------------------------------------------------------------------
// The column loop of one shrink item for NMB 16-rank blocks, UNROLL steps
// of 32 columns per warp in flight.
template <int NMB, int UNROLL>
__device__ __forceinline__ void shrink_steps(float (&acc)[4][2][4], const uint16_t *xr0, const uint16_t *xr1,
                                             const uint16_t *As, int tok0, int tok1, int r, int d_in, int c0,
                                             int c1, int vec) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll UNROLL
    for (int col = c0 + warp * 32; col < c1; col += kWarps * 32) {
        const int cc = col + 8 * tq;
        const uint4 xa = load8_bf16(xr0, cc, d_in, tok0 >= 0, vec);
        const uint4 xb = load8_bf16(xr1, cc, d_in, tok1 >= 0, vec);
        uint4 a0[NMB], a1[NMB];
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            const int k0 = m * 16 + gq, k1 = k0 + 8;
            a0[m] = load8_bf16(As + (size_t)k0 * d_in, cc, d_in, k0 < r, vec);
            a1[m] = load8_bf16(As + (size_t)k1 * d_in, cc, d_in, k1 < r, vec);
        }
        // first halves of K for every accumulator, then the second halves: each
        // accumulator adds in the same order, and no MMA waits on the one
        // issued just before it
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            mma_bf16(acc[m][0], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xa.x, xa.y);
            mma_bf16(acc[m][1], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xb.x, xb.y);
        }
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            mma_bf16(acc[m][0], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xa.z, xa.w);
            mma_bf16(acc[m][1], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xb.z, xb.w);
        }
    }
}

// The same loop when every row is 16-byte aligned and the chunk is a whole
// number of 32-column steps (d_in % 32 == 0): plain 16-byte loads, predicated
// only on the token existing and the rank being below the slot's rank.
template <int NMB, int UNROLL>
__device__ __forceinline__ void shrink_steps_fast(float (&acc)[4][2][4], const uint16_t *xr0, const uint16_t *xr1,
                                                  const uint16_t *As, bool ok0, bool ok1, int r, int d_in, int c0,
                                                  int c1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint16_t *ar0[NMB], *ar1[NMB];
    bool ak0[NMB], ak1[NMB];
#pragma unroll
    for (int m = 0; m < NMB; ++m) {
        const int k0 = m * 16 + gq, k1 = k0 + 8;
        ar0[m] = As + (size_t)k0 * d_in;
        ar1[m] = As + (size_t)k1 * d_in;
        ak0[m] = k0 < r;
        ak1[m] = k1 < r;
    }
#pragma unroll UNROLL
    for (int cc = c0 + warp * 32 + 8 * tq; cc < c1; cc += kWarps * 32) {
        const uint4 xa = ok0 ? __ldg(reinterpret_cast<const uint4 *>(xr0 + cc)) : zero;
        const uint4 xb = ok1 ? __ldg(reinterpret_cast<const uint4 *>(xr1 + cc)) : zero;
        uint4 a0[NMB], a1[NMB];
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            a0[m] = ak0[m] ? __ldg(reinterpret_cast<const uint4 *>(ar0[m] + cc)) : zero;
            a1[m] = ak1[m] ? __ldg(reinterpret_cast<const uint4 *>(ar1[m] + cc)) : zero;
        }
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            mma_bf16(acc[m][0], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xa.x, xa.y);
            mma_bf16(acc[m][1], a0[m].x, a1[m].x, a0[m].y, a1[m].y, xb.x, xb.y);
        }
#pragma unroll
        for (int m = 0; m < NMB; ++m) {
            mma_bf16(acc[m][0], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xa.z, xa.w);
            mma_bf16(acc[m][1], a0[m].z, a1[m].z, a0[m].w, a1[m].w, xb.z, xb.w);
        }
    }
}

__device__ __forceinline__ void shrink_bf16_tile(const LayerArgs &L, const GroupView &g, int chunk, int tile_i) {
    const int4 tile = g.tiles[tile_i];
    const int s = tile.x, p0 = tile.y, cnt = tile.z;
    const int r = tile.w;                      // the slot's rank, from the grouping
    const int nmb = (r + 15) >> 4;
    const int R = g.R, d_in = L.d_in;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2;

    const int tok0 = gq < cnt ? g.perm[p0 + gq] : -1;
    const int tok1 = gq + 8 < cnt ? g.perm[p0 + 8 + gq] : -1;
    const uint16_t *x = static_cast<const uint16_t *>(L.x);
    const uint16_t *xr0 = x + (size_t)(tok0 < 0 ? 0 : tok0) * d_in;
    const uint16_t *xr1 = x + (size_t)(tok1 < 0 ? 0 : tok1) * d_in;
    const uint16_t *As = static_cast<const uint16_t *>(L.A) + (size_t)s * R * d_in;

    float acc[4][2][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[m][n][j] = 0.f;

    const int c0 = chunk * L.chunk_cols;
    const int c1 = min(d_in, c0 + L.chunk_cols);
    // The rank-block count is a template argument of the loop, so that no
    // runtime condition stands between the loads of several steps.
    if (L.vec && (d_in & 31) == 0) {
        if (nmb <= 1) shrink_steps_fast<1, 4>(acc, xr0, xr1, As, tok0 >= 0, tok1 >= 0, r, d_in, c0, c1);
        else if (nmb == 2) shrink_steps_fast<2, 2>(acc, xr0, xr1, As, tok0 >= 0, tok1 >= 0, r, d_in, c0, c1);
        else shrink_steps_fast<4, 2>(acc, xr0, xr1, As, tok0 >= 0, tok1 >= 0, r, d_in, c0, c1);
    } else {
        if (nmb <= 1) shrink_steps<1, 4>(acc, xr0, xr1, As, tok0, tok1, r, d_in, c0, c1, L.vec);
        else if (nmb == 2) shrink_steps<2, 2>(acc, xr0, xr1, As, tok0, tok1, r, d_in, c0, c1, L.vec);
        else shrink_steps<4, 2>(acc, xr0, xr1, As, tok0, tok1, r, d_in, c0, c1, L.vec);
    }

    // Cross-warp sum through shared memory.
    __shared__ float red[kWarps][4 * 2 * 4][32];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) red[warp][(m * 2 + n) * 4 + j][lane] = acc[m][n][j];
    __syncthreads();
    // ranks r .. 16 nmb - 1 come out as exact zeros (their A rows are
    // masked) and are written too: the expand reads whole 16-rank blocks
    // (rows of v and of the partials hold whole blocks)
    const bool split = L.n_chunks > 1;
    const int PS = v_stride(R);
    float *part = L.part + (size_t)chunk * g.T * PS;
    for (int e = threadIdx.x; e < nmb * 256; e += kThreads) {
        const int ln = e & 31, slot_j = e >> 5;          // slot_j = (m*2+n)*4 + j
        const int j = slot_j & 3, n = (slot_j >> 2) & 1, m = slot_j >> 3;
        float v = red[0][slot_j][ln] + red[1][slot_j][ln] + red[2][slot_j][ln] + red[3][slot_j][ln];
        const int k = m * 16 + (ln >> 2) + ((j & 2) ? 8 : 0);
        const int tk = n * 8 + 2 * (ln & 3) + (j & 1);
        if (tk < cnt) {
            if (split) part[(size_t)(p0 + tk) * PS + k] = v;
            else store_vfrag(L.v, v_stride(R), p0 + tk, k, v);
        }
    }
    if (split) finish_split(L, g, tile_i, p0, cnt, 16 * nmb, true);
}

// ---------------------------------------------------------------------------
// bf16 expand-add. CTA = (256-column block of d_out, slot, layer): the block's
// B rows of the slot cross HBM once and serve every tile of that slot (the
// tiles of one slot are consecutive in the tile list). Each warp owns 64
// columns (two 32-column groups). Per group and tile: 4 MMAs with M = 16
// tokens, N = 8 columns, K = 16 ranks, columns permuted so that each lane ends
// with 8 consecutive outputs of two token rows (one 128-bit y access per row).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int bkey(int P) { return (((P >> 3) & 3) << 1) | (P & 1); }

__device__ __forceinline__ void expand_bf16_run(const LayerArgs &L, const GroupView &g, int dblock, int t0,
                                                int n_tiles) {
    const int d_out = L.d_out;
    const int4 head = g.tiles[t0];
    const int s = head.x;
    const int r = head.w;                      // the slot's rank, from the grouping
    const int nkb = (r + 15) >> 4;
    const float scale = g.scale[s];
    const int R = g.R, VS = v_stride(R);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;

    // This block's B rows (the slot's first 16 * nkb ranks) go to shared memory
    // in one burst of 16-byte cp.async: row P of the block at bs + 64 P, chunk
    // c of the row at chunk c ^ key(P). One fragment read touches rows
    // P0 + 8a + b (a < 4, b < 2), so the key takes bits 3..4 and 0 of P and
    // those eight rows land in distinct bank groups. Thread i copies chunk
    // i % 8 of rows i / 8, i / 8 + 16, ...; in the rank-blocked pool chunk
    // ch of row P lies in block ch * 8 / kb, at P * kb + ch * 8 % kb there.
    __shared__ __align__(16) uint16_t bs[kExpandCols * 64];
    const uint16_t *Bs = static_cast<const uint16_t *>(L.B) + (size_t)s * d_out * R;
    const int c0 = dblock * kExpandCols;
    {
        const int ch = threadIdx.x & 7;
        const int rows = min(kExpandCols, d_out - c0);
        if (ch < 2 * nkb && ch * 8 < R) {
            const int kb = b_block(R);
            const uint16_t *src = Bs + ((size_t)((ch * 8) / kb) * d_out + c0) * kb + (ch * 8) % kb;
            for (int P = threadIdx.x >> 3; P < rows; P += kThreads / 8)
                cp_async16(bs + P * 64 + ((ch ^ bkey(P)) << 3), src + (size_t)P * kb);
        } else if (ch < 2 * nkb) {
            // ranks past max_lora_rank inside the last 16-rank block: zeros
            // (the MMA multiplies them with v's zero ranks)
            for (int P = threadIdx.x >> 3; P < rows; P += kThreads / 8)
                *reinterpret_cast<uint4 *>(bs + P * 64 + ((ch ^ bkey(P)) << 3)) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
    }

    uint16_t *y = static_cast<uint16_t *>(L.y);
    const int vec = L.vec;
    bool staged = false;
    for (int t = t0; t < n_tiles; ++t) {
        int4 tile = head;
        if (t != t0) {
            tile = g.tiles[t];
            if (tile.x != s) break;              // the next slot's tiles
        }
        const int p0 = tile.y, cnt = tile.z;
        const int tok0 = gq < cnt ? g.perm[p0 + gq] : -1;
        const int tok1 = gq + 8 < cnt ? g.perm[p0 + 8 + gq] : -1;

        // A fragments of V (rows = tokens gq, gq+8; k = 4tq..4tq+3 of each
        // 16-rank block): one 16-byte load per row and block of the high and
        // low parts the shrink stored in fragment order.
        uint32_t ahi[4][4], alo[4][4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            if (kb >= nkb) break;
            const int grp = kb * 4 + tq;                 // ranks 4 grp .. 4 grp + 3
            uint4 q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
            if (gq < cnt) q0 = *reinterpret_cast<const uint4 *>(L.v + (size_t)(p0 + gq) * VS + grp * 4);
            if (gq + 8 < cnt) q1 = *reinterpret_cast<const uint4 *>(L.v + (size_t)(p0 + gq + 8) * VS + grp * 4);
            ahi[kb][0] = q0.x;
            ahi[kb][1] = q1.x;
            ahi[kb][2] = q0.y;
            ahi[kb][3] = q1.y;
            alo[kb][0] = q0.z;
            alo[kb][1] = q1.z;
            alo[kb][2] = q0.w;
            alo[kb][3] = q1.w;
        }

        // y of both column groups and both token rows, fetched before the
        // MMAs so that their latency overlaps the B loads.
        uint4 ypre[2][2];
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int cc = c0 + warp * 64 + grp * 32 + 8 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tok = h ? tok1 : tok0;
                ypre[grp][h] = (vec && tok >= 0 && cc + 8 <= d_out)
                                   ? *reinterpret_cast<const uint4 *>(y + (size_t)tok * d_out + cc)
                                   : make_uint4(0, 0, 0, 0);
            }
        }

        if (!staged) {                           // (the same for every thread of the CTA)
            cp_async_wait_all();                 // this thread's B chunks have landed
            __syncthreads();                     // and every other thread's
            staged = true;
        }

#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int c = c0 + warp * 64 + grp * 32;
            if (c >= d_out) break;
            // Every B fragment of the group first, then per 16-rank block the
            // high-part MMAs of the four column blocks and after them the
            // low-part ones: each accumulator adds in the order of a
            // one-block-at-a-time loop, while four independent MMAs go out
            // back to back. (ranks >= r are zero in the pool and in v, so no
            // mask is needed)
            // The rows this lane reads, P = c + 8 (gq >> 1) + 2 j + (gq & 1),
            // all have key(P - c0) = gq (c - c0 is a multiple of 32), so the
            // swizzled chunk of rank block kb is (2 kb + tq / 2) ^ gq.
            uint2 bb[4][4];
            const uint16_t *brow = bs + (c - c0 + 8 * (gq >> 1) + (gq & 1)) * 64 + 4 * (tq & 1);
            const bool full_grp = c + 32 <= d_out;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int P = c + 8 * (gq >> 1) + 2 * j + (gq & 1);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    bb[j][kb] = make_uint2(0, 0);
                    if (kb < nkb && (full_grp || P < d_out))
                        bb[j][kb] = *reinterpret_cast<const uint2 *>(brow + 2 * j * 64 + (((2 * kb + (tq >> 1)) ^ gq) << 3));
                }
            }
            float acc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb >= nkb) break;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16(acc[j], ahi[kb][0], ahi[kb][1], ahi[kb][2], ahi[kb][3], bb[j][kb].x, bb[j][kb].y);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16(acc[j], alo[kb][0], alo[kb][1], alo[kb][2], alo[kb][3], bb[j][kb].x, bb[j][kb].y);
            }
            // Lane owns columns c + 8tq .. c + 8tq + 7 of rows tok0 (acc[.][0..1]) and tok1 (acc[.][2..3]).
            const int cc = c + 8 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tok = h ? tok1 : tok0;
                if (tok < 0) continue;
                uint16_t *row = y + (size_t)tok * d_out;
                float dlt[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    dlt[2 * j] = acc[j][2 * h];
                    dlt[2 * j + 1] = acc[j][2 * h + 1];
                }
                if (vec && cc + 8 <= d_out) {
                    const uint4 yv = ypre[grp][h];
                    uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        w[q] = pack_bf16(fmaf(scale, dlt[2 * q], bf_lo(w[q])),
                                         fmaf(scale, dlt[2 * q + 1], bf_hi(w[q])));
                    *reinterpret_cast<uint4 *>(row + cc) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (cc + i < d_out) {
                            float yo = __uint_as_float((uint32_t)row[cc + i] << 16);
                            __nv_bfloat16 o = __float2bfloat16_rn(fmaf(scale, dlt[i], yo));
                            row[cc + i] = *reinterpret_cast<uint16_t *>(&o);
                        }
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// fp32 shrink: one warp per token of the tile, lanes stride the chunk, one
// warp-shuffle reduction per rank.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void shrink_f32_tile(const LayerArgs &L, const GroupView &g, int chunk, int tile_i) {
    const int4 tile = g.tiles[tile_i];
    const int s = tile.x, p0 = tile.y, cnt = tile.z;
    const int r = tile.w;                      // the slot's rank, from the grouping
    const int R = g.R, d_in = L.d_in;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *x = static_cast<const float *>(L.x);
    const float *As = static_cast<const float *>(L.A) + (size_t)s * R * d_in;
    const int c0 = chunk * L.chunk_cols;
    const int c1 = min(d_in, c0 + L.chunk_cols);
    // v rows hold R floats, partial rows v_stride(R)
    const int ds = L.n_chunks == 1 ? R : v_stride(R);
    float *dst_base = L.n_chunks == 1 ? L.v : L.part + (size_t)chunk * g.T * ds;
    for (int i = warp; i < cnt; i += kWarps) {
        const float *xr = x + (size_t)g.perm[p0 + i] * d_in;
        for (int k = 0; k < r; ++k) {
            const float *ar = As + (size_t)k * d_in;
            float a = 0.f;
            for (int c = c0 + lane; c < c1; c += 32) a = fmaf(ar[c], xr[c], a);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) dst_base[(size_t)(p0 + i) * ds + k] = a;
        }
    }
    if (L.n_chunks > 1) finish_split(L, g, tile_i, p0, cnt, r, false);
}

// fp32 expand-add: each thread owns two columns of the 256-column block.
__device__ __forceinline__ void expand_f32_tile(const LayerArgs &L, const GroupView &g, int dblock, int tile_i) {
    const int d_out = L.d_out;
    const int4 tile = g.tiles[tile_i];
    const int s = tile.x, p0 = tile.y, cnt = tile.z;
    const int r = tile.w;                      // the slot's rank, from the grouping
    const float scale = g.scale[s];
    const int R = g.R;
    extern __shared__ float sv[];                     // [kTileTokens][r]
    for (int e = threadIdx.x; e < cnt * r; e += kThreads)
        sv[e] = L.v[(size_t)(p0 + e / r) * R + e % r];
    __syncthreads();
    const float *Bs = static_cast<const float *>(L.B) + (size_t)s * d_out * R;
    float *y = static_cast<float *>(L.y);
    for (int h = 0; h < 2; ++h) {
        const int col = dblock * kExpandCols + h * kThreads + threadIdx.x;
        if (col >= d_out) continue;
        const int kb = b_block(R), kbs = kb == 32 ? 5 : (kb == 16 ? 4 : 3);
        const float *br = Bs + (size_t)col * kb;         // rank k at br[(k / kb) * d_out * kb + k % kb]
        for (int i = 0; i < cnt; ++i) {
            float a = 0.f;
            for (int k = 0; k < r; ++k)
                a = fmaf(br[(size_t)(k >> kbs) * d_out * kb + (k & (kb - 1))], sv[i * r + k], a);
            float *yp = y + (size_t)g.perm[p0 + i] * d_out + col;
            *yp = fmaf(scale, a, *yp);
        }
    }
}

// Work item w = (t * n + l) * inner + i (tile t, layer l, chunk or column
// block i), walked with a stride of gridDim.x from blockIdx.x: the indices
// are carried from one item to the next, so a CTA divides once, not three
// times per item (most items of a mixed batch are skipped, so this is most of
// what a skipped item costs).
struct ItemWalk {
    int i, l, t, si, sl, st, inner, n;
    __device__ ItemWalk(int inner_, int n_) : inner(inner_), n(n_) {
        const int w = (int)blockIdx.x, g = (int)gridDim.x;
        i = w % inner;
        l = (w / inner) % n;
        t = w / (inner * n);
        si = g % inner;
        sl = (g / inner) % n;
        st = g / (inner * n);
    }
    __device__ void next() {
        i += si;
        l += sl;
        t += st;
        if (i >= inner) {
            i -= inner;
            ++l;
        }
        if (l >= n) {
            l -= n;
            ++t;
        }
    }
};

// The kernels are persistent: work items are (tile, layer, chunk) for the
// shrink and (tile, layer, 256-column block) for the expand, taken with a
// stride of gridDim.x. The tile count is known on the device only (a prefill
// batch may leave few or no decode tiles), so the grid is sized from the SM
// count and items past the count cost nothing.
__global__ void __launch_bounds__(kThreads)
shrink_bf16_kernel(MultiArgs ma, GroupView g, int max_chunks) {
    grid_dependency_wait();            // launched early: the kernel before has to finish first
    grid_launch_dependents();
    const int n_tiles = g.hdr[kHdrTiles];
    for (ItemWalk it(max_chunks, ma.n); it.t < n_tiles; it.next()) {
        const int chunk = it.i, l = it.l, t = it.t;
        const LayerArgs &L = ma.l[l];
        if (chunk >= L.n_chunks) continue;
        shrink_bf16_tile(L, g, chunk, t);
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads, 4)
expand_bf16_kernel(MultiArgs ma, GroupView g, int max_dblocks) {
    grid_dependency_wait();            // launched early: the kernel before has to finish first
    grid_launch_dependents();
    const int n_tiles = g.hdr[kHdrTiles];
    for (ItemWalk it(max_dblocks, ma.n); it.t < n_tiles; it.next()) {
        const int db = it.i, l = it.l, t = it.t;
        const LayerArgs &L = ma.l[l];
        if (db * kExpandCols >= L.d_out) continue;
        // Items of a slot's first tile cover all of that slot's tiles.
        if (t > 0 && g.tiles[t - 1].x == g.tiles[t].x) continue;
        expand_bf16_run(L, g, db, t, n_tiles);
        __syncthreads();                     // the staged B rows are free for the next item
    }
}

__global__ void __launch_bounds__(kThreads)
shrink_f32_kernel(MultiArgs ma, GroupView g, int max_chunks) {
    grid_dependency_wait();            // launched early: the kernel before has to finish first
    grid_launch_dependents();
    const int n_tiles = g.hdr[kHdrTiles];
    for (ItemWalk it(max_chunks, ma.n); it.t < n_tiles; it.next()) {
        const int chunk = it.i, l = it.l, t = it.t;
        const LayerArgs &L = ma.l[l];
        if (chunk >= L.n_chunks) continue;
        shrink_f32_tile(L, g, chunk, t);
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads)
expand_f32_kernel(MultiArgs ma, GroupView g, int max_dblocks) {
    grid_dependency_wait();            // launched early: the kernel before has to finish first
    grid_launch_dependents();
    const int n_tiles = g.hdr[kHdrTiles];
    for (ItemWalk it(max_dblocks, ma.n); it.t < n_tiles; it.next()) {
        const int db = it.i, l = it.l, t = it.t;
        const LayerArgs &L = ma.l[l];
        if (db * kExpandCols >= L.d_out) continue;
        expand_f32_tile(L, g, db, t);
        __syncthreads();
    }
}

// A wait that nothing completes, bounded like every wait of the kernels: it
// gives up after `limit` probes and records that in the error word.
__global__ void selftest_wait_kernel(int *err_word, uint32_t limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool done = mbar_wait_bounded(&bar, 0, limit);
    if (!done && threadIdx.x == 0) atomicExch(err_word, 1);
}

__global__ void set_slot_kernel(float *scale_dev, int *rank_dev, int slot, float scale, int rank) {
    scale_dev[slot] = scale;
    rank_dev[slot] = rank;
}

}  // namespace

cudaError_t launch_decode(const MultiArgs &ma, const GroupView &gv, int dtype, int grid_tiles,
                          int max_chunks, int max_dblocks, int num_sms, cudaStream_t st) {
    if (grid_tiles <= 0) return cudaSuccess;
    // Persistent grids: at most 8 resident-sized waves of CTAs per SM.
    const long long cap = 8LL * (num_sms > 0 ? num_sms : 1);
    auto grid = [&](int per_tile) {
        long long items = (long long)grid_tiles * per_tile * ma.n;
        return (int)(items < cap ? items : cap);
    };
    cudaError_t e;
    if (dtype == 1) {
        e = launch_pdl(shrink_bf16_kernel, dim3(grid(max_chunks)), dim3(kThreads), 0, st, ma, gv, max_chunks);
        if (e == cudaSuccess)
            e = launch_pdl(expand_bf16_kernel, dim3(grid(max_dblocks)), dim3(kThreads), 0, st, ma, gv, max_dblocks);
    } else {
        e = launch_pdl(shrink_f32_kernel, dim3(grid(max_chunks)), dim3(kThreads), 0, st, ma, gv, max_chunks);
        size_t smem = (size_t)kTileTokens * gv.R * sizeof(float);
        if (e == cudaSuccess)
            e = launch_pdl(expand_f32_kernel, dim3(grid(max_dblocks)), dim3(kThreads), smem, st, ma, gv, max_dblocks);
    }
    return e;
}

cudaError_t launch_selftest_wait(int *err_word, uint32_t limit, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(err_word, limit);
    return cudaGetLastError();
}

cudaError_t launch_set_slot(float *scale_dev, int *rank_dev, int slot, float scale, int rank,
                            cudaStream_t st) {
    set_slot_kernel<<<1, 1, 0, st>>>(scale_dev, rank_dev, slot, scale, rank);
    return cudaGetLastError();
}

}  // namespace lora
