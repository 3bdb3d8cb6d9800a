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
// One CTA owns one tile (<= 128 rows of one run) and one range of d_out
// columns. Warp roles:
//   warp 0      TMA producer: X / A_s k-blocks (64 columns), then y / B_s
//               n-blocks (64 columns), through one 3-stage shared-memory ring;
//   warp 1      allocates TMEM and issues every tcgen05.mma from one thread;
//   warps 4..7  epilogue, one TMEM lane (= one tile row) per thread:
//               V (fp32 in TMEM) -> bf16 high + low parts in swizzled shared
//               memory (the A operand of the expand, so V keeps ~16
//               significant bits); then per n-block y = round(y + scale * D).
// TMEM columns: [0, R) shrink accumulator, [64, 128) and [128, 192) the two
// expand accumulators. Every mbarrier wait is bounded.
#include "device_util.cuh"
#include "kernels.cuh"
#include "tc_util.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_bf16.h>

namespace lora {
namespace {

constexpr int kPT = 256;                   // 8 warps
constexpr int kStages = 3;
constexpr int kStageBytes = 24576;         // 16 KB (X or y tile) + 8 KB (A or B tile)
constexpr int kTileBytes = 16384;          // 128 rows x 64 bf16
constexpr int kTmemCols = 256;
constexpr uint32_t kAcc2Col = 64;
constexpr uint32_t kWaitLimit = 1u << 24;

struct PrefillSmem {
    uint64_t full[kStages], empty[kStages];
    uint64_t acc1_full, v_ready;
    uint64_t acc2_full[2], acc2_empty[2];
    uint32_t tmem_base;
    int error;
};

__host__ __device__ constexpr size_t prefill_smem_bytes(int R) {
    return 1024 /* alignment slack */ + (size_t)kStages * kStageBytes + 2 * 128 * (size_t)R * 2 +
           sizeof(PrefillSmem);
}

__device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, int *err) {
    if (mbar_wait_bounded(bar, parity, kWaitLimit)) return true;
    *err = 1;
    return false;
}

template <int R>
__global__ void __launch_bounds__(kPT, 2)
prefill_tc_kernel(const __grid_constant__ PrefillArgs pa) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = base;
    uint8_t *v_hi = base + kStages * kStageBytes;
    uint8_t *v_lo = v_hi + 128 * R * 2;
    PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(v_lo + 128 * R * 2);
    constexpr int W = R * 2;                                   // bytes per V / B row
    constexpr uint32_t kSwzRank = R == 64 ? tc::kSwz128 : (R == 32 ? tc::kSwz64 : tc::kSwz32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = pa.hdr[kHdrPrefillTiles];
    if ((int)blockIdx.x >= n_tiles) return;
    const int4 pt = pa.ptiles[blockIdx.x];
    const int s = pt.x, row0 = pt.y, rows = pt.z;
    const int o_begin = blockIdx.y * pa.cols_per_split;
    const int o_end = min(pa.d_out, o_begin + pa.cols_per_split);
    if (o_begin >= o_end) return;
    const int nk = (pa.d_in + 63) / 64;
    const int nn = (o_end - o_begin + 63) / 64;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 2);          // MMA completion + epilogue (n-blocks) or MMA again
        }
        mbar_init(&sm.acc1_full, 1);
        mbar_init(&sm.v_ready, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc2_full[i], 1);
            mbar_init(&sm.acc2_empty[i], 128);
        }
        sm.error = 0;
        fence_mbar_init();
        tc::prefetch_tensormap(&pa.mx);
        tc::prefetch_tensormap(&pa.ma);
        tc::prefetch_tensormap(&pa.mb);
        tc::prefetch_tensormap(&pa.my);
    }
    if (warp == 1) {
        tc::tmem_alloc(&sm.tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    int err = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer ----------------
            for (int i = 0; i < nk + nn; ++i) {
                const int st = i % kStages;
                const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                wait(&sm.empty[st], ph ^ 1u, &err);
                uint8_t *tile = ring + st * kStageBytes;
                if (i < nk) {
                    mbar_arrive_expect_tx(&sm.full[st], kTileBytes + R * 128);
                    tc::tma_load_2d(tile, &pa.mx, i * 64, row0, &sm.full[st]);
                    tc::tma_load_2d(tile + kTileBytes, &pa.ma, i * 64, s * R, &sm.full[st]);
                } else {
                    const int col = o_begin + (i - nk) * 64;
                    mbar_arrive_expect_tx(&sm.full[st], kTileBytes + 64 * W);
                    tc::tma_load_2d(tile, &pa.my, col, row0, &sm.full[st]);
                    tc::tma_load_2d(tile + kTileBytes, &pa.mb, 0, s * pa.d_out + col, &sm.full[st]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t id1 = tc::idesc_bf16(128, R);
            constexpr uint32_t id2 = tc::idesc_bf16(128, 64);
            for (int kb = 0; kb < nk; ++kb) {
                const int st = kb % kStages;
                wait(&sm.full[st], (uint32_t)(kb / kStages) & 1u, &err);
                tc::fence_after_sync();
                const uint32_t xa = smem_u32(ring + st * kStageBytes);
                const uint32_t aa = xa + kTileBytes;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc::mma_bf16(tmem, tc::smem_desc(xa + k * 32, 128, tc::kSwz128),
                                 tc::smem_desc(aa + k * 32, 128, tc::kSwz128), id1, (kb | k) != 0);
                tc::mma_commit(&sm.empty[st]);
                tc::mbar_arrive(&sm.empty[st]);
            }
            tc::mma_commit(&sm.acc1_full);
            wait(&sm.v_ready, 0, &err);
            tc::fence_after_sync();
            const uint32_t vh = smem_u32(v_hi), vl = smem_u32(v_lo);
            for (int j = 0; j < nn; ++j) {
                const int i = nk + j, st = i % kStages, b = j & 1;
                wait(&sm.full[st], (uint32_t)(i / kStages) & 1u, &err);
                wait(&sm.acc2_empty[b], ((uint32_t)(j >> 1) & 1u) ^ 1u, &err);
                tc::fence_after_sync();
                const uint32_t ba = smem_u32(ring + st * kStageBytes + kTileBytes);
                const uint32_t d = tmem + kAcc2Col + 64u * b;
#pragma unroll
                for (int k = 0; k < R / 16; ++k)
                    tc::mma_bf16(d, tc::smem_desc(vh + k * 32, W, kSwzRank),
                                 tc::smem_desc(ba + k * 32, W, kSwzRank), id2, k != 0);
#pragma unroll
                for (int k = 0; k < R / 16; ++k)
                    tc::mma_bf16(d, tc::smem_desc(vl + k * 32, W, kSwzRank),
                                 tc::smem_desc(ba + k * 32, W, kSwzRank), id2, 1);
                tc::mma_commit(&sm.acc2_full[b]);
                tc::mma_commit(&sm.empty[st]);
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: row i of the tile ----------------
        const int q = warp & 3;                        // TMEM lane quarter of this warp
        const int i = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        wait(&sm.acc1_full, 0, &err);
        __syncwarp();
        tc::fence_after_sync();
        float v[R];
        if constexpr (R == 16) {
            uint32_t r[16];
            tc::tmem_ld16_sync(tmem + lane_addr, r);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
        } else {
#pragma unroll
            for (int c = 0; c < R / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32_sync(tmem + lane_addr + 32 * c, r);
#pragma unroll
                for (int k = 0; k < 32; ++k) v[32 * c + k] = __uint_as_float(r[k]);
            }
        }
        // V row i -> bf16 high and low parts, K-major with the rank swizzle.
#pragma unroll
        for (int c = 0; c < R / 8; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = v[8 * c + 2 * e], b2 = v[8 * c + 2 * e + 1];
                const float ha = round_bf16(a), hb = round_bf16(b2);
                hw[e] = pack_bf16(ha, hb);
                lw[e] = pack_bf16(a - ha, b2 - hb);
            }
            int pc = c;
            if constexpr (R == 64) pc ^= (i & 7);
            else if constexpr (R == 32) pc ^= (i >> 1) & 3;
            else pc ^= (i >> 2) & 1;
            *reinterpret_cast<uint4 *>(v_hi + i * W + pc * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(v_lo + i * W + pc * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&sm.v_ready);

        const float scale = pa.scale[s];
        uint16_t *yg = pa.y;
        for (int j = 0; j < nn; ++j) {
            const int ii = nk + j, st = ii % kStages, b = j & 1;
            wait(&sm.acc2_full[b], (uint32_t)(j >> 1) & 1u, &err);
            wait(&sm.full[st], (uint32_t)(ii / kStages) & 1u, &err);
            __syncwarp();
            tc::fence_after_sync();
            uint32_t d0[32], d1[32];
            tc::tmem_ld32_sync(tmem + lane_addr + kAcc2Col + 64u * b, d0);
            tc::tmem_ld32_sync(tmem + lane_addr + kAcc2Col + 64u * b + 32, d1);
            tc::fence_before_sync();
            tc::mbar_arrive(&sm.acc2_empty[b]);
            const uint8_t *yt = ring + st * kStageBytes + i * 128;     // row i, 128B swizzle
            const int col0 = o_begin + j * 64;
            uint4 out[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 yv = *reinterpret_cast<const uint4 *>(yt + ((c ^ (i & 7)) * 16));
                uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = 8 * c + 2 * e;
                    const float da = __uint_as_float(n < 32 ? d0[n] : d1[n - 32]);
                    const float db = __uint_as_float(n + 1 < 32 ? d0[n + 1] : d1[n + 1 - 32]);
                    w[e] = pack_bf16(fmaf(scale, da, bf_lo(w[e])), fmaf(scale, db, bf_hi(w[e])));
                }
                out[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            // The stage goes back to the TMA (async proxy) after these generic
            // reads: order them before the release, or a refill can land first.
            tc::fence_proxy_async_smem();
            tc::named_bar(1, 128);                     // every row read from this stage
            if (i == 0) tc::mbar_arrive(&sm.empty[st]);
            if (i < rows && !err) {
                uint16_t *dst = yg + (size_t)(row0 + i) * pa.d_out + col0;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (col0 + 8 * c < o_end) *reinterpret_cast<uint4 *>(dst + 8 * c) = out[c];
            }
        }
    }

    if (err) atomicExch(&sm.error, 1);
    tc::fence_before_sync();
    __syncthreads();
    if (sm.error && tid == 0) atomicExch(pa.hdr + kHdrError, 1);
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

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
cudaError_t launch_r(const PrefillArgs &pa, int grid_tiles, int nsplit, cudaStream_t st) {
    static bool attr = false;
    const size_t smem = prefill_smem_bytes(R);
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    prefill_tc_kernel<R><<<dim3(grid_tiles, nsplit, 1), kPT, smem, st>>>(pa);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int R) { return R == 16 || R == 32 || R == 64; }

cudaError_t launch_prefill_tc(const void *x, void *y, int T, int d_in, int d_out, const void *A_pool,
                              const void *B_pool, int S, int R, const float *scale, const int *hdr,
                              const int4 *ptiles, int grid_tiles, int nsplit, cudaStream_t st) {
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    PrefillArgs pa{};
    const CUtensorMapSwizzle swz_rank = R == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                      : (R == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    bool ok = encode_2d(&pa.mx, x, (uint64_t)d_in, (uint64_t)T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&pa.ma, A_pool, (uint64_t)d_in, (uint64_t)S * R, 64, (uint32_t)R,
                        CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&pa.my, y, (uint64_t)d_out, (uint64_t)T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&pa.mb, B_pool, (uint64_t)R, (uint64_t)S * d_out, (uint32_t)R, 64, swz_rank);
    if (!ok) return cudaErrorInvalidValue;
    pa.y = static_cast<uint16_t *>(y);
    pa.d_in = d_in;
    pa.d_out = d_out;
    pa.scale = scale;
    pa.hdr = const_cast<int *>(hdr);
    pa.ptiles = ptiles;
    pa.cols_per_split = ((d_out + nsplit - 1) / nsplit + 63) / 64 * 64;
    switch (R) {
    case 16: return launch_r<16>(pa, grid_tiles, nsplit, st);
    case 32: return launch_r<32>(pa, grid_tiles, nsplit, st);
    case 64: return launch_r<64>(pa, grid_tiles, nsplit, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace lora
