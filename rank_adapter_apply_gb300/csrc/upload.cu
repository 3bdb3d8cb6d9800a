// Batched slot upload: one kernel copies every adapter of a call from pinned
// host memory into its slot rows, zero-fills the padded ranks and sets the
// slots' scale and rank.
//
// The uploads are the CPU-hit tier of the "Multi-LoRA 适配器缓存生产实战" page
// (section 冷加载延迟, L1: CPU hit -> H2D), whose cost is the adapter_h2d term
// of the TTFT decomposition there. On a Grace-Blackwell node the GPU reads
// pinned host memory directly over the chip-to-chip link, so a batch of small
// adapters (a few hundred KB each) moves in one launch with thousands of
// 16-byte loads in flight, instead of four copy-engine requests per adapter.
//
// Work units (host-computed prefix sums): per entry, 16 KB chunks of the
// A region [R][d_in] (source rows r x d_in contiguous, the rest zero) and
// blocks of 64 rows of B (source rows of r elements, [d_out][r]) written
// into the pool's rank-blocked layout (blocks of b_block(R) ranks, each
// [d_out][b_block(R)]; ranks past r zero).
#include "kernels.cuh"

#include <cuda_runtime.h>

namespace lora {
namespace {

constexpr int kThreads = 256;
constexpr int kAChunk = 16384;   // bytes of the A region per work unit
constexpr int kBRows = 64;       // rows of the B region per work unit

__device__ __forceinline__ uint4 ld_host16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kThreads)
upload_slots_kernel(const __grid_constant__ UploadArgs a) {
    // Which entry and unit this CTA copies.
    const int u = blockIdx.x;
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_start[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const UploadEntry &e = a.e[lo];
    const int local = u - a.unit_start[lo];
    const size_t es = (size_t)a.esize;
    const size_t a_bytes = (size_t)a.R * e.d_in * es;           // whole A region of the slot
    const size_t a_src = (size_t)e.r * e.d_in * es;             // copied part
    const int a_units = (int)((a_bytes + kAChunk - 1) / kAChunk);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (local < a_units) {
        const size_t b0 = (size_t)local * kAChunk;
        const size_t b1 = b0 + kAChunk < a_bytes ? b0 + kAChunk : a_bytes;
        const char *src = static_cast<const char *>(e.A_src);
        char *dst = static_cast<char *>(e.A_dst);
#pragma unroll 4
        for (size_t off = b0 + threadIdx.x * 16; off < b1; off += kThreads * 16) {
            const uint4 v = off < a_src ? ld_host16(src + off) : zero;
            *reinterpret_cast<uint4 *>(dst + off) = v;
        }
    } else {
        const int p0 = (local - a_units) * kBRows;
        const int p1 = p0 + kBRows < e.d_out ? p0 + kBRows : e.d_out;
        const int row_chunks = (int)((size_t)a.R * es / 16);     // 16-byte chunks per slot row
        const int src_chunks = (int)((size_t)e.r * es / 16);
        const int bchunks = (int)((size_t)b_block(a.R) * es / 16); // 16-byte chunks per block row
        const char *src = static_cast<const char *>(e.B_src);
        char *dst = static_cast<char *>(e.B_dst);
        const int total = (p1 - p0) * row_chunks;
#pragma unroll 4
        for (int i = threadIdx.x; i < total; i += kThreads) {
            const int p = p0 + i / row_chunks, c = i % row_chunks;
            const uint4 v = c < src_chunks ? ld_host16(src + ((size_t)p * src_chunks + c) * 16) : zero;
            // chunk c of row p: rank block c / bchunks, chunk c % bchunks of its row there
            const int blk = c / bchunks, w = c - blk * bchunks;
            *reinterpret_cast<uint4 *>(dst + (((size_t)blk * e.d_out + p) * bchunks + w) * 16) = v;
        }
    }
    // The scale and rank of every slot of the call, once.
    if (blockIdx.x == 0 && threadIdx.x < a.n_slots) {
        a.scale_dev[a.slots[threadIdx.x]] = a.scale[threadIdx.x];
        a.rank_dev[a.slots[threadIdx.x]] = a.rank[threadIdx.x];
    }
}

}  // namespace

int upload_units(const UploadEntry &e, int R, int esize) {
    const size_t a_bytes = (size_t)R * e.d_in * esize;
    return (int)((a_bytes + kAChunk - 1) / kAChunk) + (e.d_out + kBRows - 1) / kBRows;
}

cudaError_t launch_upload_slots(const UploadArgs &a, int total_units, cudaStream_t st) {
    if (a.n <= 0 || total_units <= 0) return cudaSuccess;
    upload_slots_kernel<<<total_units, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace lora
