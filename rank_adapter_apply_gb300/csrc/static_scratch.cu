// lora_apply_static_scratch: the grouped decode path of one layer with its
// scratch in a fixed device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand the library a workspace because they
// cannot allocate device memory when they set it up -- a plugin whose host
// application owns every device allocation through its own pool, a process
// that reserved all device memory up front, or a latency-critical path that
// must not call the allocator (cudaMalloc may synchronise the device and can
// fail at run time). Those callers still pass their inputs and outputs; the
// scratch (token grouping, tile lists, split partials, rank-r intermediates)
// comes from `g_scratch` below.
//
// Properties callers must know:
//  * g_scratch is kStaticScratchBytes (4 MiB) of device memory that every GPU
//    which loads this library holds until the process exits.
//  * Every call looks up the array's device address on the current device
//    with cudaGetSymbolAddress (which allocates nothing), so the address is
//    right after a device reset or in another context of the same device. The
//    first call on a device also loads the library's device code there: make
//    that first call before any stream capture.
//  * All calls share the one array and it keeps the previous call's contents.
//    The arrival counters that must start at zero are cleared on the caller's
//    stream at the start of every call. Two calls whose work overlaps on the
//    GPU (different streams, or different host threads) race on the array and
//    give wrong results; serialise them.
//  * Problems whose scratch does not fit are rejected with LORA_ERR_ARG.
#include "rank_adapter_apply.h"
#include "kernels.cuh"

#include <cuda_runtime.h>

#include <cstdio>
#include <string>

namespace lora {
namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

int fail_static(int code, const char *msg) { return set_last_error(code, msg); }

// Scratch layout for one layer inside the static array: the same regions as a
// context workspace, with the split-partial rows cut to what fits.
bool static_layout(int S, int R, int T, WsLayout *out) {
    WsLayout w = ws_layout(S, R, T, 1);
    const size_t fixed = w.part;                         // everything before the partials
    const size_t row = (size_t)R * sizeof(float);
    if (fixed > kStaticScratchBytes) return false;
    size_t rows = (kStaticScratchBytes - fixed) / row;
    if (rows < (size_t)T) return false;                  // at least one chunk (n_chunks = 1)
    if (rows > (size_t)w.part_rows) rows = (size_t)w.part_rows;
    w.part_rows = (int)rows;
    w.total = fixed + rows * row;
    *out = w;
    return true;
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" int lora_apply_static_scratch(const void *x, void *y, const int32_t *token_slot_idx,
                                         int n_tokens, int d_in, int d_out, int max_loras,
                                         int max_lora_rank, int dtype, const void *A_pool,
                                         const void *B_pool, const float *scale_dev,
                                         const int32_t *rank_dev, void *stream) {
    if (dtype != LORA_DTYPE_F32 && dtype != LORA_DTYPE_BF16)
        return fail_static(LORA_ERR_ARG, "unknown dtype");
    const int rmax = dtype == LORA_DTYPE_BF16 ? 64 : 256;
    if (max_loras < 1 || max_loras > kMaxSlots || max_lora_rank < 8 || max_lora_rank > rmax ||
        max_lora_rank % 8 != 0 || d_in < 1 || d_out < 1 || n_tokens < 0)
        return fail_static(LORA_ERR_ARG, "bad shape: max_loras 1..256, max_lora_rank a multiple "
                                         "of 8 (<= 64 for bf16), d_in, d_out >= 1");
    if (n_tokens == 0) return LORA_OK;
    if (!x || !y || !token_slot_idx || !A_pool || !B_pool || !scale_dev || !rank_dev)
        return fail_static(LORA_ERR_ARG, "NULL pointer argument");
    if (reinterpret_cast<uintptr_t>(A_pool) % 16 || reinterpret_cast<uintptr_t>(B_pool) % 16)
        return fail_static(LORA_ERR_ARG, "slot pools must be 16-byte aligned");
    WsLayout lay;
    if (!static_layout(max_loras, max_lora_rank, n_tokens, &lay)) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "n_tokens %d needs more than the %zu-byte static scratch at max_lora_rank %d",
                 n_tokens, kStaticScratchBytes, max_lora_rank);
        return fail_static(LORA_ERR_ARG, buf);
    }

    // The array's address on the current device, looked up on every call (a
    // cached address would go stale after a device reset or in another
    // context). In host code the name g_scratch is only a host-side stand-in.
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_static(LORA_ERR_CUDA, "cudaGetDevice failed");
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess)
        return fail_static(LORA_ERR_CUDA,
                           (std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e)).c_str());
    char *scratch = static_cast<char *>(p);
    int num_sms = 0;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_static(LORA_ERR_CUDA, "cudaDeviceGetAttribute failed");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Arrival counters of the split reduction and the header start at zero.
    e = cudaMemsetAsync(scratch + lay.counters, 0, (size_t)lay.max_tiles * sizeof(int), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch + lay.hdr, 0, 64 * sizeof(int), st);
    if (e == cudaSuccess)
        e = launch_group_tokens(token_slot_idx, n_tokens, rank_dev, max_loras, 0, scratch, lay, num_sms, st);
    if (e != cudaSuccess)
        return fail_static(LORA_ERR_CUDA, (std::string("launch: ") + cudaGetErrorString(e)).c_str());

    const size_t eb = dtype == LORA_DTYPE_F32 ? 4 : 2;
    const int T = n_tokens;
    const int est_tiles = (T + kTileTokens - 1) / kTileTokens + (max_loras < T ? max_loras : T);
    MultiArgs ma{};
    ma.n = 1;
    LayerArgs &a = ma.l[0];
    a.x = x;
    a.y = y;
    a.A = A_pool;
    a.B = B_pool;
    a.d_in = d_in;
    a.d_out = d_out;
    a.v = reinterpret_cast<float *>(scratch + lay.v);
    a.part = reinterpret_cast<float *>(scratch + lay.part);
    a.counters = reinterpret_cast<int *>(scratch + lay.counters);
    int chunks = (2 * num_sms + est_tiles - 1) / est_tiles;
    if (chunks > kMaxChunks) chunks = kMaxChunks;
    // partial rows of v_stride(R) floats in part_rows rows of R floats
    const long long max_split = (long long)lay.part_rows * max_lora_rank / ((long long)T * v_stride(max_lora_rank));
    if (chunks > max_split) chunks = (int)max_split;
    if (chunks < 1) chunks = 1;
    int cols = ((d_in + chunks - 1) / chunks + 127) / 128 * 128;
    a.chunk_cols = cols;
    a.n_chunks = (d_in + cols - 1) / cols;
    a.vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
             (size_t)d_in * eb % 16 == 0 && (size_t)d_out * eb % 16 == 0) ? 1 : 0;
    GroupView gv{};
    gv.hdr = reinterpret_cast<const int *>(scratch + lay.hdr);
    gv.perm = reinterpret_cast<const int *>(scratch + lay.perm);
    gv.tiles = reinterpret_cast<const int4 *>(scratch + lay.tiles);
    gv.scale = scale_dev;
    gv.rank = rank_dev;
    gv.R = max_lora_rank;
    gv.T = T;
    const int grid_tiles = est_tiles < lay.max_tiles ? est_tiles : lay.max_tiles;
    e = launch_decode(ma, gv, dtype, grid_tiles, a.n_chunks, (d_out + 255) / 256, num_sms, st);
    if (e != cudaSuccess)
        return fail_static(LORA_ERR_CUDA, (std::string("launch: ") + cudaGetErrorString(e)).c_str());
    return LORA_OK;
}
