// Internal declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

namespace lora {

constexpr int kTileTokens = 16;      // decode tile: tokens of one slot per CTA row
constexpr int kPrefillRows = 128;    // prefill tile: rows of one same-slot segment
constexpr int kMinPrefillRun = 32;   // shortest run the prefill path may be given (workspace bound)
constexpr int kDefaultPrefillRun = 64;   // shortest run routed to the prefill path by default
constexpr int kMaxLayersPerCall = 8;
constexpr int kMaxChunks = 16;       // split of d_in in the decode shrink
constexpr int kPartialRowCap = 65536;
constexpr int kMaxSlots = 256;

// Header words at the start of the workspace.
enum HdrWord {
    kHdrTiles = 0, kHdrPrefillTiles = 1, kHdrInvalid = 2, kHdrDecodeTokens = 3,
    kHdrError = 6,      // non-zero: a bounded wait gave up (the affected rows were skipped)
    // grouping kernel's grid barrier, finished-CTA count and failure flag (zero between calls)
    kHdrGroupBar = 8, kHdrGroupDone = 9, kHdrGroupFail = 10,
    kHdrSelftest = 11,  // CTAs of the cluster self-test that gave up
};
constexpr int kFusedMaxTokens = 1024;   // batches up to this size take the cluster decode kernel

struct WsLayout {
    size_t hdr, perm, gx, tiles, ptiles, counters, v, part, dpart, total;
    size_t gx_ints;     // ints of the grouping kernel's exchange area
    int max_tiles, max_ptiles, part_rows, max_tokens, R, max_layers;
};

// Grouping kernel (group.cu): CTAs for a batch of T tokens, and the largest
// batch it takes on a GPU with num_sms SMs.
int group_ctas(int T);
int group_max_tokens(int num_sms);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// B pool layout: slot s holds B_s in blocks of kb = b_block(R) consecutive
// ranks, each block [d_out][kb] contiguous; element (i, k) of slot s at
// s * d_out * R + (k / kb) * d_out * kb + i * kb + k % kb. A slot of rank r
// occupies ceil(r / kb) contiguous runs, so reading it touches no padding
// past them. kb = 32 where max_lora_rank allows it (at rank 32 and below the
// layout is the plain [d_out][R] one), else 16, else 8.
__host__ __device__ constexpr int b_block(int R) { return R % 32 == 0 ? 32 : (R % 16 == 0 ? 16 : 8); }

// Row stride (floats) of the decode path's v: whole 16-rank blocks, which the
// bf16 path stores in MMA fragment order (the fp32 path uses the first R).
__host__ __device__ constexpr int v_stride(int R) { return (R + 15) / 16 * 16; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the kernel before it in the stream still runs (its launch and ramp-up
// overlap that kernel's tail). Every kernel launched this way calls
// grid_dependency_wait() before it touches memory that an earlier kernel of
// the stream may read or write; once the wait returns, every earlier kernel
// has completed (each of them waited on its own predecessor in turn).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Kernel attributes (e.g. the dynamic shared-memory limit) are per device:
// one bit per device (ids 0..63) records that the current device has them.
inline bool device_bit(const std::atomic<uint64_t> &f) {
    int d = 0;
    cudaGetDevice(&d);
    return (f.load(std::memory_order_acquire) >> (d & 63)) & 1u;
}
inline void set_device_bit(std::atomic<uint64_t> &f) {
    int d = 0;
    cudaGetDevice(&d);
    f.fetch_or(uint64_t(1) << (d & 63), std::memory_order_release);
}

inline WsLayout ws_layout(int S, int R, int max_tokens, int max_layers) {
    WsLayout w{};
    int T = max_tokens > 0 ? max_tokens : 1;
    w.max_tokens = T;
    w.R = R;
    w.max_layers = max_layers;
    w.max_tiles = (T + kTileTokens - 1) / kTileTokens + (S < T ? S : T) + 1;
    w.max_ptiles = T / kPrefillRows + T / kMinPrefillRun + 2;
    long long pr = (long long)kMaxChunks * T;
    w.part_rows = (int)(pr < kPartialRowCap ? pr : (kPartialRowCap > T ? kPartialRowCap : T));
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    w.hdr = take(64 * sizeof(int));
    w.perm = take((size_t)T * sizeof(int));
    const int G = group_ctas(T);
    w.gx_ints = G > 1 ? (size_t)G * (3 + S) : 1;
    w.gx = take(w.gx_ints * sizeof(int));
    w.tiles = take((size_t)w.max_tiles * sizeof(int4));
    w.ptiles = take((size_t)w.max_ptiles * sizeof(int4));
    w.counters = take((size_t)max_layers * w.max_tiles * sizeof(int));
    w.v = take((size_t)max_layers * T * v_stride(R) * sizeof(float));
    w.part = take((size_t)max_layers * w.part_rows * R * sizeof(float));
    // The decode kernels' own partials: they run beside the prefill kernels
    // (which use `part`) on a second stream.
    w.dpart = take((size_t)max_layers * w.part_rows * R * sizeof(float));
    w.total = o;
    return w;
}

// Per-layer arguments of one decode launch (blockIdx.z selects the layer).
struct LayerArgs {
    const void *x;
    void *y;
    const void *A;       // pool base [S][R][d_in]
    const void *B;       // pool base [S][d_out][R]
    float *v;            // [T][R] fp32 rank-r intermediates, by grouped position
    float *part;         // split partials: chunk c, row t at (c * T + t) * v_stride(R)
    int *counters;       // [max_tiles] arrival counters (self-resetting)
    int d_in, d_out;
    int n_chunks, chunk_cols;
    int out_cols;        // cluster decode: output columns per CTA of a cluster
    int vec;             // 1: rows are 16-byte aligned, 128-bit accesses allowed
};

struct MultiArgs {
    LayerArgs l[kMaxLayersPerCall];
    int n;
};

// Grouping results shared by every layer of a call.
struct GroupView {
    const int *hdr;
    const int *perm;
    const int4 *tiles;
    const float *scale;
    const int *rank;
    int R;
    int T;
};

cudaError_t launch_group_tokens(const int32_t *idx, int T, const int *rank_dev, int S,
                                int min_run, char *ws, const WsLayout &lay, int num_sms, cudaStream_t st);
cudaError_t launch_decode(const MultiArgs &ma, const GroupView &gv, int dtype, int grid_tiles,
                          int max_chunks, int max_dblocks, int num_sms, cudaStream_t st);
// Single-launch decode step on 8-CTA clusters, batches of at most
// kFusedMaxTokens bf16 tokens: one cluster per (layer, tile of <= 16 tokens),
// CTA c of a cluster owns columns [c*chunk_cols, ...) of d_in and
// [c*out_cols, ...) of d_out.
struct FusedArgs {
    LayerArgs l[kMaxLayersPerCall];   // x, y, A, B, d_in, d_out, chunk_cols, out_cols
    int n;
    const int32_t *idx;
    int T, S, R;
    const int *rank;
    const float *scale;
    int *hdr;                         // workspace header: invalid-index count, error word
    int early;                        // read all but y before waiting on the previous kernel
};
constexpr int kClusterSize = 8;
int cluster_decode_kb(int R);
size_t cluster_decode_smem(int R);
cudaError_t launch_cluster_decode(const FusedArgs &fa, int tiles, cudaStream_t st, bool pdl);

// Tensor-core prefill over the prefill tiles of the workspace, every layer of
// one call: a shrink kernel that reads each x tile once for all the layers
// sharing that input and writes fp32 partials of V = x A^T, then a persistent
// expand kernel that streams y through a TMA ring and adds scale * V B^T.
struct PrefillLayer {
    const void *x;        // [T][d_in] bf16
    void *y;              // [T][d_out] bf16, updated in place
    const void *A;        // pool [S][R][d_in]
    const void *B;        // pool [S][d_out][R]
    float *part;          // [part_rows][R] fp32 partials of V (chunk c at row c*T)
    int d_in, d_out;
};
bool prefill_tc_supported(int R);
// *kernels (if not NULL) is increased by the number of kernels queued (2 or 3).
cudaError_t launch_prefill_tc(const PrefillLayer *layers, int n, int T, int S, int R, const float *scale,
                              int *hdr, const int4 *ptiles, int grid_tiles, int part_rows, int num_sms,
                              cudaStream_t st, int *kernels);

// Batched slot upload (upload.cu): one kernel reads every adapter of a call
// from page-locked host memory (device-mapped) into its slot rows.
constexpr int kMaxUploadSlots = 128;
constexpr int kMaxUploadEntries = 256;     // adapters x layers per launch
struct UploadEntry {
    const void *A_src;      // host, device-mapped: [r][d_in]
    const void *B_src;      // host, device-mapped: [d_out][r]
    void *A_dst;            // slot rows of the A pool: [R][d_in]
    void *B_dst;            // slot rows of the B pool: [d_out][R]
    int d_in, d_out, r, pad;
};
struct UploadArgs {
    UploadEntry e[kMaxUploadEntries];
    int unit_start[kMaxUploadEntries];
    int slots[kMaxUploadSlots];
    float scale[kMaxUploadSlots];
    int rank[kMaxUploadSlots];
    float *scale_dev;
    int *rank_dev;
    int n, n_slots, R, esize;
};
int upload_units(const UploadEntry &e, int R, int esize);
cudaError_t launch_upload_slots(const UploadArgs &a, int total_units, cudaStream_t st);

// Record the message returned by lora_last_error() for this thread; returns code.
int set_last_error(int code, const char *msg);

cudaError_t launch_set_slot(float *scale_dev, int *rank_dev, int slot, float scale, int rank,
                            cudaStream_t st);
cudaError_t launch_selftest_wait(int *err_word, uint32_t limit, cudaStream_t st);
// The cluster decode kernel's exchange wait on a barrier nothing arrives on
// (two-CTA cluster); *gave_up += 1 for each CTA that gave up.
cudaError_t launch_selftest_cluster_wait(int *err_word, int *gave_up, uint32_t limit, cudaStream_t st);

}  // namespace lora
