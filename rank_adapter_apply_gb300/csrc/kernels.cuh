// Internal declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace lora {

constexpr int kTileTokens = 16;      // decode tile: tokens of one slot per CTA row
constexpr int kPrefillRows = 128;    // prefill tile: rows of one same-slot segment
constexpr int kMinPrefillRun = 64;   // shortest run routed to the prefill path
constexpr int kMaxLayersPerCall = 8;
constexpr int kMaxChunks = 16;       // split of d_in in the decode shrink
constexpr int kPartialRowCap = 65536;
constexpr int kMaxSlots = 256;

// Header words at the start of the workspace.
enum HdrWord {
    kHdrTiles = 0, kHdrPrefillTiles = 1, kHdrInvalid = 2, kHdrDecodeTokens = 3,
    kHdrEpoch = 4,      // launches of the fused decode kernel so far (flag target = epoch + 1)
    kHdrExit = 5,       // CTAs of the running fused launch that have finished
    kHdrError = 6,      // non-zero: a bounded wait gave up (the affected rows were skipped)
};
constexpr int kFusedMaxTokens = 1024;   // batches up to this size take the fused decode kernel

struct WsLayout {
    size_t hdr, perm, run_start, run_of, tiles, ptiles, counters, flags, v, part, total;
    int max_tiles, max_ptiles, part_rows, max_tokens, R, max_layers;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

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
    w.run_start = take((size_t)(T + 1) * sizeof(int));
    w.run_of = take((size_t)T * sizeof(int));
    w.tiles = take((size_t)w.max_tiles * sizeof(int4));
    w.ptiles = take((size_t)w.max_ptiles * sizeof(int4));
    w.counters = take((size_t)max_layers * w.max_tiles * sizeof(int));
    w.flags = take((size_t)max_layers * w.max_tiles * kMaxChunks * sizeof(unsigned));
    w.v = take((size_t)max_layers * T * R * sizeof(float));
    w.part = take((size_t)max_layers * w.part_rows * R * sizeof(float));
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
    float *part;         // [n_chunks * T][R] split partials
    int *counters;       // [max_tiles] arrival counters (self-resetting)
    int d_in, d_out;
    int n_chunks, chunk_cols;
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
                                int min_run, char *ws, const WsLayout &lay, cudaStream_t st);
cudaError_t launch_decode(const MultiArgs &ma, const GroupView &gv, int dtype, int grid_tiles,
                          int max_chunks, int max_dblocks, cudaStream_t st);
// Fused decode step for batches of at most kFusedMaxTokens tokens (bf16 only).
struct FusedArgs {
    LayerArgs l[kMaxLayersPerCall];   // x, y, A, B, d_in, d_out, n_chunks, chunk_cols
    int n;
    const int32_t *idx;
    int T, S, R;
    const int *rank;
    const float *scale;
    float *part;                      // layer l at part + l * part_layer_stride
    size_t part_layer_stride;         // floats
    unsigned *flags;                  // [n][max_tiles][kMaxChunks]
    int max_tiles;
    int *hdr;
};
int fused_decode_ctas_per_sm(int max_lora_rank);
cudaError_t launch_fused_decode(const FusedArgs &fa, int grid, cudaStream_t st);

cudaError_t launch_set_slot(float *scale_dev, int *rank_dev, int slot, float scale, int rank,
                            cudaStream_t st);

}  // namespace lora
