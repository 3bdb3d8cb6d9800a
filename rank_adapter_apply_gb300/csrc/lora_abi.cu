// C ABI of the multi-LoRA delta library: context, slot uploads, apply calls
// and the host slot table. Every declaration lives in include/rank_adapter_apply.h.
#include "rank_adapter_apply.h"
#include "kernels.cuh"
#include "slot_table.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

using namespace lora;

namespace {

// Tiles of <= kTileTokens tokens over the slots a batch uses: each used slot
// adds at most kTileTokens - 1 padding places, so
// sum_s ceil(n_s / 16) <= (T + 15 * min(S, T)) / 16.
int max_decode_tiles(int T, int S) {
    const long long used = S < T ? S : T;
    return (int)(((long long)T + (kTileTokens - 1) * used) / kTileTokens);
}


thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

#define CUDA_TRY(call)                                                                   \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return fail(LORA_ERR_CUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_),   \
                        __FILE__, __LINE__);                                             \
    } while (0)

}  // namespace

int lora::set_last_error(int code, const char *msg) {
    g_err = msg;
    return code;
}

namespace {

struct UploadTiming {
    cudaEvent_t start, end;
};

}  // namespace

struct lora_ctx {
    int S = 0, R = 0, max_tokens = 0, max_layers = 0, dtype = 0, n_layers = 0;
    bool device = false;
    std::vector<lora_layer_desc> layers;
    float *scale_dev = nullptr;
    int32_t *rank_dev = nullptr;
    char *ws = nullptr;
    size_t ws_bytes = 0;
    WsLayout lay{};
    cudaStream_t compute = nullptr, upload = nullptr;
    SlotTable table;
    // Uploads and evictions: call k records up_ev[k % size] on the upload
    // stream; slot_up[s] = the newest such call that wrote slot s and that no
    // apply has waited for yet (-1: none).
    std::vector<cudaEvent_t> up_ev;
    std::vector<int64_t> slot_up;
    int64_t n_up = 0;
    cudaEvent_t compute_done = nullptr;
    bool compute_recorded = false;
    std::vector<UploadTiming> timing;
    std::vector<UploadTiming> timing_free;   // timing events of harvested uploads, reused
    double upload_seconds = 0.0;
    uint64_t uploads = 0, upload_bytes = 0, invalid_seen = 0;
    uint64_t cluster_applies = 0, grouped_applies = 0;   // which path served each apply
    uint64_t launches = 0;        // kernels queued by this context's calls
    int prefill_min = 0;          // shortest same-slot run sent to the tensor-core prefill kernel
    int small_batch = -1;         // batches up to this size take the cluster decode kernel; -1: by rank
    int inputs_ready = 0;         // caller: x, slot ids, pools not written by the preceding kernel
    int num_sms = 148;
    // Per-slot tracking (lora_set_slot_tracking): apply i records ring[i % kRing];
    // slot_gen[s] is the last apply issued while slot s was in flight.
    int track = 0;
    std::vector<cudaEvent_t> ring;
    std::vector<int64_t> slot_gen;
    int64_t n_apply = 0;
    // Host-buffer path: call k records host_ev[k % kHostRing] on the download
    // stream after its copies back (on the compute stream under capture);
    // buf_use maps each device staging buffer to the last call that used it;
    // h2d_done marks a call's copies in (upload stream), apply_done its apply.
    std::vector<cudaEvent_t> host_ev;
    std::vector<std::pair<const void *, int64_t>> buf_use;
    int64_t n_host = 0, host_forgot = -1;
    cudaEvent_t h2d_done = nullptr, apply_done = nullptr;
    cudaStream_t down = nullptr;    // copies back of the host-buffer path (created on first use)
    // The decode kernels of a grouped apply run on `side`, beside the prefill
    // kernels on the compute stream: fork after the grouping, join at the end.
    cudaStream_t side = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    // lora_assign_tokens: open-addressing table adapter id -> distinct index
    std::vector<uint64_t> tok_key;
    std::vector<int> tok_val, tok_rank;
    // lora_serve_step: the registered host adapter store (id -> index; per
    // adapter rank, alpha and per-layer host pointers), the warm set, scratch
    std::unordered_map<uint64_t, int> store;
    std::vector<int> store_rank;
    std::vector<float> store_alpha;
    std::vector<const void *> store_A, store_B;
    std::unordered_set<uint64_t> warm;
    std::vector<int> step_tok, step_group, step_slot, step_need;
    std::vector<uint64_t> step_id, step_ev;
    std::vector<int> up_slots, up_ranks;     // uploads of one serving-step group
    std::vector<float> up_alphas;
    std::vector<const void *> up_A, up_B;

    lora_ctx(int S_, int R_) : table(S_, R_) {}
};

namespace {

int elem_bytes(int dtype) { return dtype == LORA_DTYPE_F32 ? 4 : 2; }

constexpr int kRing = 64;

// After the launches of one apply: the stream-wide event, and with slot
// tracking the ring event of this apply for every slot in flight.
cudaError_t note_apply(lora_ctx *c) {
    cudaError_t e = cudaEventRecord(c->compute_done, c->compute);
    if (e != cudaSuccess) return e;
    c->compute_recorded = true;
    if (!c->track) return cudaSuccess;
    e = cudaEventRecord(c->ring[c->n_apply % kRing], c->compute);
    if (e != cudaSuccess) return e;
    for (int s = 0; s < c->S; ++s)
        if (c->table.refs(s) > 0) c->slot_gen[s] = c->n_apply;
    ++c->n_apply;
    return cudaSuccess;
}

// Order the upload stream after every queued apply that may read `slot`:
// all of them by default; with slot tracking only the last apply issued while
// the slot was in flight (a ring event reused by a later apply only makes the
// wait longer, never too short).
cudaError_t wait_slot_reads(lora_ctx *c, int slot) {
    if (c->track) {
        const int64_t g = c->slot_gen[slot];
        return g >= 0 ? cudaStreamWaitEvent(c->upload, c->ring[g % kRing], 0) : cudaSuccess;
    }
    return c->compute_recorded ? cudaStreamWaitEvent(c->upload, c->compute_done, 0) : cudaSuccess;
}

// After the upload-stream work of one upload or eviction call: one event for
// every slot it wrote.
cudaError_t note_upload(lora_ctx *c, const int *slots, int n) {
    const int64_t k = c->n_up++;
    cudaError_t e = cudaEventRecord(c->up_ev[k % (int64_t)c->up_ev.size()], c->upload);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < n; ++i) c->slot_up[slots[i]] = k;
    return cudaSuccess;
}

// wait_slot_reads for several slots, each distinct event waited on once.
cudaError_t wait_slots_reads(lora_ctx *c, const std::vector<int> &slots) {
    if (!c->track) return slots.empty() ? cudaSuccess : wait_slot_reads(c, slots[0]);
    std::vector<int> idx;
    for (int s : slots) {
        const int64_t g = c->slot_gen[s];
        if (g >= 0) idx.push_back((int)(g % kRing));
    }
    std::sort(idx.begin(), idx.end());
    idx.erase(std::unique(idx.begin(), idx.end()), idx.end());
    for (int i : idx) {
        cudaError_t e = cudaStreamWaitEvent(c->upload, c->ring[i], 0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// True when the current device reads host memory through the host's page
// tables (any host address is valid in a kernel); checked once per device.
bool host_pages_visible() {
    static std::atomic<uint64_t> known{0}, yes{0};
    if (device_bit(known)) return device_bit(yes);
    int dev = 0, a = 0, b = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&a, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&b, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) != cudaSuccess) {
        cudaGetLastError();
        a = b = 0;
    }
    if (a == 1 && b == 1) set_device_bit(yes);
    set_device_bit(known);
    return a == 1 && b == 1;
}

// Move finished upload timings into upload_seconds (blocking when `wait`).
int harvest_timings(lora_ctx *c, bool wait) {
    std::vector<UploadTiming> keep;
    for (auto &t : c->timing) {
        cudaError_t q = wait ? cudaEventSynchronize(t.end) : cudaEventQuery(t.end);
        if (q == cudaErrorNotReady) {
            keep.push_back(t);
            continue;
        }
        if (q != cudaSuccess) return fail(LORA_ERR_CUDA, "upload event: %s", cudaGetErrorString(q));
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, t.start, t.end) == cudaSuccess) c->upload_seconds += ms * 1e-3;
        c->timing_free.push_back(t);
    }
    c->timing.swap(keep);
    return LORA_OK;
}

// A pair of timing events for one upload call: a harvested pair if there is
// one (creating events costs a driver call each), else a new pair.
cudaError_t take_timing(lora_ctx *c, UploadTiming *t) {
    if (!c->timing_free.empty()) {
        *t = c->timing_free.back();
        c->timing_free.pop_back();
        return cudaSuccess;
    }
    cudaError_t e = cudaEventCreate(&t->start);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&t->end);
    if (e != cudaSuccess) cudaEventDestroy(t->start);
    return e;
}

bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return false;
    return st != cudaStreamCaptureStatusNone;
}

constexpr int kHostRing = 8;

struct Copy {
    void *dst;
    const void *src;
    size_t bytes;
};

// Joins copies that continue one another in both address spaces (in the
// order given; the first copy of a run keeps its place).
std::vector<Copy> merge_copies(const std::vector<Copy> &cs) {
    std::vector<Copy> out;
    for (const Copy &c : cs) {
        if (!out.empty()) {
            Copy &p = out.back();
            if (static_cast<const char *>(p.src) + p.bytes == c.src &&
                static_cast<char *>(p.dst) + p.bytes == c.dst) {
                p.bytes += c.bytes;
                continue;
            }
        }
        out.push_back(c);
    }
    return out;
}

}  // namespace

extern "C" {

const char *lora_last_error(void) { return g_err.c_str(); }

size_t lora_workspace_bytes(int max_loras, int max_lora_rank, int max_tokens,
                            int max_layers_per_call) {
    if (max_loras < 1 || max_lora_rank < 1 || max_tokens < 0 || max_layers_per_call < 1 ||
        max_layers_per_call > kMaxLayersPerCall)
        return 0;
    return ws_layout(max_loras, max_lora_rank, max_tokens, max_layers_per_call).total;
}

uint64_t lora_adapter_bytes(int n_layers, const int *d_in, const int *d_out, int rank,
                            int bytes_per_param) {
    if (n_layers < 0 || (n_layers > 0 && (!d_in || !d_out)) || rank < 0 || bytes_per_param < 0)
        return 0;
    uint64_t b = 0;
    for (int l = 0; l < n_layers; ++l)
        b += ((uint64_t)d_in[l] + (uint64_t)d_out[l]) * (uint64_t)rank * (uint64_t)bytes_per_param;
    return b;
}

int lora_slots_init(lora_ctx **out, int max_loras, int max_lora_rank, int max_tokens,
                    int max_layers_per_call, int dtype, int n_layers,
                    const lora_layer_desc *layers, float *scale_dev, int32_t *rank_dev,
                    void *workspace, size_t workspace_bytes, void *compute_stream,
                    void *upload_stream) {
    if (!out) return fail(LORA_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (max_loras < 1 || max_loras > kMaxSlots)
        return fail(LORA_ERR_ARG, "max_loras must be in 1..%d", kMaxSlots);
    if (dtype != LORA_DTYPE_F32 && dtype != LORA_DTYPE_BF16)
        return fail(LORA_ERR_ARG, "unknown dtype %d", dtype);
    const int rmax = dtype == LORA_DTYPE_BF16 ? 64 : 256;
    if (max_lora_rank < 8 || max_lora_rank > rmax || max_lora_rank % 8 != 0)
        return fail(LORA_ERR_ARG, "max_lora_rank must be a multiple of 8 in 8..%d", rmax);
    if (n_layers < 0) return fail(LORA_ERR_ARG, "n_layers < 0");
    auto *c = new lora_ctx(max_loras, max_lora_rank);
    c->S = max_loras;
    c->R = max_lora_rank;
    c->dtype = dtype;
    c->n_layers = n_layers;
    if (n_layers == 0) {          // host-only slot table: no CUDA call at all
        *out = c;
        return LORA_OK;
    }
    auto reject = [&](int code, const char *msg) {
        delete c;
        return fail(code, "%s", msg);
    };
    if (!layers || !scale_dev || !rank_dev || !workspace)
        return reject(LORA_ERR_ARG, "layers, scale_dev, rank_dev and workspace are required");
    if (max_tokens < 1) return reject(LORA_ERR_ARG, "max_tokens must be >= 1");
    if (max_layers_per_call < 1 || max_layers_per_call > kMaxLayersPerCall)
        return reject(LORA_ERR_ARG, "max_layers_per_call must be in 1..8");
    for (int l = 0; l < n_layers; ++l)
        if (layers[l].d_in < 1 || layers[l].d_out < 1 || !layers[l].A_pool || !layers[l].B_pool)
            return reject(LORA_ERR_ARG, "layer with bad shape or NULL pool");
    for (int l = 0; l < n_layers; ++l)
        if (reinterpret_cast<uintptr_t>(layers[l].A_pool) % 16 != 0 ||
            reinterpret_cast<uintptr_t>(layers[l].B_pool) % 16 != 0)
            return reject(LORA_ERR_ARG, "slot pools must be 16-byte aligned");
    c->lay = ws_layout(max_loras, max_lora_rank, max_tokens, max_layers_per_call);
    if (workspace_bytes < c->lay.total) return reject(LORA_ERR_ARG, "workspace too small");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return reject(LORA_ERR_ARG, "workspace must be 256-byte aligned");
    c->device = true;
    c->prefill_min = kDefaultPrefillRun;
    c->max_tokens = max_tokens;
    c->max_layers = max_layers_per_call;
    c->layers.assign(layers, layers + n_layers);
    c->scale_dev = scale_dev;
    c->rank_dev = rank_dev;
    c->ws = static_cast<char *>(workspace);
    c->ws_bytes = workspace_bytes;
    c->compute = static_cast<cudaStream_t>(compute_stream);
    c->upload = static_cast<cudaStream_t>(upload_stream);
    c->up_ev.assign(max_loras, nullptr);
    c->slot_up.assign(max_loras, -1);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && max_tokens > group_max_tokens(c->num_sms)) {
        delete c;
        return fail(LORA_ERR_ARG, "max_tokens %d above the %d tokens one apply may take on this GPU", max_tokens,
                    group_max_tokens(c->num_sms));
    }
    for (int s = 0; s < max_loras && e == cudaSuccess; ++s)
        e = cudaEventCreateWithFlags(&c->up_ev[s], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->compute_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->fork_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->join_ev, cudaEventDisableTiming);
    // Empty table: every slot rank 0; workspace zeroed (arrival counters start at 0).
    if (e == cudaSuccess) e = cudaMemsetAsync(rank_dev, 0, sizeof(int32_t) * max_loras, c->compute);
    if (e == cudaSuccess) e = cudaMemsetAsync(scale_dev, 0, sizeof(float) * max_loras, c->compute);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, c->lay.total, c->compute);
    if (e == cudaSuccess) e = cudaEventRecord(c->compute_done, c->compute);
    if (e != cudaSuccess) {
        lora_destroy(c);
        return fail(LORA_ERR_CUDA, "lora_slots_init: %s", cudaGetErrorString(e));
    }
    c->compute_recorded = true;
    *out = c;
    return LORA_OK;
}

void lora_destroy(lora_ctx *c) {
    if (!c) return;
    if (c->device) {
        if (c->upload) cudaStreamSynchronize(c->upload);
        if (c->compute) cudaStreamSynchronize(c->compute);
        harvest_timings(c, true);
        for (auto &t : c->timing) {                // (only if a harvest failed)
            cudaEventDestroy(t.start);
            cudaEventDestroy(t.end);
        }
        for (auto &t : c->timing_free) {
            cudaEventDestroy(t.start);
            cudaEventDestroy(t.end);
        }
        for (auto ev : c->up_ev)
            if (ev) cudaEventDestroy(ev);
        if (c->compute_done) cudaEventDestroy(c->compute_done);
        for (auto ev : c->ring)
            if (ev) cudaEventDestroy(ev);
        if (c->down) cudaStreamSynchronize(c->down);
        if (c->side) cudaStreamSynchronize(c->side);
        if (c->fork_ev) cudaEventDestroy(c->fork_ev);
        if (c->join_ev) cudaEventDestroy(c->join_ev);
        if (c->side) cudaStreamDestroy(c->side);
        for (auto ev : c->host_ev)
            if (ev) cudaEventDestroy(ev);
        if (c->h2d_done) cudaEventDestroy(c->h2d_done);
        if (c->apply_done) cudaEventDestroy(c->apply_done);
        if (c->down) cudaStreamDestroy(c->down);
    }
    delete c;
}

int lora_load_slot(lora_ctx *c, int slot, const void *const *A_host, const void *const *B_host,
                   int rank, float alpha) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (slot < 0 || slot >= c->S) return fail(LORA_ERR_ARG, "slot %d out of range", slot);
    if (rank < 1 || rank > c->R)
        return fail(LORA_ERR_RANK, "LoRA rank %d exceeds maximum %d (or is < 1)", rank, c->R);
    if (!std::isfinite(alpha)) return fail(LORA_ERR_ARG, "alpha is not finite");
    if (!c->device) {                 // host-only table: the upload is only recorded
        c->table.mark_loaded(slot);
        c->uploads += 1;
        return LORA_OK;
    }
    if (!A_host || !B_host) return fail(LORA_ERR_ARG, "A_host / B_host is NULL");
    for (int l = 0; l < c->n_layers; ++l)
        if (!A_host[l] || !B_host[l]) return fail(LORA_ERR_ARG, "layer %d weights are NULL", l);

    const size_t e = elem_bytes(c->dtype);
    const size_t R = c->R, r = rank;
    UploadTiming tm{};
    CUDA_TRY(take_timing(c, &tm));
    // Never overwrite a slot that queued compute work may still read.
    CUDA_TRY(wait_slot_reads(c, slot));
    CUDA_TRY(cudaEventRecord(tm.start, c->upload));
    uint64_t bytes = 0;
    for (int l = 0; l < c->n_layers; ++l) {
        const lora_layer_desc &L = c->layers[l];
        const size_t din = L.d_in, dout = L.d_out;
        char *A = static_cast<char *>(L.A_pool) + (size_t)slot * R * din * e;
        char *B = static_cast<char *>(L.B_pool) + (size_t)slot * dout * R * e;
        CUDA_TRY(cudaMemcpyAsync(A, A_host[l], r * din * e, cudaMemcpyHostToDevice, c->upload));
        if (r < R) CUDA_TRY(cudaMemsetAsync(A + r * din * e, 0, (R - r) * din * e, c->upload));
        // B into the rank-blocked pool layout: one 2D copy per block of
        // kb ranks (rows of kb elements, the host rows r elements apart);
        // ranks past r zero
        const size_t kb = (size_t)b_block(c->R);
        if (r < R) CUDA_TRY(cudaMemsetAsync(B, 0, dout * R * e, c->upload));
        for (size_t k0 = 0; k0 < r; k0 += kb) {
            const size_t w = std::min(kb, r - k0);
            CUDA_TRY(cudaMemcpy2DAsync(B + k0 * dout * e, kb * e, static_cast<const char *>(B_host[l]) + k0 * e,
                                       r * e, w * e, dout, cudaMemcpyHostToDevice, c->upload));
        }
        bytes += (din + dout) * r * e;
    }
    CUDA_TRY(launch_set_slot(c->scale_dev, c->rank_dev, slot, alpha / (float)rank, rank, c->upload));
    ++c->launches;
    CUDA_TRY(cudaEventRecord(tm.end, c->upload));
    CUDA_TRY(note_upload(c, &slot, 1));
    c->timing.push_back(tm);
    c->uploads += 1;
    c->upload_bytes += bytes;
    c->table.mark_loaded(slot);
    if (c->timing.size() > 256) harvest_timings(c, false);
    return LORA_OK;
}

int lora_load_slots(lora_ctx *c, int n, const int *slots, const void *const *A_host,
                    const void *const *B_host, const int *ranks, const float *alphas) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!c->device) return fail(LORA_ERR_STATE, "host-only context has no slot pools");
    if (n < 0) return fail(LORA_ERR_ARG, "n must be >= 0");
    if (n == 0) return LORA_OK;
    if (!slots || !A_host || !B_host || !ranks || !alphas) return fail(LORA_ERR_ARG, "NULL argument");
    const int L = c->n_layers;
    const size_t e = elem_bytes(c->dtype);
    // Validate everything before anything is queued.
    std::vector<char> seen(c->S, 0);
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= c->S) return fail(LORA_ERR_ARG, "slot %d out of range", slots[i]);
        if (seen[slots[i]]) return fail(LORA_ERR_ARG, "slot %d appears twice", slots[i]);
        seen[slots[i]] = 1;
        if (ranks[i] < 1 || ranks[i] > c->R)
            return fail(LORA_ERR_RANK, "LoRA rank %d exceeds maximum %d (or is < 1)", ranks[i], c->R);
        if (!std::isfinite(alphas[i])) return fail(LORA_ERR_ARG, "alpha %d is not finite", i);
        for (int l = 0; l < L; ++l)
            if (!A_host[(size_t)i * L + l] || !B_host[(size_t)i * L + l])
                return fail(LORA_ERR_ARG, "adapter %d layer %d weights are NULL", i, l);
    }
    // Adapters the kernel can read: host pointers the GPU reaches at the same
    // address, 16-byte aligned rows. When the GPU walks the host's page tables
    // every host address qualifies and no per-pointer lookup is needed;
    // otherwise each pointer must be device-mapped pinned memory. The others
    // take the copy-engine path of lora_load_slot.
    const bool all_host = host_pages_visible();
    std::vector<int> direct, copies;
    for (int i = 0; i < n; ++i) {
        bool ok = ((size_t)ranks[i] * e) % 16 == 0;
        for (int l = 0; l < L && ok; ++l) {
            const void *p[2] = {A_host[(size_t)i * L + l], B_host[(size_t)i * L + l]};
            for (int q = 0; q < 2 && ok; ++q) {
                ok = reinterpret_cast<uintptr_t>(p[q]) % 16 == 0;
                if (ok && !all_host) {
                    void *dp = nullptr;
                    ok = cudaHostGetDevicePointer(&dp, const_cast<void *>(p[q]), 0) == cudaSuccess && dp == p[q];
                }
            }
            ok = ok && ((size_t)c->layers[l].d_in * e) % 16 == 0;
        }
        if (!all_host) cudaGetLastError();     // clear a lookup failure of an unmapped pointer
        (ok ? direct : copies).push_back(i);
    }
    for (int i : copies) {
        int rc = lora_load_slot(c, slots[i], A_host + (size_t)i * L, B_host + (size_t)i * L, ranks[i], alphas[i]);
        if (rc != LORA_OK) return rc;
    }
    const int per_launch = std::min(kMaxUploadSlots, kMaxUploadEntries / (L > 0 ? L : 1));
    for (size_t b0 = 0; b0 < direct.size(); b0 += per_launch) {
        const size_t b1 = std::min(direct.size(), b0 + (size_t)per_launch);
        UploadArgs ua{};
        ua.R = c->R;
        ua.esize = (int)e;
        ua.scale_dev = c->scale_dev;
        ua.rank_dev = c->rank_dev;
        int units = 0;
        uint64_t bytes = 0;
        std::vector<int> wslots;
        for (size_t k = b0; k < b1; ++k) wslots.push_back(slots[direct[k]]);
        CUDA_TRY(wait_slots_reads(c, wslots));
        for (size_t k = b0; k < b1; ++k) {
            const int i = direct[k], s = slots[i];
            for (int l = 0; l < L; ++l) {
                const lora_layer_desc &D = c->layers[l];
                UploadEntry &u = ua.e[ua.n];
                u.A_src = A_host[(size_t)i * L + l];
                u.B_src = B_host[(size_t)i * L + l];
                u.A_dst = static_cast<char *>(D.A_pool) + (size_t)s * c->R * D.d_in * e;
                u.B_dst = static_cast<char *>(D.B_pool) + (size_t)s * D.d_out * c->R * e;
                u.d_in = D.d_in;
                u.d_out = D.d_out;
                u.r = ranks[i];
                ua.unit_start[ua.n] = units;
                units += upload_units(u, c->R, (int)e);
                bytes += ((uint64_t)D.d_in + D.d_out) * ranks[i] * e;
                ++ua.n;
            }
            ua.slots[ua.n_slots] = s;
            ua.scale[ua.n_slots] = alphas[i] / (float)ranks[i];
            ua.rank[ua.n_slots] = ranks[i];
            ++ua.n_slots;
        }
        UploadTiming tm{};
        CUDA_TRY(take_timing(c, &tm));
        CUDA_TRY(cudaEventRecord(tm.start, c->upload));
        CUDA_TRY(launch_upload_slots(ua, units, c->upload));
        ++c->launches;
        CUDA_TRY(cudaEventRecord(tm.end, c->upload));
        CUDA_TRY(note_upload(c, ua.slots, ua.n_slots));
        c->timing.push_back(tm);
        c->uploads += (uint64_t)ua.n_slots;
        c->upload_bytes += bytes;
        for (int k = 0; k < ua.n_slots; ++k) c->table.mark_loaded(ua.slots[k]);
    }
    if (c->timing.size() > 256) harvest_timings(c, false);
    return LORA_OK;
}

namespace {

// Single-launch decode step on 8-CTA clusters. Returns LORA_OK, an error, or 1
// when the shapes or alignment do not allow it.
int fused_apply(lora_ctx *c, int n, const int *layers, const void *const *xs, void *const *ys,
                const int32_t *idx, int T) {
    if (c->S > 255) return 1;
    for (int i = 0; i < n; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        if (L.d_in % 8 || L.d_out % 8 || reinterpret_cast<uintptr_t>(xs[i]) % 16 ||
            reinterpret_cast<uintptr_t>(ys[i]) % 16)
            return 1;
    }
    const int est_tiles = max_decode_tiles(T, c->S);
    FusedArgs fa{};
    fa.n = n;
    for (int i = 0; i < n; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        LayerArgs &a = fa.l[i];
        a.x = xs[i];
        a.y = ys[i];
        a.A = L.A_pool;
        a.B = L.B_pool;
        a.d_in = L.d_in;
        a.d_out = L.d_out;
        a.vec = 1;
        a.chunk_cols = ((L.d_in + kClusterSize - 1) / kClusterSize + 31) / 32 * 32;
        a.out_cols = ((L.d_out + kClusterSize - 1) / kClusterSize + 31) / 32 * 32;
        a.n_chunks = kClusterSize;
    }
    fa.idx = idx;
    fa.T = T;
    fa.S = c->S;
    fa.R = c->R;
    fa.rank = c->rank_dev;
    fa.scale = c->scale_dev;
    fa.hdr = reinterpret_cast<int *>(c->ws + c->lay.hdr);
    fa.early = c->inputs_ready;
    CUDA_TRY(launch_cluster_decode(fa, est_tiles, c->compute, true));
    ++c->launches;
    if (!capturing(c->compute)) CUDA_TRY(note_apply(c));
    return LORA_OK;
}

// Largest batch the cluster decode kernel takes. Unless the caller set it,
// it follows max_lora_rank: the kernel's registers grow with the rank (five
// CTAs per SM at rank 16, three at rank 32, one at rank 64), and measured on
// GB300 (q_proj + v_proj 4096 x 4096) it beats the grouped kernels at every
// batch size up to 1024 tokens at rank 16, up to 768 at rank 32 (slower at
// 1024), and at none at rank 64 (three times slower at 1024 tokens).
int small_batch_limit(const lora_ctx *c) {
    if (c->small_batch >= 0) return c->small_batch;
    return c->R <= 16 ? kFusedMaxTokens : (c->R <= 32 ? 768 : 0);
}

int apply_impl(lora_ctx *c, int n, const int *layers, const void *const *xs, void *const *ys,
               const int32_t *idx, int T) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!c->device) return fail(LORA_ERR_STATE, "host-only context cannot apply");
    if (n < 1 || n > c->max_layers) return fail(LORA_ERR_ARG, "n must be in 1..%d", c->max_layers);
    if (T < 0 || T > c->max_tokens) return fail(LORA_ERR_ARG, "n_tokens %d out of 0..%d", T, c->max_tokens);
    if (!layers || !xs || !ys) return fail(LORA_ERR_ARG, "layers / xs / ys is NULL");
    for (int i = 0; i < n; ++i) {
        if (layers[i] < 0 || layers[i] >= c->n_layers) return fail(LORA_ERR_ARG, "bad layer %d", layers[i]);
        if (T > 0 && (!xs[i] || !ys[i])) return fail(LORA_ERR_ARG, "NULL x or y for entry %d", i);
    }
    if (T == 0) return LORA_OK;
    if (!idx) return fail(LORA_ERR_ARG, "token_slot_idx is NULL");

    // Uploads queued since the last apply must land before any kernel reads a
    // slot: one wait on the newest of them covers the older ones (the upload
    // stream runs in order; a ring event re-recorded since only waits longer).
    if (!capturing(c->compute)) {
        int64_t newest = -1;
        for (int s = 0; s < c->S; ++s) {
            newest = std::max(newest, c->slot_up[s]);
            c->slot_up[s] = -1;
        }
        if (newest >= 0)
            CUDA_TRY(cudaStreamWaitEvent(c->compute, c->up_ev[newest % (int64_t)c->up_ev.size()], 0));
    } else {
        for (int s = 0; s < c->S; ++s)
            if (c->slot_up[s] >= 0)
                return fail(LORA_ERR_STATE, "slot %d upload pending during stream capture; "
                                            "call lora_sync_uploads before capturing", s);
    }

    if (c->dtype == LORA_DTYPE_BF16 && T <= small_batch_limit(c)) {
        int rc = fused_apply(c, n, layers, xs, ys, idx, T);
        if (rc == LORA_OK) ++c->cluster_applies;
        if (rc != 1) return rc;          // 1: shapes not eligible, take the general path
    }
    ++c->grouped_applies;

    // Long same-slot runs go to the tensor-core prefill kernel when every layer allows it.
    bool prefill = c->prefill_min > 0 && c->dtype == LORA_DTYPE_BF16 && prefill_tc_supported(c->R) &&
                   T >= c->prefill_min;
    for (int i = 0; i < n && prefill; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        prefill = L.d_in % 8 == 0 && L.d_out % 64 == 0 && reinterpret_cast<uintptr_t>(xs[i]) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(ys[i]) % 16 == 0;
    }
    CUDA_TRY(launch_group_tokens(idx, T, c->rank_dev, c->S, prefill ? c->prefill_min : 0, c->ws, c->lay,
                                 c->num_sms, c->compute));
    ++c->launches;
    // The decode kernels read only the grouping's lists and write other rows
    // of y and their own partials: they run on the side stream while the
    // prefill kernels run on the compute stream, which waits for both at the
    // end. (Under stream capture the side stream joins the capture through
    // the event and leaves it through the join.)
    CUDA_TRY(cudaEventRecord(c->fork_ev, c->compute));
    CUDA_TRY(cudaStreamWaitEvent(c->side, c->fork_ev, 0));
    if (prefill) {
        // upper bound on prefill tiles: T/128 full tiles plus one ragged tile per run
        int grid_tiles = T / kPrefillRows + T / c->prefill_min + 2;
        if (grid_tiles > c->lay.max_ptiles) grid_tiles = c->lay.max_ptiles;
        PrefillLayer pl[kMaxLayersPerCall];
        for (int i = 0; i < n; ++i) {
            const lora_layer_desc &L = c->layers[layers[i]];
            pl[i].x = xs[i];
            pl[i].y = ys[i];
            pl[i].A = L.A_pool;
            pl[i].B = L.B_pool;
            pl[i].part = reinterpret_cast<float *>(c->ws + c->lay.part) + (size_t)i * c->lay.part_rows * c->R;
            pl[i].d_in = L.d_in;
            pl[i].d_out = L.d_out;
        }
        int queued = 0;
        cudaError_t e = launch_prefill_tc(pl, n, T, c->S, c->R, c->scale_dev, reinterpret_cast<int *>(c->ws + c->lay.hdr),
                                          reinterpret_cast<const int4 *>(c->ws + c->lay.ptiles), grid_tiles,
                                          c->lay.part_rows, c->num_sms, c->compute, &queued);
        c->launches += (uint64_t)queued;
        if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    }

    const size_t e = elem_bytes(c->dtype);
    const int est_tiles = max_decode_tiles(T, c->S);
    MultiArgs ma{};
    ma.n = n;
    int max_chunks = 1, max_dblocks = 1;
    for (int i = 0; i < n; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        LayerArgs &a = ma.l[i];
        a.x = xs[i];
        a.y = ys[i];
        a.A = L.A_pool;
        a.B = L.B_pool;
        a.d_in = L.d_in;
        a.d_out = L.d_out;
        a.v = reinterpret_cast<float *>(c->ws + c->lay.v) + (size_t)i * c->lay.max_tokens * v_stride(c->R);
        a.part = reinterpret_cast<float *>(c->ws + c->lay.dpart) + (size_t)i * c->lay.part_rows * c->R;
        a.counters = reinterpret_cast<int *>(c->ws + c->lay.counters) + (size_t)i * c->lay.max_tiles;
        // Split d_in into chunks of ~256 columns so that a tile's shrink is
        // spread over many CTAs (the host cannot tell how many decode tiles a
        // batch has), as long as a tile's fp32 partials (written and read,
        // 16 tokens x R) stay under 1/8 of the x and A bytes the tile reads.
        int chunks = (L.d_in + 255) / 256;
        const int by_bytes = (int)((size_t)(kTileTokens + c->R) * L.d_in * e / (8 * 2 * kTileTokens * 4 * (size_t)c->R));
        if (chunks > by_bytes) chunks = by_bytes;
        if (chunks > kMaxChunks) chunks = kMaxChunks;
        // a layer's partials hold part_rows rows of R floats; the decode
        // kernels' partial rows are v_stride(R) floats
        const long long max_split = (long long)c->lay.part_rows * c->R / ((long long)T * v_stride(c->R));
        if (chunks > max_split) chunks = (int)max_split;
        if (chunks < 1) chunks = 1;
        int cols = (L.d_in + chunks - 1) / chunks;
        cols = (cols + 127) / 128 * 128;
        a.chunk_cols = cols;
        a.n_chunks = (L.d_in + cols - 1) / cols;
        const bool al = (reinterpret_cast<uintptr_t>(xs[i]) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(ys[i]) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(L.A_pool) % 16 == 0) &&
                        ((size_t)L.d_in * e % 16 == 0) && ((size_t)L.d_out * e % 16 == 0);
        a.vec = al ? 1 : 0;
        if (a.n_chunks > max_chunks) max_chunks = a.n_chunks;
        int db = (L.d_out + 255) / 256;
        if (db > max_dblocks) max_dblocks = db;
    }
    GroupView gv{};
    gv.hdr = reinterpret_cast<const int *>(c->ws + c->lay.hdr);
    gv.perm = reinterpret_cast<const int *>(c->ws + c->lay.perm);
    gv.tiles = reinterpret_cast<const int4 *>(c->ws + c->lay.tiles);
    gv.scale = c->scale_dev;
    gv.rank = c->rank_dev;
    gv.R = c->R;
    gv.T = T;
    int grid_tiles = est_tiles < c->lay.max_tiles ? est_tiles : c->lay.max_tiles;
    CUDA_TRY(launch_decode(ma, gv, c->dtype, grid_tiles, max_chunks, max_dblocks, c->num_sms, c->side));
    if (grid_tiles > 0) c->launches += 2;          // shrink and expand
    CUDA_TRY(cudaEventRecord(c->join_ev, c->side));
    CUDA_TRY(cudaStreamWaitEvent(c->compute, c->join_ev, 0));
    if (!capturing(c->compute)) CUDA_TRY(note_apply(c));
    return LORA_OK;
}

}  // namespace

int lora_apply(lora_ctx *c, int layer, const void *x, void *y, const int32_t *idx, int n_tokens) {
    const void *xs[1] = {x};
    void *ys[1] = {y};
    return apply_impl(c, 1, &layer, xs, ys, idx, n_tokens);
}

int lora_apply_multi(lora_ctx *c, int n, const int *layers, const void *const *xs, void *const *ys,
                     const int32_t *idx, int n_tokens) {
    return apply_impl(c, n, layers, xs, ys, idx, n_tokens);
}

int lora_apply_multi_host(lora_ctx *c, int n, const int *layers, const void *const *xs_host,
                          void *const *ys_host, const int32_t *idx_host, int T,
                          void *const *xs_dev, void *const *ys_dev, int32_t *idx_dev) {
    if (!c || !c->device) return fail(LORA_ERR_STATE, "needs a device context");
    if (n < 1 || n > c->max_layers || !layers || !xs_host || !ys_host || !xs_dev || !ys_dev)
        return fail(LORA_ERR_ARG, "bad arguments");
    if (T < 0 || T > c->max_tokens) return fail(LORA_ERR_ARG, "n_tokens out of range");
    if (T == 0) return LORA_OK;
    if (!idx_host || !idx_dev) return fail(LORA_ERR_ARG, "token_slot_idx is NULL");
    for (int i = 0; i < n; ++i)
        if (layers[i] < 0 || layers[i] >= c->n_layers) return fail(LORA_ERR_ARG, "bad layer");
    const size_t e = elem_bytes(c->dtype);
    // Device staging buffers of this call (the distinct ones).
    std::vector<const void *> bufs{idx_dev};
    for (int i = 0; i < n; ++i) {
        bufs.push_back(xs_dev[i]);
        bufs.push_back(ys_dev[i]);
    }
    std::sort(bufs.begin(), bufs.end());
    bufs.erase(std::unique(bufs.begin(), bufs.end()), bufs.end());
    // Copies in, then copies back; a copy that continues the previous one in
    // both host and device memory joins it (a caller that packs its staging
    // buffers back to back gets one copy each way).
    std::vector<Copy> in_copies{{idx_dev, idx_host, sizeof(int32_t) * (size_t)T}};
    for (int i = 0; i < n; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        bool dup = false;                          // layers sharing one input copy it once
        for (int j = 0; j < i; ++j) dup = dup || (xs_host[j] == xs_host[i] && xs_dev[j] == xs_dev[i]);
        if (!dup) in_copies.push_back({xs_dev[i], xs_host[i], (size_t)T * L.d_in * e});
        in_copies.push_back({ys_dev[i], ys_host[i], (size_t)T * L.d_out * e});
    }
    std::vector<Copy> out_copies;
    for (int i = 0; i < n; ++i) {
        const lora_layer_desc &L = c->layers[layers[i]];
        out_copies.push_back({ys_host[i], ys_dev[i], (size_t)T * L.d_out * e});
    }
    in_copies = merge_copies(in_copies);
    out_copies = merge_copies(out_copies);
    // Copies in run on the upload stream, after the copies back of the last
    // call that used any of this call's device buffers; the apply on the
    // compute stream; the copies back on the context's own download stream.
    // A caller rotating two or more buffer sets thus keeps both directions of
    // the host link and the GPU busy at once. Under stream capture everything
    // stays on the compute stream.
    const bool split = !capturing(c->compute);
    if (split && !c->h2d_done) CUDA_TRY(cudaEventCreateWithFlags(&c->h2d_done, cudaEventDisableTiming));
    if (split && !c->apply_done) CUDA_TRY(cudaEventCreateWithFlags(&c->apply_done, cudaEventDisableTiming));
    if (split && !c->down) CUDA_TRY(cudaStreamCreateWithFlags(&c->down, cudaStreamNonBlocking));
    if (split && c->host_ev.empty()) {
        c->host_ev.assign(kHostRing, nullptr);
        for (auto &ev : c->host_ev) CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    cudaStream_t in = split ? c->upload : c->compute;
    if (split) {
        // Newest earlier use of any of these buffers. A ring event re-recorded
        // by a later call only lengthens the wait: every call records on the
        // download stream, in call order.
        int64_t last = -1;
        for (const void *b : bufs) {
            bool found = false;
            for (auto &bu : c->buf_use)
                if (bu.first == b) {
                    last = std::max(last, bu.second);
                    found = true;
                }
            if (!found) last = std::max(last, c->host_forgot);   // maybe a forgotten buffer
        }
        if (last >= 0) CUDA_TRY(cudaStreamWaitEvent(c->upload, c->host_ev[last % kHostRing], 0));
    }
    for (const Copy &cp : in_copies)
        CUDA_TRY(cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyHostToDevice, in));
    if (split) {
        CUDA_TRY(cudaEventRecord(c->h2d_done, c->upload));
        CUDA_TRY(cudaStreamWaitEvent(c->compute, c->h2d_done, 0));
    }
    int rc = apply_impl(c, n, layers, xs_dev, ys_dev, idx_dev, T);
    if (rc != LORA_OK) return rc;
    cudaStream_t out = split ? c->down : c->compute;
    if (split) {
        CUDA_TRY(cudaEventRecord(c->apply_done, c->compute));
        CUDA_TRY(cudaStreamWaitEvent(c->down, c->apply_done, 0));
    }
    for (const Copy &cp : out_copies)
        CUDA_TRY(cudaMemcpyAsync(cp.dst, cp.src, cp.bytes, cudaMemcpyDeviceToHost, out));
    if (split) {
        const int64_t k = c->n_host++;
        CUDA_TRY(cudaEventRecord(c->host_ev[k % kHostRing], c->down));
        for (const void *b : bufs) {
            bool found = false;
            for (auto &bu : c->buf_use)
                if (bu.first == b) {
                    bu.second = k;
                    found = true;
                }
            if (!found) c->buf_use.emplace_back(b, k);
        }
        // Keep the list short: forget buffers not used for a whole ring and
        // remember the newest call forgotten; a buffer not on the list then
        // waits for that call (or a later one), which covers its last use.
        if (c->buf_use.size() > 64) {
            for (auto &bu : c->buf_use)
                if (bu.second + kHostRing <= k) c->host_forgot = std::max(c->host_forgot, bu.second);
            c->buf_use.erase(std::remove_if(c->buf_use.begin(), c->buf_use.end(),
                                            [&](const std::pair<const void *, int64_t> &bu) {
                                                return bu.second + kHostRing <= k;
                                            }),
                             c->buf_use.end());
        }
    }
    return LORA_OK;
}

int lora_lookup(lora_ctx *c, uint64_t id, int *slot) {
    if (!c || !slot) return fail(LORA_ERR_ARG, "NULL argument");
    *slot = c->table.lookup(id);
    return LORA_OK;
}

int lora_assign(lora_ctx *c, uint64_t id, int rank, int *slot, int *needs_load, uint64_t *evicted_id) {
    if (!c || !slot || !needs_load || !evicted_id) return fail(LORA_ERR_ARG, "NULL argument");
    *needs_load = 0;
    switch (c->table.assign(id, rank, slot, evicted_id)) {
    case AssignResult::Hit:
        return LORA_OK;
    case AssignResult::Loaded:
        *needs_load = 1;
        return LORA_OK;
    case AssignResult::BadRank:
        return fail(LORA_ERR_RANK, "LoRA rank %d exceeds maximum %d (or is < 1)", rank, c->R);
    case AssignResult::NoSlot:
    default:
        return fail(LORA_ERR_NO_SLOT, "no occupied slot may be evicted (in flight, pinned or cooling)");
    }
}

int lora_assign_batch(lora_ctx *c, int n, const uint64_t *ids, const int *ranks, int acquire, int *slots,
                      int *needs_load, uint64_t *evicted_ids, int *n_done) {
    if (!c || n_done == nullptr) return fail(LORA_ERR_ARG, "NULL argument");
    *n_done = 0;
    if (n < 0) return fail(LORA_ERR_ARG, "n must be >= 0");
    if (n > 0 && (!ids || !ranks || !slots || !needs_load || !evicted_ids))
        return fail(LORA_ERR_ARG, "NULL argument");
    for (int i = 0; i < n; ++i) {
        int rc = lora_assign(c, ids[i], ranks[i], &slots[i], &needs_load[i], &evicted_ids[i]);
        if (rc != LORA_OK) return rc;
        if (acquire) c->table.acquire(slots[i]);
        *n_done = i + 1;
    }
    return LORA_OK;
}

int lora_assign_tokens(lora_ctx *c, int T, const uint64_t *adapter_ids, const int *ranks, int acquire,
                       int32_t *token_slot_idx, int max_distinct, uint64_t *distinct_ids, int *slots,
                       int *needs_load, uint64_t *evicted_ids, int *n_distinct, int *n_done) {
    if (!c || !n_distinct || !n_done) return fail(LORA_ERR_ARG, "NULL argument");
    *n_distinct = 0;
    *n_done = 0;
    if (T < 0 || max_distinct < 0) return fail(LORA_ERR_ARG, "negative size");
    if (T == 0) return LORA_OK;
    if (!adapter_ids || !ranks || !token_slot_idx ||
        (max_distinct > 0 && (!distinct_ids || !slots || !needs_load || !evicted_ids)))
        return fail(LORA_ERR_ARG, "NULL argument");
    // Distinct adapters in order of first appearance (open addressing on the
    // id); until the slots are known token_slot_idx holds each token's index
    // among them.
    size_t cap = 16;
    while (cap < 2 * (size_t)T) cap <<= 1;
    if (c->tok_key.size() < cap) {
        c->tok_key.resize(cap);
        c->tok_val.resize(cap);
    }
    std::fill(c->tok_key.begin(), c->tok_key.begin() + cap, LORA_NO_ADAPTER);
    const size_t mask = cap - 1;
    std::vector<int> &first_rank = c->tok_rank;
    first_rank.clear();
    for (int t = 0; t < T; ++t) {
        const uint64_t id = adapter_ids[t];
        if (id == LORA_NO_ADAPTER) {
            token_slot_idx[t] = -1;
            continue;
        }
        size_t h = (size_t)((id * 0x9E3779B97F4A7C15ull) >> 17) & mask;
        while (c->tok_key[h] != LORA_NO_ADAPTER && c->tok_key[h] != id) h = (h + 1) & mask;
        if (c->tok_key[h] == LORA_NO_ADAPTER) {
            const int nd = (int)first_rank.size();
            if (nd == max_distinct) {        // nothing admitted: the table is unchanged
                for (int u = 0; u < T; ++u) token_slot_idx[u] = -1;
                return fail(LORA_ERR_ARG, "more than max_distinct (%d) adapters in the batch", max_distinct);
            }
            c->tok_key[h] = id;
            c->tok_val[h] = nd;
            distinct_ids[nd] = id;
            first_rank.push_back(ranks[t]);
        }
        token_slot_idx[t] = c->tok_val[h];
    }
    const int nd = (int)first_rank.size();
    *n_distinct = nd;
    for (int i = 0; i < nd; ++i) {
        slots[i] = -1;
        needs_load[i] = 0;
        evicted_ids[i] = LORA_NO_ADAPTER;
    }
    int rc = LORA_OK;
    for (int i = 0; i < nd; ++i) {           // lora_assign_batch over the distinct list
        rc = lora_assign(c, distinct_ids[i], first_rank[i], &slots[i], &needs_load[i], &evicted_ids[i]);
        if (rc != LORA_OK) break;
        if (acquire) c->table.acquire(slots[i]);
        *n_done = i + 1;
    }
    for (int t = 0; t < T; ++t) {
        const int i = token_slot_idx[t];
        if (i >= 0) token_slot_idx[t] = i < *n_done ? slots[i] : -1;
    }
    return rc;
}

int lora_register_host_adapters(lora_ctx *c, int n, const uint64_t *ids, const int *ranks,
                                const float *alphas, const void *const *A_host, const void *const *B_host) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (n < 0) return fail(LORA_ERR_ARG, "n must be >= 0");
    const int L = c->n_layers;
    if (n > 0 && (!ids || !ranks || !alphas || (L > 0 && (!A_host || !B_host))))
        return fail(LORA_ERR_ARG, "NULL argument");
    std::unordered_map<uint64_t, int> m;
    m.reserve((size_t)n * 2);
    for (int i = 0; i < n; ++i) {
        if (ids[i] == LORA_NO_ADAPTER) return fail(LORA_ERR_ARG, "adapter %d has the no-adapter id", i);
        if (!m.emplace(ids[i], i).second) return fail(LORA_ERR_ARG, "adapter id of entry %d appears twice", i);
        if (ranks[i] < 1 || ranks[i] > c->R)
            return fail(LORA_ERR_RANK, "LoRA rank %d exceeds maximum %d (or is < 1)", ranks[i], c->R);
        if (!std::isfinite(alphas[i])) return fail(LORA_ERR_ARG, "alpha %d is not finite", i);
        for (int l = 0; l < L; ++l)
            if (!A_host[(size_t)i * L + l] || !B_host[(size_t)i * L + l])
                return fail(LORA_ERR_ARG, "adapter %d layer %d weights are NULL", i, l);
    }
    c->store.swap(m);
    c->store_rank.assign(ranks, ranks + n);
    c->store_alpha.assign(alphas, alphas + n);
    c->store_A.assign(A_host, A_host + (size_t)n * L);
    c->store_B.assign(B_host, B_host + (size_t)n * L);
    return LORA_OK;
}

int lora_set_warm_set(lora_ctx *c, int n, const uint64_t *ids) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (n < 0 || (n > 0 && !ids)) return fail(LORA_ERR_ARG, "bad arguments");
    c->warm.clear();
    c->warm.insert(ids, ids + n);
    return LORA_OK;
}

int lora_serve_step(lora_ctx *c, int T, const uint64_t *adapter_ids, int n, const int *layers,
                    const void *const *xs, void *const *ys, int32_t *idx_bufs, int max_groups, int max_distinct,
                    uint64_t *out_ids, int *out_slots, int *out_needs_load, uint64_t *out_evicted,
                    int *n_distinct, int *n_groups) {
    if (!c || !n_distinct || !n_groups) return fail(LORA_ERR_ARG, "NULL argument");
    *n_distinct = 0;
    *n_groups = 0;
    if (T < 0 || max_groups < 0 || max_distinct < 0) return fail(LORA_ERR_ARG, "negative size");
    if (T > 0 && !adapter_ids) return fail(LORA_ERR_ARG, "adapter_ids is NULL");
    if (max_distinct > 0 && (!out_ids || !out_slots || !out_needs_load || !out_evicted))
        return fail(LORA_ERR_ARG, "NULL output array");
    if (c->device && T > 0) {
        if (T > c->max_tokens) return fail(LORA_ERR_ARG, "n_tokens %d above max_tokens %d", T, c->max_tokens);
        if (n < 1 || n > c->max_layers || !layers || !xs || !ys || !idx_bufs)
            return fail(LORA_ERR_ARG, "layers, xs, ys and idx_bufs are required (n in 1..%d)", c->max_layers);
        for (int i = 0; i < n; ++i)
            if (layers[i] < 0 || layers[i] >= c->n_layers || !xs[i] || !ys[i])
                return fail(LORA_ERR_ARG, "bad layer entry %d", i);
    }
    // Distinct adapters in order of first appearance; each token's index among them.
    size_t cap = 16;
    while (cap < 2 * (size_t)T) cap <<= 1;
    if (c->tok_key.size() < cap) {
        c->tok_key.resize(cap);
        c->tok_val.resize(cap);
    }
    std::fill(c->tok_key.begin(), c->tok_key.begin() + cap, LORA_NO_ADAPTER);
    const size_t mask = cap - 1;
    std::vector<uint64_t> &dist = c->step_id;
    std::vector<int> &tok = c->step_tok;
    dist.clear();
    tok.resize((size_t)T);
    for (int t = 0; t < T; ++t) {
        const uint64_t id = adapter_ids[t];
        if (id == LORA_NO_ADAPTER) {
            tok[t] = -1;
            continue;
        }
        size_t h = (size_t)((id * 0x9E3779B97F4A7C15ull) >> 17) & mask;
        while (c->tok_key[h] != LORA_NO_ADAPTER && c->tok_key[h] != id) h = (h + 1) & mask;
        if (c->tok_key[h] == LORA_NO_ADAPTER) {
            if (!c->store.count(id)) return fail(LORA_ERR_ARG, "adapter id %llu is not registered",
                                                 (unsigned long long)id);
            c->tok_key[h] = id;
            c->tok_val[h] = (int)dist.size();
            dist.push_back(id);
        }
        tok[t] = c->tok_val[h];
    }
    const int nd = (int)dist.size();
    if (max_distinct > 0 && nd > max_distinct)
        return fail(LORA_ERR_ARG, "more than max_distinct (%d) adapters in the batch", max_distinct);
    // Groups: at most max_loras minus the pinned slots need a slot each; an
    // adapter resident in a pinned slot needs none. A warm-set adapter not in
    // a pinned slot pins its slot when its group is admitted, so every later
    // group has one evictable slot fewer.
    int pinned = 0;
    for (int s = 0; s < c->S; ++s) pinned += c->table.pinned(s) ? 1 : 0;
    int capacity = c->S - pinned;
    std::vector<int> &grp = c->step_group;
    grp.resize((size_t)nd);
    int ng = 0, cost = 0, in_cur = 0, new_pins = 0;
    for (int i = 0; i < nd; ++i) {
        const int s = c->table.find(dist[i]);
        const int k = (s >= 0 && c->table.pinned(s)) ? 0 : 1;
        if (in_cur > 0 && cost + k > capacity) {
            ++ng;
            cost = 0;
            in_cur = 0;
            capacity -= new_pins;
            new_pins = 0;
        }
        grp[i] = ng;
        cost += k;
        ++in_cur;
        if (k && c->warm.count(dist[i])) ++new_pins;
    }
    if (nd > 0) ++ng;
    if (c->device && ng > max_groups)
        return fail(LORA_ERR_ARG, "the batch needs %d adapter groups, idx_bufs holds %d", ng, max_groups);
    std::vector<int> &slot = c->step_slot, &need = c->step_need;
    std::vector<uint64_t> &ev = c->step_ev;
    slot.assign((size_t)nd, -1);
    need.assign((size_t)nd, 0);
    ev.assign((size_t)nd, LORA_NO_ADAPTER);
    const int L = c->n_layers;
    std::vector<int> &up_slots = c->up_slots, &up_ranks = c->up_ranks;
    std::vector<float> &up_alphas = c->up_alphas;
    std::vector<const void *> &up_A = c->up_A, &up_B = c->up_B;
    // The misses collected so far go up in one batched upload.
    auto flush_uploads = [&]() {
        int rc = LORA_OK;
        if (!up_slots.empty()) {
            if (c->device) {
                rc = lora_load_slots(c, (int)up_slots.size(), up_slots.data(), up_A.data(), up_B.data(),
                                     up_ranks.data(), up_alphas.data());
            } else {
                for (int s : up_slots) c->table.mark_loaded(s);
                c->uploads += up_slots.size();
            }
        }
        up_slots.clear();
        up_ranks.clear();
        up_alphas.clear();
        up_A.clear();
        up_B.clear();
        return rc;
    };
    int i0 = 0;
    for (int g = 0; g < ng; ++g) {
        int i1 = i0;
        while (i1 < nd && grp[i1] == g) ++i1;
        // admission of the group's adapters, in order: hit (touch) or bind, and
        // an in-flight reference on each. (Measured: sending the first 16
        // misses up while the host admits the rest made the step slower; two
        // upload kernels move the same bytes more slowly than one.)
        for (int i = i0; i < i1; ++i) {
            const int si = c->store.at(dist[i]);
            int rc = lora_assign(c, dist[i], c->store_rank[si], &slot[i], &need[i], &ev[i]);
            if (rc != LORA_OK) {
                for (int q = i0; q < i; ++q) c->table.release(slot[q]);
                flush_uploads();            // the misses bound so far still get their weights
                return rc;
            }
            c->table.acquire(slot[i]);
            if (c->warm.count(dist[i]) && !c->table.pinned(slot[i])) c->table.pin(slot[i], true);
            if (need[i]) {
                up_slots.push_back(slot[i]);
                up_ranks.push_back(c->store_rank[si]);
                up_alphas.push_back(c->store_alpha[si]);
                for (int l = 0; l < L; ++l) {
                    up_A.push_back(c->store_A[(size_t)si * L + l]);
                    up_B.push_back(c->store_B[(size_t)si * L + l]);
                }
            }
        }
        int rc = flush_uploads();
        if (rc == LORA_OK && c->device && T > 0) {
            int32_t *idx = idx_bufs + (size_t)g * T;
            for (int t = 0; t < T; ++t) {
                const int i = tok[t];
                idx[t] = (i >= i0 && i < i1) ? slot[i] : -1;
            }
            rc = apply_impl(c, n, layers, xs, ys, idx, T);
        }
        for (int i = i0; i < i1; ++i) c->table.release(slot[i]);
        if (rc != LORA_OK) return rc;
        i0 = i1;
    }
    c->table.tick();
    for (int i = 0; i < nd && i < max_distinct; ++i) {
        out_ids[i] = dist[i];
        out_slots[i] = slot[i];
        out_needs_load[i] = need[i];
        out_evicted[i] = ev[i];
    }
    *n_distinct = nd;
    *n_groups = ng;
    return LORA_OK;
}

int lora_release_batch(lora_ctx *c, int n, const int *slots) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (n < 0 || (n > 0 && !slots)) return fail(LORA_ERR_ARG, "bad arguments");
    for (int i = 0; i < n; ++i)
        if (!c->table.release(slots[i])) return fail(LORA_ERR_STATE, "slot %d is not in flight", slots[i]);
    return LORA_OK;
}

int lora_acquire(lora_ctx *c, int slot) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    return c->table.acquire(slot) ? LORA_OK : fail(LORA_ERR_STATE, "slot %d is not occupied", slot);
}

int lora_release(lora_ctx *c, int slot) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    return c->table.release(slot) ? LORA_OK : fail(LORA_ERR_STATE, "slot %d is not in flight", slot);
}

int lora_set_slot_tracking(lora_ctx *c, int on) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!c->device) return fail(LORA_ERR_STATE, "host-only context has no uploads");
    if (on && c->ring.empty()) {
        c->ring.assign(kRing, nullptr);
        for (auto &ev : c->ring) CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    if (on && !c->track) {
        // Everything queued so far may read any slot: start from the stream-wide event.
        CUDA_TRY(cudaEventRecord(c->ring[c->n_apply % kRing], c->compute));
        c->slot_gen.assign(c->S, c->n_apply);
        ++c->n_apply;
    }
    c->track = on ? 1 : 0;
    return LORA_OK;
}

int lora_pin(lora_ctx *c, int slot, int pinned) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (slot < 0 || slot >= c->S) return fail(LORA_ERR_ARG, "slot %d out of range", slot);
    return c->table.pin(slot, pinned != 0) ? LORA_OK : fail(LORA_ERR_STATE, "slot %d is empty", slot);
}

int lora_set_min_residency(lora_ctx *c, int epochs) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (epochs < 0) return fail(LORA_ERR_ARG, "epochs must be >= 0");
    c->table.set_min_residency(epochs);
    return LORA_OK;
}

int lora_set_policy(lora_ctx *c, int policy) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (policy != LORA_POLICY_LRU && policy != LORA_POLICY_KEEP_SCORE)
        return fail(LORA_ERR_ARG, "unknown policy %d", policy);
    c->table.set_policy(policy == LORA_POLICY_LRU ? EvictPolicy::Lru : EvictPolicy::KeepScore);
    return LORA_OK;
}

int lora_set_keep_score_weights(lora_ctx *c, const double *w) {
    if (!c || !w) return fail(LORA_ERR_ARG, "NULL argument");
    for (int i = 0; i < 5; ++i)
        if (!std::isfinite(w[i])) return fail(LORA_ERR_ARG, "weight %d is not finite", i);
    c->table.set_weights(w);
    return LORA_OK;
}

int lora_set_adapter_priority(lora_ctx *c, uint64_t adapter_id, double priority) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!std::isfinite(priority)) return fail(LORA_ERR_ARG, "priority is not finite");
    c->table.set_priority(adapter_id, priority);
    return LORA_OK;
}

}  // extern "C"

namespace {

// A slot emptied in the host table reads as empty (rank 0) for device work
// queued after the call; compute already queued that may read it finishes first.
int mark_slot_empty_on_device(lora_ctx *c, int slot) {
    if (!c->device) return LORA_OK;
    CUDA_TRY(wait_slot_reads(c, slot));
    CUDA_TRY(launch_set_slot(c->scale_dev, c->rank_dev, slot, 0.f, 0, c->upload));
    ++c->launches;
    CUDA_TRY(note_upload(c, &slot, 1));
    return LORA_OK;
}

}  // namespace

extern "C" {

int lora_evict_lru(lora_ctx *c, int *evicted_slot, uint64_t *evicted_id) {
    if (!c || !evicted_slot || !evicted_id) return fail(LORA_ERR_ARG, "NULL argument");
    if (!c->table.evict_lru(evicted_slot, evicted_id))
        return fail(LORA_ERR_NO_SLOT, "no occupied slot may be evicted (in flight, pinned or cooling)");
    return *evicted_slot >= 0 ? mark_slot_empty_on_device(c, *evicted_slot) : LORA_OK;
}

int lora_abort_load(lora_ctx *c, int slot, uint64_t *unbound_id) {
    if (!c || !unbound_id) return fail(LORA_ERR_ARG, "NULL argument");
    if (slot < 0 || slot >= c->S) return fail(LORA_ERR_ARG, "slot %d out of range", slot);
    if (!c->table.abort_load(slot, unbound_id))
        return fail(LORA_ERR_STATE, "slot %d is empty or its upload was already queued", slot);
    return mark_slot_empty_on_device(c, slot);
}

int lora_tick(lora_ctx *c) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    c->table.tick();
    return LORA_OK;
}

int lora_set_thrash_window(lora_ctx *c, int epochs) {
    if (!c || epochs < 0) return fail(LORA_ERR_ARG, "bad arguments");
    c->table.set_window(epochs);
    return LORA_OK;
}

int lora_set_prefill_min_tokens(lora_ctx *c, int n) {
    if (!c || n < 0) return fail(LORA_ERR_ARG, "bad arguments");
    c->prefill_min = n == 0 ? 0 : (n < kMinPrefillRun ? kMinPrefillRun : n);
    return LORA_OK;
}

int lora_set_small_batch_tokens(lora_ctx *c, int n) {
    if (!c || n < -1 || n > kFusedMaxTokens)
        return fail(LORA_ERR_ARG, "n must be -1 (by rank) or in 0..%d", kFusedMaxTokens);
    c->small_batch = n;
    return LORA_OK;
}

int lora_set_inputs_ready(lora_ctx *c, int on) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    c->inputs_ready = on ? 1 : 0;
    return LORA_OK;
}

int lora_sync_host(lora_ctx *c) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!c->device) return LORA_OK;
    CUDA_TRY(cudaStreamSynchronize(c->down ? c->down : c->compute));
    return LORA_OK;
}

int lora_sync_uploads(lora_ctx *c) {
    if (!c) return fail(LORA_ERR_ARG, "ctx is NULL");
    if (!c->device) return LORA_OK;
    CUDA_TRY(cudaStreamSynchronize(c->upload));
    return harvest_timings(c, true);
}

int lora_selftest_wait_timeout(lora_ctx *c, int *gave_up) {
    if (!c || !gave_up) return fail(LORA_ERR_ARG, "NULL argument");
    if (!c->device) return fail(LORA_ERR_STATE, "host-only context has no device");
    *gave_up = 0;
    int *hdr = reinterpret_cast<int *>(c->ws + c->lay.hdr);
    CUDA_TRY(cudaMemsetAsync(hdr + kHdrSelftest, 0, sizeof(int), c->compute));
    CUDA_TRY(launch_selftest_wait(hdr + kHdrError, 1u << 14, c->compute));
    CUDA_TRY(launch_selftest_cluster_wait(hdr + kHdrError, hdr + kHdrSelftest, 1u << 14, c->compute));
    c->launches += 2;
    CUDA_TRY(cudaStreamSynchronize(c->compute));
    int v[2] = {0, 0};
    CUDA_TRY(cudaMemcpy(&v[0], hdr + kHdrError, sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(&v[1], hdr + kHdrSelftest, sizeof(int), cudaMemcpyDeviceToHost));
    *gave_up = v[0] != 0 && v[1] == 2;
    return LORA_OK;
}

int lora_stats(lora_ctx *c, lora_stats_t *o) {
    if (!c || !o) return fail(LORA_ERR_ARG, "NULL argument");
    memset(o, 0, sizeof *o);
    if (c->device) {
        CUDA_TRY(cudaStreamSynchronize(c->compute));
        int hdr[8] = {0};
        CUDA_TRY(cudaMemcpy(hdr, c->ws + c->lay.hdr, sizeof hdr, cudaMemcpyDeviceToHost));
        c->invalid_seen = (uint64_t)hdr[kHdrInvalid];
        o->device_wait_timeouts = (uint64_t)hdr[kHdrError];
        int rc = harvest_timings(c, false);
        if (rc != LORA_OK) return rc;
    }
    o->cluster_applies = c->cluster_applies;
    o->grouped_applies = c->grouped_applies;
    o->kernel_launches = c->launches;
    o->aborted_loads = c->table.aborted_loads;
    o->hits = c->table.hits;
    o->misses = c->table.misses;
    o->evictions = c->table.evictions;
    o->reloads_after_eviction = c->table.reloads;
    o->rejected = c->table.rejected;
    o->uploads = c->uploads;
    o->upload_bytes = c->upload_bytes;
    o->invalid_token_index = c->invalid_seen;
    o->upload_seconds = c->upload_seconds;
    o->epoch = c->table.epoch();
    return LORA_OK;
}

}  // extern "C"
