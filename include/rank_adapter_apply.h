/*
 * rank_adapter_apply -- multi-LoRA delta and GPU adapter slot table, GB300.
 *
 * For every token t of a batch and every injected linear layer l:
 *
 *     y_l[t] += (lora_alpha_s / r_s) * B_{l,s} * (A_{l,s} * x_l[t]),
 *     s = token_slot_idx[t];  s == -1 means base model only (y untouched).
 *
 * r_s and lora_alpha_s are the adapter's "r" and "lora_alpha" (the PEFT
 * adapter_config.json example on the "vLLM LoRA Resolver 插件详解" page, section
 * 3.2, with use_rslora and use_dora false). The slot table follows the
 * "Multi-LoRA 适配器缓存生产实战" page: max_loras GPU slots, ranks padded to
 * max_lora_rank (section 核心原理, parameter table); CPU-resident adapters are
 * uploaded host-to-device on a miss (section 冷加载延迟, tier L1); eviction is
 * LRU with touch on hit and never removes an adapter in use (section 核心原理,
 * last paragraph; section 数据面).
 *
 * Conventions for every call:
 *  - All functions return LORA_OK (0) or a negative lora_status; none throws,
 *    aborts or exits. lora_last_error() gives a message for the calling thread.
 *  - Device memory (slot pools, scale/rank arrays, workspace, activations) is
 *    allocated and owned by the caller. The library owns host bookkeeping and
 *    CUDA events only.
 *  - Streams are passed as cudaStream_t cast to void*. Kernels run on the
 *    compute stream; slot uploads on the upload stream. No call synchronises
 *    the host except lora_sync_uploads, lora_sync_host and lora_stats.
 *  - Layouts are row-major. A pool of layer l: [max_loras][max_lora_rank][d_in].
 *    B pool: [max_loras][max_lora_rank / kb][d_out][kb] with kb = 32 when
 *    max_lora_rank is a multiple of 32, else 16 when it is a multiple of 16,
 *    else 8 (so [max_loras][d_out][max_lora_rank] up to rank 32): slot s's
 *    B_s (d_out x rank)
 *    in blocks of kb consecutive ranks, element (i, k) of slot s at
 *    s * d_out * max_lora_rank + (k / kb) * d_out * kb + i * kb + k % kb, so a
 *    slot of rank r occupies ceil(r / kb) contiguous runs of d_out * kb
 *    elements and kernels read no padding past them. Ranks at or past r are
 *    zero in both pools. Element type = the context's dtype. Activations x:
 *    [n_tokens][d_in]; outputs y: [n_tokens][d_out]. The upload calls write
 *    this layout from host adapters in the PEFT layout (A [r][d_in], B
 *    [d_out][r]).
 *  - A context is not thread-safe: one host thread at a time.
 */
#ifndef RANK_ADAPTER_APPLY_H
#define RANK_ADAPTER_APPLY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_ctx lora_ctx;

/* Adapter id meaning "base model only" in lora_assign_tokens (never bound). */
#define LORA_NO_ADAPTER UINT64_MAX

enum lora_status {
    LORA_OK = 0,
    LORA_ERR_ARG = -1,      /* bad pointer, size, index or layout */
    LORA_ERR_RANK = -2,     /* r > max_lora_rank ("LoRA rank exceeds maximum",
                               "vLLM LoRA Resolver 插件详解" page, section 6.1 item 4) */
    LORA_ERR_NO_SLOT = -3,  /* no occupied slot may be evicted (in flight, pinned or cooling) */
    LORA_ERR_CUDA = -4,     /* a CUDA runtime call failed (message has the detail) */
    LORA_ERR_STATE = -5,    /* call not valid in the current state */
};

enum lora_dtype {
    LORA_DTYPE_F32 = 0,     /* fp32 activations, weights and fp32 arithmetic */
    LORA_DTYPE_BF16 = 1,    /* bf16 storage, fp32 accumulation, one final rounding */
};

/* One injected linear layer: its shapes and its caller-owned device slot pools. */
typedef struct {
    int d_in;
    int d_out;
    void *A_pool;           /* device, [max_loras][max_lora_rank][d_in] */
    void *B_pool;           /* device, max_loras x d_out x max_lora_rank elements, blocked by rank (see above) */
} lora_layer_desc;

typedef struct {
    uint64_t hits;                  /* lookups/assigns that found the adapter resident */
    uint64_t misses;                /* assigns that bound a new adapter to a slot */
    uint64_t evictions;             /* adapters removed from a slot */
    uint64_t reloads_after_eviction;/* misses within thrash_window epochs of that adapter's eviction */
    uint64_t rejected;              /* assigns refused before any eviction (bad rank) */
    uint64_t uploads;               /* adapters uploaded (lora_load_slot, lora_load_slots) */
    uint64_t upload_bytes;          /* sum of (d_in + d_out) * r * bytes_per_param per upload */
    uint64_t invalid_token_index;   /* tokens with index < -1 or >= max_loras (skipped) */
    double upload_seconds;          /* device time of completed uploads */
    int64_t epoch;                  /* current epoch (lora_tick) */
    uint64_t device_wait_timeouts;  /* non-zero: a bounded device-side wait gave up and the
                                       rows it guarded were left unchanged (never expected) */
    uint64_t cluster_applies;       /* applies served by the single-launch cluster decode kernel */
    uint64_t grouped_applies;       /* applies served by grouping + prefill / decode kernels */
    uint64_t kernel_launches;       /* kernels queued by this context's calls: 1 per cluster
                                       apply; 3 per grouped apply (grouping, decode shrink,
                                       decode expand) plus 2-3 tensor-core prefill kernels when
                                       the batch has at least the prefill threshold of tokens
                                       (queued even if no run is that long; they then exit at
                                       once); 1 per lora_load_slot, per upload kernel of
                                       lora_load_slots and per device-side eviction. A call
                                       made during stream capture counts once, when captured,
                                       however often the graph runs. */
    uint64_t aborted_loads;         /* lora_abort_load calls that emptied a slot */
} lora_stats_t;

/*
 * Bytes of device workspace a context needs. The workspace holds the token
 * grouping, the fp32 rank-r intermediates and the split reduction partials.
 * max_tokens bounds n_tokens of every apply call; max_layers_per_call bounds n
 * of lora_apply_multi (1..8).
 */
size_t lora_workspace_bytes(int max_loras, int max_lora_rank, int max_tokens,
                            int max_layers_per_call);

/*
 * Create a context: the GPU slot table of the "Multi-LoRA 适配器缓存生产实战"
 * page (section 核心原理, parameter table: max_loras adapters usable in one
 * batch, ranks up to max_lora_rank). max_loras: 1..256 slots. max_lora_rank:
 * 8..256, a multiple of 8. dtype: lora_dtype. layers[n_layers]: shapes and pools (d_in,
 * d_out >= 1). scale_dev / rank_dev: device arrays [max_loras] (fp32 / int32)
 * that the library writes on every upload or eviction. workspace: device,
 * lora_workspace_bytes(...) bytes, 256-byte aligned; it is zeroed here (on the
 * compute stream). compute_stream / upload_stream: caller-owned cudaStream_t.
 * max_tokens: at most 4,096 x the GPU's SM count (622,592 tokens on a
 * 152-SM GB300), else LORA_ERR_ARG.
 *
 * n_layers == 0 creates a host-only slot table: no CUDA call is made, and only
 * the slot-table calls (lookup, assign and its batched forms, acquire,
 * release, evict_lru, abort_load, pin, the policy settings, tick, stats) and
 * lora_load_slot (bookkeeping only) may be used. That is how the slot-table
 * decisions are tested without a GPU.
 *
 * On success *out owns host state and CUDA events; free it with lora_destroy.
 */
int lora_slots_init(lora_ctx **out, int max_loras, int max_lora_rank, int max_tokens,
                    int max_layers_per_call, int dtype,
                    int n_layers, const lora_layer_desc *layers,
                    float *scale_dev, int32_t *rank_dev,
                    void *workspace, size_t workspace_bytes,
                    void *compute_stream, void *upload_stream);

/* Release events and host state. Waits for work the library queued. NULL ok.
 * (Resource handling only; no counterpart on the source pages.) */
void lora_destroy(lora_ctx *ctx);

/*
 * Upload one adapter into slot `slot` (tier L1 of the "Multi-LoRA
 * 适配器缓存生产实战" page, section 冷加载延迟: CPU hit -> H2D upload).
 * A_host[l] is [rank][d_in] and B_host[l] is [d_out][rank] for every layer l,
 * host memory (pinned for a truly asynchronous copy) that the caller keeps
 * alive and unchanged until the upload completes (lora_sync_uploads, or any
 * later host sync on the upload stream). Ranks below max_lora_rank are padded
 * with zeros; scale_dev[slot] = alpha / rank, rank_dev[slot] = rank.
 * Validation (slot range, 1 <= rank <= max_lora_rank, non-NULL pointers,
 * finite alpha) happens before anything is queued: a rejected call changes
 * nothing. The copies wait for compute work already queued (so a slot being
 * read is never overwritten) and the next apply waits for the copies. On a
 * host-only context (n_layers == 0) nothing is copied: the call only records
 * that the slot's adapter has arrived (see lora_abort_load), after the same
 * validation of slot, rank and alpha.
 */
int lora_load_slot(lora_ctx *ctx, int slot, const void *const *A_host,
                   const void *const *B_host, int rank, float alpha);

/*
 * Apply the delta of one layer: y[t] += scale_s * B_s (A_s x[t]) for the
 * n_tokens rows of x / y (device), scale_s = lora_alpha / r of the adapter in
 * slot s (the PEFT adapter_config.json on the "vLLM LoRA Resolver 插件详解"
 * page, section 3.2). token_slot_idx: device int32 [n_tokens].
 * Index -1, an index >= max_loras or < -1 (counted in invalid_token_index), or
 * an empty slot (rank 0) leaves y[t] bit-for-bit unchanged. Stream-ordered on
 * the compute stream; no host synchronisation. 0 <= n_tokens <= max_tokens.
 * Rows of x must not alias rows of y.
 */
int lora_apply(lora_ctx *ctx, int layer, const void *x, void *y,
               const int32_t *token_slot_idx, int n_tokens);

/*
 * Apply n layers (a layer set: the adapter's target_modules, q_proj and v_proj
 * in the PEFT config of the "vLLM LoRA Resolver 插件详解" page, section 3.2;
 * q/k/v/o in the adapter manifest of the "Multi-LoRA 适配器缓存生产实战" page,
 * section "Adapter 容量不能只按「个数」规划") that share one token
 * batch and one token_slot_idx. xs[i] / ys[i] are the device input / output of
 * layer layers[i]. Layers may share an input pointer (q, k, v read the same
 * hidden state). The grouping of tokens by slot is computed once for the set.
 */
int lora_apply_multi(lora_ctx *ctx, int n, const int *layers, const void *const *xs,
                     void *const *ys, const int32_t *token_slot_idx, int n_tokens);

/*
 * The same as lora_apply_multi with HOST buffers: copies the inputs (distinct
 * xs_host once each, ys_host, idx_host) to the caller's device staging buffers
 * xs_dev / ys_dev / idx_dev, applies, and copies every y back to ys_host.
 * The copies in run on the upload stream, each device buffer after the copies
 * back of the last call that used it; the apply runs on the compute stream and
 * the copies back on a download stream the context creates on first use (it
 * owns and destroys it). A caller rotating two or more sets of device buffers
 * thus keeps both directions of the host link and the kernels busy at once;
 * reusing one set is also correct (the calls then serialise). The staging
 * buffers belong to this path until lora_sync_host returns: other work on them
 * must not be queued before that. Copies that continue one another
 * in both host and device memory, in the order idx, then per layer x (once per
 * distinct input) and y, are merged: a caller that packs idx | x | y_0 | y_1 ...
 * back to back in one pinned block and one device block gets one copy in and
 * one copy back per call. Under stream capture everything runs on the compute
 * stream. Returns after queuing; call lora_sync_host before reading ys_host or
 * reusing a host buffer. Host buffers should be pinned.
 */
int lora_apply_multi_host(lora_ctx *ctx, int n, const int *layers,
                          const void *const *xs_host, void *const *ys_host,
                          const int32_t *idx_host, int n_tokens,
                          void *const *xs_dev, void *const *ys_dev, int32_t *idx_dev);

/* Blocks until the copies back of every queued lora_apply_multi_host call have
 * landed in host memory (LORA_OK at once for a host-only context).
 * (Host-buffer plumbing; no counterpart on the source pages.) */
int lora_sync_host(lora_ctx *ctx);

/*
 * Host slot table (the LRU of the "Multi-LoRA 适配器缓存生产实战" page, section
 * 核心原理). adapter ids are opaque 64-bit keys. The LRU clock advances by one
 * on every touch or bind, so no two slots tie.
 */

/* Hit: touch and return the slot in *slot. Miss: *slot = -1 (no state change). */
int lora_lookup(lora_ctx *ctx, uint64_t adapter_id, int *slot);

/*
 * Hit: touch, *slot = its slot, *needs_load = 0. Miss: validate rank first
 * (LORA_ERR_RANK, nothing evicted), then take the lowest free slot (bound to
 * no adapter and holding no reference; see lora_abort_load), else evict
 * the slot the eviction policy picks among those not in flight, not pinned and
 * not cooling (least recently used by default; LORA_ERR_NO_SLOT if none);
 * bind the id, *needs_load = 1, *evicted_id = the removed id or UINT64_MAX.
 * The caller then uploads with lora_load_slot.
 */
int lora_assign(lora_ctx *ctx, uint64_t adapter_id, int rank, int *slot,
                int *needs_load, uint64_t *evicted_id);

/*
 * n lora_assign calls in order (and, if acquire != 0, lora_acquire on each
 * resulting slot), for serving loops that admit a batch's adapters at once.
 * Outputs per entry as for lora_assign. Stops at the first failure and returns
 * its status; *n_done = entries completed (their effects stay).
 */
int lora_assign_batch(lora_ctx *ctx, int n, const uint64_t *adapter_ids, const int *ranks, int acquire,
                      int *slots, int *needs_load, uint64_t *evicted_ids, int *n_done);

/*
 * Admission for one batch given per token: adapter_ids[t] is the adapter of
 * token t (LORA_NO_ADAPTER: base model only) and ranks[t] its rank (read where
 * the adapter first appears). The distinct adapters, in order of first
 * appearance, go through lora_assign_batch exactly (same decisions, same
 * acquire); their ids, slots, load flags and evicted ids are written to
 * distinct_ids / slots / needs_load / evicted_ids[max_distinct], and
 * *n_distinct = their number. token_slot_idx[T] (host memory; may be the
 * pinned buffer handed to lora_apply_multi_host) receives each token's slot,
 * -1 for base tokens and for tokens whose adapter was not admitted. More than
 * max_distinct adapters: LORA_ERR_ARG before any admission (table unchanged).
 * Otherwise returns the first failed admission's status (LORA_ERR_RANK,
 * LORA_ERR_NO_SLOT), with *n_done = adapters admitted (their effects stay).
 * This is the slot lookup of a serving step (touch on hit, bind on miss;
 * section 核心原理 of the "Multi-LoRA 适配器缓存生产实战" page) done in one call.
 */
int lora_assign_tokens(lora_ctx *ctx, int n_tokens, const uint64_t *adapter_ids, const int *ranks,
                       int acquire, int32_t *token_slot_idx, int max_distinct, uint64_t *distinct_ids,
                       int *slots, int *needs_load, uint64_t *evicted_ids, int *n_distinct, int *n_done);

/*
 * The host adapter store of lora_serve_step: the CPU-resident adapters that a
 * miss uploads (tier L1 of the "Multi-LoRA 适配器缓存生产实战" page, section
 * 冷加载延迟). Entry i: id ids[i] (distinct, not LORA_NO_ADAPTER), rank
 * ranks[i] (1..max_lora_rank, else LORA_ERR_RANK), lora_alpha alphas[i], and
 * per layer l the host pointers A_host[i * n_layers + l] ([rank][d_in]) and
 * B_host[i * n_layers + l] ([d_out][rank]) laid out as for lora_load_slot (NULL
 * allowed on a host-only context). The library copies the table, not the
 * weights: the caller keeps that memory alive and unchanged while it stays
 * registered. A new call replaces the whole store; a rejected call changes
 * nothing.
 */
int lora_register_host_adapters(lora_ctx *ctx, int n, const uint64_t *ids, const int *ranks,
                                const float *alphas, const void *const *A_host, const void *const *B_host);

/*
 * The warm set of lora_serve_step: adapters pinned (lora_pin) when a step binds
 * them or finds them resident unpinned, so the eviction policy never removes
 * them (the warm set / pin of the "Multi-LoRA 适配器缓存生产实战" page, section
 * 为什么纯 LRU 在多租户场景下容易失效). Replaces the previous set; removing an id
 * does not unpin a slot already pinned.
 */
int lora_set_warm_set(lora_ctx *ctx, int n, const uint64_t *ids);

/*
 * One serving step in one call: the batch's tokens name their adapters
 * (adapter_ids[t], LORA_NO_ADAPTER for base-model tokens), every adapter
 * registered with lora_register_host_adapters. The distinct adapters, in order
 * of first appearance, are cut into groups that fit the slots (max_loras
 * adapters per batch, section 核心原理 of the "Multi-LoRA 适配器缓存生产实战"
 * page): each adapter needs a slot except one already resident in a pinned
 * slot, and the first group takes at most max_loras minus the slots pinned
 * when the step starts; each later group takes that many minus the warm-set
 * adapters pinned by the groups before it (step 1). Group after group:
 *   1. each adapter is admitted as by lora_assign (hit: touch; miss: lowest
 *      free slot or the policy's victim among slots not in flight, pinned or
 *      cooling) and taken in flight (lora_acquire); warm-set adapters are
 *      pinned;
 *   2. the misses are uploaded from the store (lora_load_slots);
 *   3. idx_bufs[g * n_tokens + t] receives token t's slot if its adapter is in
 *      group g, else -1, and the delta of the n layers is applied to those
 *      tokens (lora_apply_multi with xs / ys, reading that buffer);
 *   4. the group's references are released.
 * Then the epoch advances (lora_tick). idx_bufs (max_groups * n_tokens int32)
 * is written by the host and read by the kernels: host memory the GPU can read
 * (page-locked, or any host memory on a GPU that walks the host's page
 * tables), which the caller does not rewrite until the step's kernels have run
 * (the compute stream). Outputs, per distinct adapter in order (when
 * max_distinct > 0): its id, slot, whether it was uploaded, and the id it
 * evicted (LORA_NO_ADAPTER if none); *n_distinct and *n_groups.
 * Errors before any admission leave the table unchanged: an unregistered id,
 * more than max_distinct adapters, more than max_groups groups (device
 * contexts), bad arguments. A failed admission (LORA_ERR_NO_SLOT) or upload
 * returns its status after releasing the references of its group (the misses
 * the group bound before a failed admission are still uploaded, so no slot is
 * left bound without its weights); the groups before it were applied and
 * released, and the epoch does not advance.
 * On a host-only context only the admission runs (uploads are recorded as by
 * lora_load_slot there; layers, xs, ys and idx_bufs may be NULL).
 */
int lora_serve_step(lora_ctx *ctx, int n_tokens, const uint64_t *adapter_ids, int n, const int *layers,
                    const void *const *xs, void *const *ys, int32_t *idx_bufs, int max_groups, int max_distinct,
                    uint64_t *out_ids, int *out_slots, int *out_needs_load, uint64_t *out_evicted,
                    int *n_distinct, int *n_groups);

/* lora_release on each of slots[n] in order; stops at the first slot not in flight (LORA_ERR_STATE).
 * The in-flight protection of the "Multi-LoRA 适配器缓存生产实战" page: section 核心原理, last
 * paragraph, and the inflight_requests field of section 数据面. */
int lora_release_batch(lora_ctx *ctx, int n, const int *slots);

/* In-flight reference count of an occupied slot (never evicted while > 0): the
 * inflight_requests field of the "Multi-LoRA 适配器缓存生产实战" page, section 数据面.
 * LORA_ERR_STATE: acquire of an empty slot, release of a slot not in flight. */
int lora_acquire(lora_ctx *ctx, int slot);
int lora_release(lora_ctx *ctx, int slot);

/*
 * Evict the occupied slot the eviction policy picks (least recently used by
 * default) among those not in flight, not pinned and not cooling.
 * *evicted_slot = -1 when no slot is occupied (LORA_OK). LORA_ERR_NO_SLOT when
 * no occupied slot may be evicted. With a device context the slot's rank is
 * set to 0 on the device, after compute work already queued.
 */
int lora_evict_lru(lora_ctx *ctx, int *evicted_slot, uint64_t *evicted_id);

/*
 * The upload into `slot` failed or was abandoned (the "load failed" outcome the
 * "vLLM LoRA Resolver 插件详解" page gives a dynamic load, section 6.1). Valid
 * only while that upload is pending: the slot was bound by a miss of
 * lora_assign (or a batched admission) and no lora_load_slot / lora_load_slots
 * into it has been queued since; an adapter whose upload was queued is removed
 * with eviction instead. The adapter is unbound, so it is no longer resident
 * and a later assign of it is a miss that loads it again; the adapter the
 * assign evicted stays evicted (its slot bytes may already be overwritten).
 * Counted in aborted_loads, not as an eviction; the pin ends. References
 * already taken on the slot (lora_acquire) stay and are released as usual: the
 * slot is bound to no adapter meanwhile and becomes free for a new adapter only
 * once none is left, so a late release can never lower the count of an adapter
 * bound to the slot later. With a device context the slot reads as empty (rank
 * 0) for work queued after this call, after compute already queued.
 * *unbound_id = the id that was bound. LORA_ERR_ARG: slot out of range or
 * NULL; LORA_ERR_STATE: the slot is empty or its upload was already queued.
 */
int lora_abort_load(lora_ctx *ctx, int slot, uint64_t *unbound_id);

/* Advance the epoch used by the thrash window (call once per step). The window
 * is the "short time window" of adapter_thrash_ratio on the "Multi-LoRA
 * 适配器缓存生产实战" page, section 需要重点监控哪些指标; the page leaves its unit
 * open, and epochs (steps) are this library's reading. */
int lora_tick(lora_ctx *ctx);

/* Set the thrash window in epochs (default 10): a reload at most this many
 * epochs after the adapter's eviction counts in reloads_after_eviction (the
 * numerator of adapter_thrash_ratio, same page and section as lora_tick).
 * < 0 is LORA_ERR_ARG. */
int lora_set_thrash_window(lora_ctx *ctx, int epochs);

/*
 * Upload several adapters at once (the CPU-hit tier, L1 of section 冷加载延迟 of
 * the "Multi-LoRA 适配器缓存生产实战" page; its cost is the adapter_h2d term of
 * the TTFT decomposition there). slots[n], ranks[n], alphas[n]; A_host and
 * B_host hold n * n_layers host pointers, adapter-major (entry i * n_layers +
 * l is layer l of adapter i), each laid out as for lora_load_slot. Adapters
 * the GPU can read in place with 16-byte aligned rows (r * bytes_per_param
 * and d_in * bytes_per_param multiples of 16) are copied by one kernel that
 * reads host memory directly and also zero-fills the padding and sets scale =
 * alpha / r and the rank: any host memory where the device walks the host's
 * page tables (pageable-memory access through host page tables, as on
 * Grace-based systems), else page-locked device-mapped buffers (cudaHostAlloc,
 * torch pin_memory). Any other adapter takes the copy-engine path of
 * lora_load_slot. Same ordering and statistics as n calls of lora_load_slot
 * (one event covers the whole call). Everything is validated before anything is queued
 * (LORA_ERR_ARG: bad slot, a slot twice, NULL; LORA_ERR_RANK). The host
 * buffers must stay alive and unchanged until lora_sync_uploads returns.
 */
int lora_load_slots(lora_ctx *ctx, int n, const int *slots, const void *const *A_host,
                    const void *const *B_host, const int *ranks, const float *alphas);

/*
 * Per-slot ordering of uploads (copy/compute overlap; the adapter_h2d term of
 * the TTFT decomposition and the H2D metric of the "Multi-LoRA 适配器缓存生产实战"
 * page, sections 冷加载延迟 and 需要重点监控哪些指标). By default an upload or an
 * eviction waits for every apply queued before it. With tracking on, the
 * caller promises that each apply's token_slot_idx names only slots it holds
 * in flight (lora_acquire) when it calls apply; an upload into slot s then
 * waits only for the last apply issued while s was in flight, so the next
 * step's adapters can be copied while the current step computes. Device
 * contexts only (LORA_ERR_STATE otherwise).
 */
int lora_set_slot_tracking(lora_ctx *ctx, int on);

/*
 * Eviction policies on top of LRU, from the "Multi-LoRA 适配器缓存生产实战" page,
 * section 为什么纯 LRU 在多租户场景下容易失效 (warm set / pin, a cooling window
 * against short bursts, a recency + frequency keep_score), and the `pinned`
 * field of section 数据面. Every policy still never evicts a slot in flight,
 * still uses the lowest free slot first and still validates the rank before
 * anything is evicted. They apply to lora_assign and lora_evict_lru alike.
 */

/*
 * Pin (pinned != 0) or unpin the adapter in an occupied slot: a pinned slot
 * is never chosen for eviction (the warm set). LORA_ERR_STATE if the slot is
 * empty, LORA_ERR_ARG if out of range. The pin ends when the slot is unpinned;
 * a pinned adapter can still be replaced only by first unpinning it.
 */
int lora_pin(lora_ctx *ctx, int slot, int pinned);

/*
 * Cooling window: an adapter accessed (hit or bound) within the last `epochs`
 * epochs (current epoch - last access epoch < epochs) is not evicted; an
 * assign that finds nothing else evictable returns LORA_ERR_NO_SLOT, and the
 * caller defers that adapter. 0 (default) turns the window off; < 0 is
 * LORA_ERR_ARG.
 */
int lora_set_min_residency(lora_ctx *ctx, int epochs);

enum lora_policy {
    LORA_POLICY_LRU = 0,         /* least recently used (default) */
    LORA_POLICY_KEEP_SCORE = 1,  /* lowest keep_score, ties to the least recently used */
};

/*
 * Select the eviction policy. keep_score of a resident adapter at epoch E:
 *   recent     = 1 / (1 + (E - last access epoch))
 *   frequency  = hits and binds in the last W epochs (epoch > E - W), W the
 *                thrash window of lora_set_thrash_window
 *   priority   = the value set with lora_set_adapter_priority (default 0)
 *   reload_cost = size = rank / max_lora_rank  (relative H2D and slot bytes)
 *   keep = w1 recent + w2 frequency + w3 priority + w4 reload_cost - w5 size
 * evaluated in double precision in that order. LORA_ERR_ARG for an unknown policy.
 */
int lora_set_policy(lora_ctx *ctx, int policy);

/* keep_score weights w1..w5 (host array of 5 doubles; default 1, 1, 1, 0, 0). */
int lora_set_keep_score_weights(lora_ctx *ctx, const double *w);

/* The tenant / SLO priority term of keep_score for one adapter id (default 0). */
int lora_set_adapter_priority(lora_ctx *ctx, uint64_t adapter_id, double priority);

/*
 * (Implementation controls from here to lora_set_inputs_ready: they choose
 * kernels and launch order, never the result; the source pages have no
 * counterpart.)
 *
 * Segment-length threshold for the tensor-core prefill path (bf16 contexts
 * with max_lora_rank 16, 32 or 64; layers with d_out a multiple of 64):
 * contiguous runs of tokens on one slot at least this long use it; shorter
 * runs and decode tokens use the grouped decode kernels. 0 disables the
 * prefill path. Values 1..31 are raised to 32. Default 64: measured on GB300,
 * runs of 32-63 tokens are 20-40 % faster on the prefill path, but a lower
 * threshold also enlarges its grid and costs batches of long runs 0.6-1.8 %.
 */
int lora_set_prefill_min_tokens(lora_ctx *ctx, int n);

/*
 * Batches of at most n tokens (0..1024) take the single-launch decode kernel
 * (thread-block clusters), which treats every token as a decode token; larger
 * batches take the grouping + tensor-core prefill + decode kernels. 0 always
 * takes the latter. By default (and after n = -1) the limit follows
 * max_lora_rank: 1024 tokens up to rank 16, 768 up to rank 32, 0 above (where
 * the grouped kernels are faster at every batch size).
 */
int lora_set_small_batch_tokens(lora_ctx *ctx, int n);

/*
 * on != 0 declares that, for every following apply call on this context, x,
 * token_slot_idx, the slot pools and scale_dev / rank_dev are not written by
 * the kernel launched immediately before that call on the compute stream (y
 * may be: the usual case of a base-model GEMM writing y right before the
 * delta is added). The single-launch decode kernel then starts while that
 * kernel finishes (programmatic dependent launch), groups the tokens and
 * loads x and the slot weights early, and waits for it only before reading y.
 * Default 0: everything waits for the preceding kernel.
 */
int lora_set_inputs_ready(lora_ctx *ctx, int on);

/* Block until every queued upload finished; accumulates upload_seconds (the
 * adapter_h2d time of the page's TTFT decomposition, section 冷加载延迟). */
int lora_sync_uploads(lora_ctx *ctx);

/* Counters; synchronises the compute stream to read the device error count.
 * hits, misses, evictions and the reload count are the residency counters of
 * the "Multi-LoRA 适配器缓存生产实战" page (section 数据面: hit_count, load_count,
 * eviction_count) and the inputs of its thrash ratio and H2D metrics (section
 * 需要重点监控哪些指标). */
int lora_stats(lora_ctx *ctx, lora_stats_t *out);

/*
 * Failure-path self test (no counterpart on the source pages): launches, on
 * the compute stream, a one-CTA kernel that waits on a barrier nothing
 * completes, with the same bounded wait every kernel of the library uses, and
 * a two-CTA cluster kernel whose CTAs wait on their partial-exchange barriers
 * with the cluster decode kernel's bounded cluster-scope wait while no peer
 * arrives. Each wait gives up after 2^14 probes, the kernel sets the device
 * error word and returns; *gave_up = 1 once all three have. The word stays
 * set, as after a real timeout, and lora_stats reports it
 * (device_wait_timeouts). Nothing faults or hangs and the context stays
 * usable. Synchronises the compute stream.
 */
int lora_selftest_wait_timeout(lora_ctx *ctx, int *gave_up);

/* Bytes one adapter upload moves: sum over layers of (d_in + d_out) * rank * bytes_per_param
 * (the capacity formula of the "Multi-LoRA 适配器缓存生产实战" page, section
 * "Adapter 容量不能只按「个数」规划"). 0 for negative or NULL arguments. */
uint64_t lora_adapter_bytes(int n_layers, const int *d_in, const int *d_out, int rank,
                            int bytes_per_param);

/*
 * One layer of the delta with no workspace and no allocation. The source pages
 * have no counterpart to this call: it exists for callers that cannot allocate
 * device memory for a context workspace -- a plugin whose host application
 * owns every device allocation through its own pool, a process that reserved
 * all device memory up front, or a latency-critical path that must not call
 * the allocator (cudaMalloc can synchronise the device and fail at run time).
 *
 * The result is the one lora_apply computes for the same layer (grouped
 * decode kernels; every token, long segments included, takes that path). The
 * caller passes inputs and outputs exactly as described for lora_apply and
 * lora_slots_init: x [n_tokens][d_in], y [n_tokens][d_out] updated in place,
 * device token_slot_idx, the layer's slot pools in the layouts given at the
 * top of this file (A_pool [max_loras][max_lora_rank][d_in], B_pool blocked by
 * rank; 16-byte aligned), scale_dev / rank_dev [max_loras] as lora_load_slot
 * fills them,
 * and the stream the work is queued on (cudaStream_t as void*).
 *
 * Scratch comes from a file-scope device array of 4 MiB that every GPU loading
 * this library holds until the process exits. Calls needing more (large
 * n_tokens at large max_lora_rank: more than 8,090 tokens at max_lora_rank 64)
 * return LORA_ERR_ARG with a message. Every call looks up that array's address
 * on the current device (so a device reset or another context on the device
 * is handled); the first call on a device also loads the library's device
 * code there: make it before any stream capture. All calls share the array,
 * which keeps the previous call's contents (what must start at zero is
 * cleared on `stream` at the start of each call): calls whose work overlaps on
 * the GPU race and must be serialised. The call calls no cudaMalloc, cudaFree
 * or other allocating routine.
 */
int lora_apply_static_scratch(const void *x, void *y, const int32_t *token_slot_idx,
                              int n_tokens, int d_in, int d_out, int max_loras,
                              int max_lora_rank, int dtype, const void *A_pool,
                              const void *B_pool, const float *scale_dev,
                              const int32_t *rank_dev, void *stream);

/* Message for the last failed call on this thread ("" if none; error reporting
 * only, no counterpart on the source pages). */
const char *lora_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RANK_ADAPTER_APPLY_H */
