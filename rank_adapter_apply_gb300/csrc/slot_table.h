// Host-side adapter slot table: adapter id -> GPU slot, eviction choice,
// in-flight reference counts and the residency counters of the "Multi-LoRA
// 适配器缓存生产实战" page (section 核心原理: touch on hit, oldest evicted,
// adapters in use never evicted; section 数据面: load / hit / eviction counts,
// pinned, inflight_requests; section 需要重点监控哪些指标: reload-after-eviction).
//
// Platform policies on top of LRU (section 为什么纯 LRU 在多租户场景下容易失效):
//  * pinned slots (warm set) are never chosen for eviction;
//  * a cooling window: an adapter accessed within the last `min_residency`
//    epochs is not evicted (0 = off);
//  * a keep_score policy: evict the evictable adapter with the lowest
//      keep = w1 recent + w2 frequency + w3 priority + w4 reload_cost - w5 size
//    with recent = 1 / (1 + epochs since the last access), frequency = hits
//    and binds in the last `window` epochs (the thrash window), priority set
//    by the caller, reload_cost = size = rank / max_lora_rank (relative bytes
//    of an H2D reload and of the slot payload). Ties go to the older LRU clock.
#pragma once

#include <cstdint>
#include <unordered_map>
#include <utility>
#include <vector>

namespace lora {

struct AdapterResidency {
    uint64_t load_count = 0;
    uint64_t hit_count = 0;
    uint64_t eviction_count = 0;
    int64_t last_evict_epoch = -1;   // -1: never evicted
    int64_t last_access_epoch = -1;
    std::vector<std::pair<int64_t, uint32_t>> accesses;   // (epoch, count), recent epochs only
    int rank = 0;
    double priority = 0.0;
};

enum class AssignResult { Hit, Loaded, BadRank, NoSlot };
enum class EvictPolicy { Lru = 0, KeepScore = 1 };

class SlotTable {
public:
    SlotTable(int max_loras, int max_lora_rank);

    // Hit: touch, return slot. Miss: -1, no state change.
    int lookup(uint64_t id);
    // The slot holding the adapter, or -1; no state change (no touch).
    int find(uint64_t id) const {
        auto it = where_.find(id);
        return it == where_.end() ? -1 : it->second;
    }
    // See lora_assign in the public header.
    AssignResult assign(uint64_t id, int rank, int *slot, uint64_t *evicted_id);
    bool acquire(int slot);
    bool release(int slot);
    // Returns false when no occupied slot may be evicted. *slot = -1 if empty.
    bool evict_lru(int *slot, uint64_t *evicted_id);
    // Unbind the adapter of a slot whose upload failed or was abandoned: only
    // while that upload is pending (bound by assign, no upload queued since).
    // The adapter is no longer resident (not counted as an eviction) and the
    // pin ends; references already taken stay until released, and the slot
    // is free again once none is left. False if the slot is out of range,
    // empty or not pending.
    bool abort_load(int slot, uint64_t *unbound_id);
    // An upload into the slot was queued: its adapter is no longer pending.
    void mark_loaded(int slot) { pending_[slot] = 0; }
    bool pending(int slot) const { return pending_[slot]; }

    bool pin(int slot, bool on);
    void set_min_residency(int epochs) { min_res_ = epochs < 0 ? 0 : epochs; }
    void set_policy(EvictPolicy p) { policy_ = p; }
    void set_weights(const double w[5]) {
        for (int i = 0; i < 5; ++i) w_[i] = w[i];
    }
    void set_priority(uint64_t id, double p) { rec_[id].priority = p; }
    double keep_score(int slot) const;

    void tick() { ++epoch_; }
    void set_window(int w) { window_ = w; }
    bool occupied(int slot) const { return occ_[slot]; }
    bool pinned(int slot) const { return pin_[slot]; }
    int refs(int slot) const { return refs_[slot]; }

    uint64_t hits = 0, misses = 0, evictions = 0, reloads = 0, rejected = 0, aborted_loads = 0;
    int64_t epoch() const { return epoch_; }

private:
    bool evictable(int slot) const;
    int victim() const;
    uint64_t evict(int slot);
    void touch(int slot);

    int S_, R_;
    int window_ = 10;
    int min_res_ = 0;
    EvictPolicy policy_ = EvictPolicy::Lru;
    double w_[5] = {1.0, 1.0, 1.0, 0.0, 0.0};
    uint64_t clock_ = 0;
    int64_t epoch_ = 0;
    int n_occ_ = 0;                     // occupied slots (no free slot is searched for when all are)
    std::vector<uint64_t> id_;
    std::vector<char> occ_, pin_, pending_;
    std::vector<uint64_t> last_use_;
    std::vector<int> refs_;
    std::unordered_map<uint64_t, int> where_;
    std::unordered_map<uint64_t, AdapterResidency> rec_;
    // The record of each occupied slot's adapter (elements of an unordered_map
    // keep their address across insertions), so victim scans need no lookup.
    std::vector<AdapterResidency *> res_;
};

}  // namespace lora
