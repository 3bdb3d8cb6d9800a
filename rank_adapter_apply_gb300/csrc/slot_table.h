// Host-side adapter slot table: adapter id -> GPU slot, LRU clock, in-flight
// reference counts and the residency counters of the "Multi-LoRA
// 适配器缓存生产实战" page (section 核心原理: touch on hit, oldest evicted,
// adapters in use never evicted; section 数据面: load / hit / eviction counts,
// inflight_requests; section 需要重点监控哪些指标: reload-after-eviction).
#pragma once

#include <cstdint>
#include <unordered_map>
#include <vector>

namespace lora {

struct AdapterResidency {
    uint64_t load_count = 0;
    uint64_t hit_count = 0;
    uint64_t eviction_count = 0;
    int64_t last_evict_epoch = -1;   // -1: never evicted
};

enum class AssignResult { Hit, Loaded, BadRank, NoSlot };

class SlotTable {
public:
    SlotTable(int max_loras, int max_lora_rank);

    // Hit: touch, return slot. Miss: -1, no state change.
    int lookup(uint64_t id);
    // See lora_assign in the public header.
    AssignResult assign(uint64_t id, int rank, int *slot, uint64_t *evicted_id);
    bool acquire(int slot);
    bool release(int slot);
    // Returns false when every occupied slot is in flight. *slot = -1 if empty.
    bool evict_lru(int *slot, uint64_t *evicted_id);

    void tick() { ++epoch_; }
    void set_window(int w) { window_ = w; }
    bool occupied(int slot) const { return occ_[slot]; }
    int refs(int slot) const { return refs_[slot]; }

    uint64_t hits = 0, misses = 0, evictions = 0, reloads = 0, rejected = 0;
    int64_t epoch() const { return epoch_; }

private:
    int victim() const;
    uint64_t evict(int slot);
    void touch(int slot) { last_use_[slot] = ++clock_; }

    int S_, R_;
    int window_ = 10;
    uint64_t clock_ = 0;
    int64_t epoch_ = 0;
    std::vector<uint64_t> id_;
    std::vector<char> occ_;
    std::vector<uint64_t> last_use_;
    std::vector<int> refs_;
    std::unordered_map<uint64_t, int> where_;
    std::unordered_map<uint64_t, AdapterResidency> rec_;
};

}  // namespace lora
