#include "slot_table.h"

namespace lora {

SlotTable::SlotTable(int max_loras, int max_lora_rank)
    : S_(max_loras), R_(max_lora_rank), id_(max_loras, 0), occ_(max_loras, 0),
      last_use_(max_loras, 0), refs_(max_loras, 0) {}

int SlotTable::lookup(uint64_t id) {
    auto it = where_.find(id);
    if (it == where_.end()) return -1;
    touch(it->second);
    ++hits;
    ++rec_[id].hit_count;
    return it->second;
}

// Least recently used occupied slot with no in-flight reference; -1 if none.
int SlotTable::victim() const {
    int best = -1;
    for (int s = 0; s < S_; ++s) {
        if (!occ_[s] || refs_[s] > 0) continue;
        if (best < 0 || last_use_[s] < last_use_[best]) best = s;
    }
    return best;
}

uint64_t SlotTable::evict(int slot) {
    uint64_t id = id_[slot];
    occ_[slot] = 0;
    refs_[slot] = 0;
    where_.erase(id);
    ++evictions;
    AdapterResidency &r = rec_[id];
    ++r.eviction_count;
    r.last_evict_epoch = epoch_;
    return id;
}

AssignResult SlotTable::assign(uint64_t id, int rank, int *slot, uint64_t *evicted_id) {
    *evicted_id = UINT64_MAX;
    int hit = lookup(id);
    if (hit >= 0) {
        *slot = hit;
        return AssignResult::Hit;
    }
    // Validate before touching any resident adapter: a rejected adapter never
    // costs another one its slot.
    if (rank < 1 || rank > R_) {
        ++rejected;
        *slot = -1;
        return AssignResult::BadRank;
    }
    int s = -1;
    for (int i = 0; i < S_; ++i)
        if (!occ_[i]) { s = i; break; }
    if (s < 0) {
        s = victim();
        if (s < 0) {
            *slot = -1;
            return AssignResult::NoSlot;
        }
        *evicted_id = evict(s);
    }
    AdapterResidency &r = rec_[id];
    if (r.last_evict_epoch >= 0 && epoch_ - r.last_evict_epoch <= window_) ++reloads;
    ++r.load_count;
    id_[s] = id;
    occ_[s] = 1;
    refs_[s] = 0;
    where_[id] = s;
    touch(s);
    ++misses;
    *slot = s;
    return AssignResult::Loaded;
}

bool SlotTable::acquire(int slot) {
    if (slot < 0 || slot >= S_ || !occ_[slot]) return false;
    ++refs_[slot];
    return true;
}

bool SlotTable::release(int slot) {
    if (slot < 0 || slot >= S_ || refs_[slot] <= 0) return false;
    --refs_[slot];
    return true;
}

bool SlotTable::evict_lru(int *slot, uint64_t *evicted_id) {
    *slot = -1;
    *evicted_id = UINT64_MAX;
    bool any = false;
    for (int s = 0; s < S_; ++s) any = any || occ_[s];
    if (!any) return true;
    int v = victim();
    if (v < 0) return false;
    *evicted_id = evict(v);
    *slot = v;
    return true;
}

}  // namespace lora
