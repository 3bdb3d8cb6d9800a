#include "slot_table.h"

namespace lora {

SlotTable::SlotTable(int max_loras, int max_lora_rank)
    : S_(max_loras), R_(max_lora_rank), id_(max_loras, 0), occ_(max_loras, 0), pin_(max_loras, 0),
      pending_(max_loras, 0), last_use_(max_loras, 0), refs_(max_loras, 0), res_(max_loras, nullptr) {}

void SlotTable::touch(int slot) {
    last_use_[slot] = ++clock_;
    AdapterResidency &r = *res_[slot];
    r.last_access_epoch = epoch_;
    if (!r.accesses.empty() && r.accesses.back().first == epoch_) ++r.accesses.back().second;
    else r.accesses.emplace_back(epoch_, 1u);
    // Entries older than the window no longer count; keep the list short.
    size_t drop = 0;
    while (drop < r.accesses.size() && r.accesses[drop].first <= epoch_ - window_) ++drop;
    if (drop) r.accesses.erase(r.accesses.begin(), r.accesses.begin() + (long)drop);
}

int SlotTable::lookup(uint64_t id) {
    auto it = where_.find(id);
    if (it == where_.end()) return -1;
    touch(it->second);
    ++hits;
    ++res_[it->second]->hit_count;
    return it->second;
}

bool SlotTable::evictable(int s) const {
    if (!occ_[s] || refs_[s] > 0 || pin_[s]) return false;
    if (min_res_ > 0) {
        const AdapterResidency &r = *res_[s];
        if (epoch_ - r.last_access_epoch < min_res_) return false;
    }
    return true;
}

// Evaluated in this order in double precision (the simulator does the same).
double SlotTable::keep_score(int s) const {
    const AdapterResidency &r = *res_[s];
    const double recent = 1.0 / (1.0 + (double)(epoch_ - r.last_access_epoch));
    uint64_t n = 0;
    for (const auto &a : r.accesses)
        if (a.first > epoch_ - window_) n += a.second;
    const double freq = (double)n;
    const double rel = (double)r.rank / (double)R_;
    double k = w_[0] * recent;
    k += w_[1] * freq;
    k += w_[2] * r.priority;
    k += w_[3] * rel;
    k -= w_[4] * rel;
    return k;
}

// The evictable slot chosen by the policy; -1 if none.
int SlotTable::victim() const {
    int best = -1;
    if (policy_ == EvictPolicy::Lru && min_res_ == 0) {
        // the first evictable slot with the smallest LRU clock, in one pass
        // over the flat arrays
        uint64_t best_t = UINT64_MAX;
        for (int s = 0; s < S_; ++s) {
            const bool ok = occ_[s] && refs_[s] == 0 && !pin_[s];
            if (ok && last_use_[s] < best_t) {
                best_t = last_use_[s];
                best = s;
            }
        }
        return best;
    }
    double best_k = 0.0;
    for (int s = 0; s < S_; ++s) {
        if (!evictable(s)) continue;
        if (policy_ == EvictPolicy::Lru) {
            if (best < 0 || last_use_[s] < last_use_[best]) best = s;
        } else {
            const double k = keep_score(s);
            if (best < 0 || k < best_k || (k == best_k && last_use_[s] < last_use_[best])) {
                best = s;
                best_k = k;
            }
        }
    }
    return best;
}

uint64_t SlotTable::evict(int slot) {
    uint64_t id = id_[slot];
    occ_[slot] = 0;
    --n_occ_;
    pin_[slot] = 0;
    pending_[slot] = 0;
    refs_[slot] = 0;
    where_.erase(id);
    ++evictions;
    AdapterResidency &r = *res_[slot];
    res_[slot] = nullptr;
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
    // A free slot: unbound and unreferenced (a slot whose load was aborted
    // stays taken until its references are released).
    int s = -1;
    if (n_occ_ < S_)
        for (int i = 0; i < S_; ++i)
            if (!occ_[i] && refs_[i] == 0) { s = i; break; }
    if (s < 0) {
        s = victim();
        if (s < 0) {
            *slot = -1;
            return AssignResult::NoSlot;
        }
        *evicted_id = evict(s);
    }
    AdapterResidency &r = rec_[id];
    res_[s] = &r;
    if (r.last_evict_epoch >= 0 && epoch_ - r.last_evict_epoch <= window_) ++reloads;
    ++r.load_count;
    r.rank = rank;
    id_[s] = id;
    occ_[s] = 1;
    ++n_occ_;
    pin_[s] = 0;
    pending_[s] = 1;
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

bool SlotTable::pin(int slot, bool on) {
    if (slot < 0 || slot >= S_ || !occ_[slot]) return false;
    pin_[slot] = on ? 1 : 0;
    return true;
}

bool SlotTable::abort_load(int slot, uint64_t *unbound_id) {
    *unbound_id = UINT64_MAX;
    if (slot < 0 || slot >= S_ || !occ_[slot] || !pending_[slot]) return false;
    const uint64_t id = id_[slot];
    occ_[slot] = 0;
    --n_occ_;
    pin_[slot] = 0;
    pending_[slot] = 0;
    where_.erase(id);
    res_[slot] = nullptr;
    ++aborted_loads;
    *unbound_id = id;
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
