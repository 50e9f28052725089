// Longest-processing-time greedy assignment ("架构设计" §3.1 "分区（全局 LPT）").
//
// Items are taken in descending size (equal sizes by ascending index) and
// each goes to the slot with the smallest current load (equal loads: lowest
// slot index).  A binary heap keyed on (load, slot) gives that slot in
// O(log R); the tie rules make the assignment unique, so it can be compared
// bit for bit with any other implementation of the same rules.
#include <stdint.h>

#include <algorithm>
#include <functional>
#include <numeric>
#include <queue>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

#include "../../include/dmuon.h"
#include "host_util.h"

namespace dmuon {

int lpt_assign_impl(const int64_t* sizes, int32_t n_items, int32_t n_slots, int32_t* out_slot,
                    int64_t* out_load, std::vector<int32_t>* order_out) {
  if (n_items < 0 || n_slots < 1 || (n_items > 0 && (!sizes || !out_slot)))
    return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign: bad counts or null pointer");
  for (int32_t i = 0; i < n_items; ++i)
    if (sizes[i] < 0) return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign: negative item size");
  std::vector<int32_t> order(static_cast<size_t>(n_items));
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t x, int32_t y) { return sizes[x] > sizes[y]; });
  using Entry = std::pair<int64_t, int32_t>;  // (load, slot)
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
  for (int32_t s = 0; s < n_slots; ++s) heap.push({0, s});
  std::vector<int64_t> load(static_cast<size_t>(n_slots), 0);
  for (int32_t i : order) {
    Entry e = heap.top();
    heap.pop();
    if (sizes[i] > INT64_MAX - e.first)
      return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign: slot load overflows int64");
    e.first += sizes[i];
    out_slot[i] = e.second;
    load[static_cast<size_t>(e.second)] = e.first;
    heap.push(e);
  }
  if (out_load)
    for (int32_t s = 0; s < n_slots; ++s) out_load[s] = load[static_cast<size_t>(s)];
  if (order_out) order_out->swap(order);
  return DMUON_OK;
}

// Layer-aware variant: same-layer units on distinct slots where possible,
// a layer's items below `small_threshold` merged into one unit.
int lpt_assign_layered_impl(const int64_t* sizes, const int32_t* layers, int32_t n_items, int32_t n_slots,
                            int64_t small_threshold, int32_t* out_slot, int64_t* out_load) {
  if (n_items < 0 || n_slots < 1 || (n_items > 0 && (!sizes || !layers || !out_slot)))
    return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign_layered: bad counts or null pointer");
  struct Unit {
    int64_t size;
    int32_t first;
    int32_t layer;
    std::vector<int32_t> items;
  };
  std::vector<Unit> units;
  std::unordered_map<int32_t, size_t> small_unit;
  for (int32_t i = 0; i < n_items; ++i) {
    if (sizes[i] < 0) return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign_layered: negative item size");
    const int32_t layer = layers[i];
    if (layer >= 0 && sizes[i] < small_threshold) {
      auto it = small_unit.find(layer);
      if (it != small_unit.end()) {
        Unit& u = units[it->second];
        if (sizes[i] > INT64_MAX - u.size)
          return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign_layered: unit size overflows int64");
        u.size += sizes[i];
        u.items.push_back(i);
        continue;
      }
      small_unit.emplace(layer, units.size());
    }
    units.push_back(Unit{sizes[i], i, layer, {i}});
  }
  std::vector<size_t> order(units.size());
  std::iota(order.begin(), order.end(), size_t(0));
  std::sort(order.begin(), order.end(), [&](size_t x, size_t y) {
    if (units[x].size != units[y].size) return units[x].size > units[y].size;
    return units[x].first < units[y].first;
  });
  std::vector<int64_t> load(static_cast<size_t>(n_slots), 0);
  // (slot, layer) pairs already placed, packed into one 64-bit key.
  std::unordered_set<uint64_t> holds;
  auto key = [](int32_t slot, int32_t layer) {
    return (static_cast<uint64_t>(static_cast<uint32_t>(slot)) << 32) | static_cast<uint32_t>(layer);
  };
  for (size_t k : order) {
    const Unit& u = units[k];
    int32_t best = -1;
    for (int pass = 0; pass < 2 && best < 0; ++pass) {
      for (int32_t j = 0; j < n_slots; ++j) {
        if (pass == 0 && u.layer >= 0 && holds.count(key(j, u.layer))) continue;
        if (best < 0 || load[static_cast<size_t>(j)] < load[static_cast<size_t>(best)]) best = j;
      }
    }
    if (u.size > INT64_MAX - load[static_cast<size_t>(best)])
      return set_error(DMUON_ERR_INVALID_ARG, "lpt_assign_layered: slot load overflows int64");
    load[static_cast<size_t>(best)] += u.size;
    if (u.layer >= 0) holds.insert(key(best, u.layer));
    for (int32_t i : u.items) out_slot[i] = best;
  }
  if (out_load)
    for (int32_t s = 0; s < n_slots; ++s) out_load[s] = load[static_cast<size_t>(s)];
  return DMUON_OK;
}

}  // namespace dmuon

extern "C" int dmuon_lpt_assign_layered(const int64_t* sizes, const int32_t* layers, int32_t n_items,
                                        int32_t n_slots, int64_t small_threshold, int32_t* out_slot,
                                        int64_t* out_load) {
  dmuon::clear_error();
  return dmuon::lpt_assign_layered_impl(sizes, layers, n_items, n_slots, small_threshold, out_slot, out_load);
}

extern "C" int dmuon_lpt_assign(const int64_t* sizes, int32_t n_items, int32_t n_slots,
                                int32_t* out_slot, int64_t* out_load) {
  dmuon::clear_error();
  return dmuon::lpt_assign_impl(sizes, n_items, n_slots, out_slot, out_load, nullptr);
}
