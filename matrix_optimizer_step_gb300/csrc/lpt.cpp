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

}  // namespace dmuon

extern "C" int dmuon_lpt_assign(const int64_t* sizes, int32_t n_items, int32_t n_slots,
                                int32_t* out_slot, int64_t* out_load) {
  dmuon::clear_error();
  return dmuon::lpt_assign_impl(sizes, n_items, n_slots, out_slot, out_load, nullptr);
}
