// Host-side helpers shared by the C ABI translation units.
#pragma once

#include <stdint.h>

#include <vector>

#include "../../include/dmuon.h"

namespace dmuon {

// Record `msg` as the calling thread's last error and return `status`.
int set_error(int status, const char* msg);
void clear_error();

// LPT core (see lpt.cpp).  When `order_out` is given it receives the order
// in which items were placed (descending size, ties by index).
int lpt_assign_impl(const int64_t* sizes, int32_t n_items, int32_t n_slots, int32_t* out_slot,
                    int64_t* out_load, std::vector<int32_t>* order_out);

// Checks of one Muon tensor descriptor (rank, dimensions, slice size,
// pointers, dtype); `idx` names it in the message (see api.cu).
int validate_matrix(const dmuon_matrix& M, int idx);

// Device address of the allocation-free entry point's error word on the
// current device (see noalloc.cu).
int noalloc_error_word(int** out);

// DMUON_ERR_INVALID_ARG (with the two ranges named) when memory a step
// writes overlaps other written memory or a gradient (see api.cu).
int check_no_overlap(const dmuon_matrix* mats, int n, const dmuon_vector* vecs, int nv);

}  // namespace dmuon
