// Host-side helpers shared by the three entry points (internal header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/vg.h"

namespace vg {

constexpr int kPageSize = 16;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

// Bound after which a pipeline wait reports VG_DEVERR_TIMEOUT (set with
// vg_set_wait_limit_ns; 1 s by default).  Kernels take it as a parameter.
uint64_t wait_report_ns();

// 4-D tiled TMA descriptor over a page pool viewed as
// [num_pages][num_kv_heads][16][head_dim] bf16, box = 64 x 16 x 1 x 1 with the
// 128-byte swizzle.  Cached per (pointer, shape).  Returns false on failure.
bool page_pool_tensor_map(const void* base, int num_pages, int num_kv_heads, int head_dim,
                          CUtensorMap* out);

// Basic checks of a vg_paged_kv; VG_OK or an error status.
vg_status check_paged_kv(const vg_paged_kv* kv);

}  // namespace vg
