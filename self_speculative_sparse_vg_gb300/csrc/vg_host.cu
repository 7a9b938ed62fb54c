// Host-side helpers: status strings, device properties, TMA descriptors.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "vg_host.h"

namespace vg {

namespace {
constexpr uint64_t kDefaultWaitNs = 1000ull * 1000ull * 1000ull;  // 1 s
std::atomic<uint64_t> g_wait_report_ns{kDefaultWaitNs};
}  // namespace

uint64_t wait_report_ns() { return g_wait_report_ns.load(std::memory_order_relaxed); }

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapEntry {
  const void* base;
  int num_pages, num_kv_heads, head_dim, device;
  CUtensorMap map;
};

}  // namespace

bool page_pool_tensor_map(const void* base, int num_pages, int num_kv_heads, int head_dim,
                          CUtensorMap* out) {
  constexpr int kEntries = 16;
  static MapEntry cache[kEntries];
  static int next = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
      if (e.base == base && e.num_pages == num_pages && e.num_kv_heads == num_kv_heads &&
          e.head_dim == head_dim && e.device == dev) {
        *out = e.map;
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  CUtensorMap map;
  cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)kPageSize, (cuuint64_t)num_kv_heads,
                        (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)kPageSize * head_dim * 2,
                           (cuuint64_t)num_kv_heads * kPageSize * head_dim * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kPageSize, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = MapEntry{base, num_pages, num_kv_heads, head_dim, dev, map};
    next = (next + 1) % kEntries;
  }
  *out = map;
  return true;
}

vg_status check_paged_kv(const vg_paged_kv* kv) {
  if (!kv || !kv->k_pages || !kv->v_pages || !kv->page_table) return VG_ERR_INVALID_ARGUMENT;
  if (kv->num_pages <= 0 || kv->max_pages_per_seq <= 0 || kv->num_kv_heads <= 0)
    return VG_ERR_INVALID_ARGUMENT;
  if (kv->page_size != kPageSize) return VG_ERR_UNSUPPORTED;
  if (kv->head_dim != 64 && kv->head_dim != 128) return VG_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(kv->k_pages) & 15) || (reinterpret_cast<uintptr_t>(kv->v_pages) & 15))
    return VG_ERR_INVALID_ARGUMENT;
  return VG_OK;
}

}  // namespace vg

extern "C" const char* vg_status_string(vg_status s) {
  switch (s) {
    case VG_OK: return "VG_OK";
    case VG_ERR_INVALID_ARGUMENT: return "VG_ERR_INVALID_ARGUMENT";
    case VG_ERR_UNSUPPORTED: return "VG_ERR_UNSUPPORTED";
    case VG_ERR_WORKSPACE_TOO_SMALL: return "VG_ERR_WORKSPACE_TOO_SMALL";
    case VG_ERR_LAUNCH: return "VG_ERR_LAUNCH";
  }
  return "VG_ERR_UNKNOWN";
}

extern "C" const char* vg_version(void) { return "0.2.0"; }

extern "C" vg_status vg_set_wait_limit_ns(uint64_t limit_ns) {
  vg::g_wait_report_ns.store(limit_ns == 0 ? vg::kDefaultWaitNs : limit_ns,
                             std::memory_order_relaxed);
  return VG_OK;
}
