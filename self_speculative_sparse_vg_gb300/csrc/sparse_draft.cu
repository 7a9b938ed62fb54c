// Sparse draft attention over the selected KV entries plus the dense tail
// (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" and Figure 1: while drafting, each draft token attends only the
// KV entries picked from the previous verification; A Sparse Glimpse of the
// Whole, "What carries the argument": the dense cache is kept, the index is a
// view into it.
//
// Design: one thread-block cluster of C CTAs per (sequence, KV head).  The
// attended list (the selection, then the tail [tail_start, cur_len)) is cut
// into 64-entry chunks; CTA r of the cluster takes chunks r, r + C, ...
//  * The sequence's page-table row is staged in shared memory while the
//    selected positions are loaded, so resolving a row's address costs no
//    further global round trip.
//  * Every chunk's K and V rows are gathered with 16-byte cp.async straight
//    into the 128-byte-swizzled tile layout the verify kernel's TMA loads
//    produce (one commit group per chunk, up to kRing chunks in flight).
//  * The g query heads of the KV head are the rows of a 16-row bf16
//    mma.sync tile (zero padded); warp w takes positions [16w, 16w + 16) of
//    each chunk, keeps an online softmax, and reuses P as the A operand.
//  * The CTA's warps merge in shared memory; the cluster's C partials merge
//    through distributed shared memory, each CTA finishing a slice of the
//    outputs.  No global workspace, atomics or second launch.
#include <cooperative_groups.h>

#include <mutex>

#include "vg_device.cuh"
#include "vg_host.h"

namespace cg = cooperative_groups;

namespace vg {
namespace {

constexpr int kChunk = 64;        // attended entries per chunk
constexpr int kDraftWarps = 4;
constexpr int kDraftThreads = kDraftWarps * 32;
constexpr int kRing = 5;          // chunks in flight per CTA
constexpr int kMaxRounds = 8;     // chunks per CTA
constexpr int kMaxDraftCluster = 16;
constexpr int kPtMax = 8192;      // page-table entries staged in shared memory

struct DraftParams {
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int32_t* page_table;
  const __nv_bfloat16* q;
  const int32_t* indices;
  const int32_t* counts;
  const int32_t* tail_start;
  const int32_t* cur_len;
  __nv_bfloat16* out;
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq;
  int ring, rounds, pt_cap;  // chunks in flight, chunks per CTA, staged page-table entries
  float scale_log2;
};

template <int HD>
struct DraftLayout {
  static constexpr int kTileBytes = kChunk * HD * 2;  // one of K / V
  static constexpr int kChunkBytes = 2 * kTileBytes;
  static constexpr int kQBytes = 16 * HD * 2;
  // dynamic shared memory of a launch: ring, query rows, entry offsets, page ids
  static size_t bytes(int ring, int rounds, int pt_cap) {
    return 1024 + (size_t)ring * kChunkBytes + kQBytes + (size_t)rounds * kChunk * 8 +
           (size_t)pt_cap * 4;
  }
  static constexpr size_t kMaxBytes =
      1024 + (size_t)kRing * kChunkBytes + kQBytes + (size_t)kMaxRounds * kChunk * 8 + kPtMax * 4;
};

template <int N>
__device__ __forceinline__ void wait_pending(int n) {
  // cp.async.wait_group takes an immediate: dispatch on the run-time count
  if (n >= N) {
    cp_async_wait<N>();
  } else if constexpr (N > 0) {
    wait_pending<N - 1>(n);
  }
}

template <int HD>
__global__ void __launch_bounds__(kDraftThreads)
    sparse_draft_kernel(const DraftParams p) {
  using Lay = DraftLayout<HD>;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DN = HD / 8;   // O n-tiles
  constexpr int CH = HD / 8;   // 16-byte chunks per row

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;                                                // [ring][K, V]
  uint8_t* qs = ring + (size_t)p.ring * Lay::kChunkBytes;              // [16][HD] bf16
  long long* off_s = reinterpret_cast<long long*>(qs + Lay::kQBytes);  // [rounds * 64]
  int32_t* pt_s = reinterpret_cast<int32_t*>(off_s + (size_t)p.rounds * kChunk);
  __shared__ float m_s[8], l_s[8];
  __shared__ float wm_s[kDraftWarps][16], wl_s[kDraftWarps][16];
  __shared__ __align__(16) float part_s[8 * HD];

  const int cnt = p.counts[(size_t)b * rows + row];
  const int ts = p.tail_start[b];
  const int cl = p.cur_len[b];
  bool ok = true;
  if (cnt < 0 || cnt > p.cap) {
    if (tid == 0 && rank == 0) flag_error(p.error_flag, VG_DEVERR_COUNT);
    ok = false;
  }
  if (ts < 0 || cl < ts || cl - ts > p.max_tail || cl <= 0 ||
      (cl + kPageSize - 1) / kPageSize > p.max_pages_per_seq) {
    if (tid == 0 && rank == 0 && h == 0) flag_error(p.error_flag, VG_DEVERR_LENGTH);
    ok = false;
  }
  if (!ok) return;  // same decision in every CTA of the cluster, before any cluster barrier

  const int n_att = cnt + (cl - ts);
  const int nch = (n_att + kChunk - 1) / kChunk;
  const int nr = rank < nch ? (nch - rank + C - 1) / C : 0;  // my chunks (<= kMaxRounds)
  const int npages = (cl + kPageSize - 1) / kPageSize;
  const bool pt_in_smem = npages <= p.pt_cap;

  // (1) stage the page-table row (overlaps the index loads below)
  if (pt_in_smem && nr > 0) {
    const int32_t* src = p.page_table + (size_t)b * p.max_pages_per_seq;
    const bool aligned = ((reinterpret_cast<uintptr_t>(src) & 15) == 0);
    if (aligned) {
      for (int i = tid; i < (npages + 3) / 4; i += kDraftThreads) {
        if (4 * i + 3 < npages)
          cp_async_16(pt_s + 4 * i, src + 4 * i);
        else
          for (int k = 4 * i; k < npages; ++k) pt_s[k] = __ldg(src + k);
      }
    } else {
      for (int i = tid; i < npages; i += kDraftThreads) pt_s[i] = __ldg(src + i);
    }
  }
  cp_async_commit();
  // (2) the selected positions of my entries, in registers
  constexpr int kPer = (kMaxRounds * kChunk + kDraftThreads - 1) / kDraftThreads;
  int pos_r[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kDraftThreads;
    int pos = -1;
    if (i < nr * kChunk) {
      const int e = (rank + (i / kChunk) * C) * kChunk + (i % kChunk);
      if (e < cnt) {
        pos = __ldg(p.indices + ((size_t)b * rows + row) * p.cap + e);
        if (pos < 0 || pos >= ts) pos = -2;  // flagged below
      } else if (e < n_att) {
        pos = ts + (e - cnt);
      }
    }
    pos_r[u] = pos;
  }
  // (3) query rows -> shared, swizzled like a K tile, rows >= g zero
  for (int idx = tid; idx < 16 * CH; idx += kDraftThreads) {
    const int r = idx / CH, ch = idx - (idx / CH) * CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < g) v = *reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.num_q_heads + h * g + r) * HD + ch * 8);
    *reinterpret_cast<uint4*>(qs + sw128_offset(r, ch, 16)) = v;
  }
  cp_async_wait<0>();
  __syncthreads();
  // (4) resolve each entry's K/V row: element offset, or -1 (zero row, masked)
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * kDraftThreads;
    if (i < nr * kChunk) {
      const int pos = pos_r[u];
      long long off = -1;
      if (pos == -2) {
        flag_error(p.error_flag, VG_DEVERR_INDEX);
      } else if (pos >= 0) {
        const int phys = pt_in_smem ? pt_s[pos / kPageSize]
                                    : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
        if (phys >= 0 && phys < p.num_pages)
          off = (((long long)phys * p.num_kv_heads + h) * kPageSize + (pos % kPageSize)) * HD;
        else
          flag_error(p.error_flag, VG_DEVERR_PAGE);
      }
      off_s[i] = off;
    }
  }
  __syncthreads();

  // (5) gather: chunk r -> ring slot r % kRing, K then V, one commit group per chunk
  auto issue = [&](int r) {
    uint8_t* kt = ring + (r % p.ring) * Lay::kChunkBytes;
    uint8_t* vt = kt + Lay::kTileBytes;
    for (int idx = tid; idx < kChunk * CH; idx += kDraftThreads) {
      const int j = idx / CH, c = idx - (idx / CH) * CH;
      const long long off = off_s[r * kChunk + j];
      const uint32_t o = sw128_offset(j, c, kChunk);
      if (off >= 0) {
        cp_async_16(kt + o, p.k_pages + off + c * 8);
        cp_async_16(vt + o, p.v_pages + off + c * 8);
      } else {
        *reinterpret_cast<uint4*>(kt + o) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vt + o) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };
  int issued = 0;
  for (; issued < nr && issued < p.ring; ++issued) issue(issued);

  // (6) per-warp online softmax over positions [16 warp, 16 warp + 16) of each chunk
  const int r = lane >> 2, c = lane & 3;
  const uint32_t qs_u = smem_u32(qs);
  uint32_t qa[KS][4];
  {
    const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(qs_u + sw128_offset(qrow, 2 * ks + (lane >> 4), 16), qa[ks][0], qa[ks][1], qa[ks][2],
              qa[ks][3]);
  }
  float mrun0 = -INFINITY, mrun1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
  const int krow = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
  const int kchk = (lane >> 3) & 1;
  const int vrow = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int vchk = lane >> 4;
  const uint32_t ring_u = smem_u32(ring);

  for (int rr = 0; rr < nr; ++rr) {
    wait_pending<kRing>(issued - rr - 1);
    __syncthreads();
    const int ne = min(kChunk, n_att - (rank + rr * C) * kChunk);
    if (warp * 16 < ne) {  // warp-uniform
      const uint32_t kt = ring_u + (rr % p.ring) * Lay::kChunkBytes;
      const uint32_t vt = kt + Lay::kTileBytes;
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + sw128_offset(krow, 2 * ks + kchk, kChunk), b0, b1, b2, b3);
        mma_16816(s[0], qa[ks], b0, b1);
        mma_16816(s[1], qa[ks], b2, b3);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = warp * 16 + nt * 8 + 2 * c + e;
          const bool valid = j < ne && off_s[rr * kChunk + j] >= 0;
          s[nt][e] = valid ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][2 + e] = valid ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, s[nt][e]);
          mx1 = fmaxf(mx1, s[nt][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(mrun0, mx0), mn1 = fmaxf(mrun1, mx1);
      const float ref0 = safe_ref(mn0), ref1 = safe_ref(mn1);
      const float corr0 = ex2(mrun0 - ref0), corr1 = ex2(mrun1 - ref1);
      mrun0 = mn0;
      mrun1 = mn1;
      l0 *= corr0;
      l1 *= corr1;
#pragma unroll
      for (int dn = 0; dn < DN; ++dn) {
        acc[dn][0] *= corr0;
        acc[dn][1] *= corr0;
        acc[dn][2] *= corr1;
        acc[dn][3] *= corr1;
      }
      uint32_t pa[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p00 = ex2(s[nt][0] - ref0), p01 = ex2(s[nt][1] - ref0);
        const float p10 = ex2(s[nt][2] - ref1), p11 = ex2(s[nt][3] - ref1);
        l0 += p00 + p01;
        l1 += p10 + p11;
        pa[nt * 2 + 0] = pack_bf16(p00, p01);
        pa[nt * 2 + 1] = pack_bf16(p10, p11);
      }
#pragma unroll
      for (int dp = 0; dp < DN / 2; ++dp) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vt + sw128_offset(vrow, 2 * dp + vchk, kChunk), v0, v1, v2, v3);
        mma_16816(acc[2 * dp], pa, v0, v1);
        mma_16816(acc[2 * dp + 1], pa, v2, v3);
      }
    }
    __syncthreads();  // slot rr % ring is free again
    if (issued < nr) issue(issued++);
  }
  cp_async_wait<0>();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // (7) merge the warps: rows < g only (the query heads)
  float* sO = reinterpret_cast<float*>(ring);  // [warps][16][HD], the ring is idle now
  {
    float* o = sO + (size_t)warp * 16 * HD;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      const int col = dn * 8 + 2 * c;
      *reinterpret_cast<float2*>(&o[r * HD + col]) = make_float2(acc[dn][0], acc[dn][1]);
      *reinterpret_cast<float2*>(&o[(r + 8) * HD + col]) = make_float2(acc[dn][2], acc[dn][3]);
    }
    if (c == 0) {
      wm_s[warp][r] = mrun0;
      wl_s[warp][r] = l0;
      wm_s[warp][r + 8] = mrun1;
      wl_s[warp][r + 8] = l1;
    }
  }
  __syncthreads();
  if (tid < g) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w) mx = fmaxf(mx, wm_s[w][tid]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w) {
      const float wt = ex2(wm_s[w][tid] - ref);
      wm_s[w][tid] = wt;  // now the warp's weight
      lt += wt * wl_s[w][tid];
    }
    m_s[tid] = mx;
    l_s[tid] = lt;
  }
  __syncthreads();
  for (int i = tid; i < g * HD; i += kDraftThreads) {
    const int qi = i / HD, d = i - (i / HD) * HD;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w) o += wm_s[w][qi] * sO[((size_t)w * 16 + qi) * HD + d];
    part_s[i] = o;
  }
  cluster.sync();  // every CTA's (m, l, part) is visible cluster-wide

  // (8) merge the cluster: CTA `rank` finishes a slice of the g x HD outputs
  const int total = g * HD;
  const int per = (total + C - 1) / C;
  const int i_end = min(total, (rank + 1) * per);
  for (int i = rank * per + tid; i < i_end; i += kDraftThreads) {
    const int qi = i / HD;
    float mc[kMaxDraftCluster], lc[kMaxDraftCluster], oc[kMaxDraftCluster];
    float mx = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < kMaxDraftCluster; ++cc) {
      if (cc < C) {
        mc[cc] = cluster.map_shared_rank(m_s, cc)[qi];
        lc[cc] = cluster.map_shared_rank(l_s, cc)[qi];
        oc[cc] = cluster.map_shared_rank(part_s, cc)[i];
        mx = fmaxf(mx, mc[cc]);
      }
    }
    const float ref = safe_ref(mx);
    float lt = 0.f, o = 0.f;
#pragma unroll
    for (int cc = 0; cc < kMaxDraftCluster; ++cc) {
      if (cc < C) {
        const float w = ex2(mc[cc] - ref);
        lt += w * lc[cc];
        o += w * oc[cc];
      }
    }
    p.out[((size_t)b * p.num_q_heads + h * g) * HD + i] =
        __float2bfloat16_rn(lt > 0.f ? o / lt : 0.f);
  }
  cluster.sync();  // no CTA leaves while its shared memory may still be read
}

// Kernel attributes (max dynamic shared memory, 16-CTA clusters), once per device.
template <int HD>
cudaError_t launch_draft_attrs() {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && attr_done[dev]) return cudaSuccess;
  auto kern = sparse_draft_kernel<HD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DraftLayout<HD>::kMaxBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev < 64) attr_done[dev] = true;
  return cudaSuccess;
}

template <int HD>
cudaError_t launch_draft(const DraftParams& p, int cluster, cudaStream_t stream) {
  auto kern = sparse_draft_kernel<HD>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kDraftThreads, 1, 1);
  cfg.dynamicSmemBytes = DraftLayout<HD>::bytes(p.ring, p.rounds, p.pt_cap);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Cluster size: one CTA per 64-entry chunk, up to 16, but no larger than
// lets every (sequence, KV head) cluster of the launch be resident at once
// (a cluster must fit in one GPC, so only a few 16-CTA clusters can run at a
// time); else the launch would run in waves.
template <int HD>
int draft_cluster_size(int entries, int clusters_needed, const DraftParams& proto) {
  const int chunks = ceil_div(std::max(entries, 1), kChunk);
  int best = 0, fallback = kMaxDraftCluster;  // fallback: smallest size within kMaxRounds
  for (int c = std::min(kMaxDraftCluster, chunks); c >= 1; c = (c > 8 ? 8 : c / 2)) {
    if (ceil_div(chunks, c) <= kMaxRounds) fallback = c;
    DraftParams p = proto;
    p.rounds = ceil_div(chunks, c);
    p.ring = std::min(kRing, p.rounds);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3(kDraftThreads, 1, 1);
    cfg.dynamicSmemBytes = DraftLayout<HD>::bytes(p.ring, p.rounds, p.pt_cap);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (p.rounds <= kMaxRounds &&
        cudaOccupancyMaxActiveClusters(&n, sparse_draft_kernel<HD>, &cfg) == cudaSuccess &&
        n >= clusters_needed) {
      best = c;
      break;
    }
    cudaGetLastError();
    if (c == 1) break;
  }
  return best ? best : fallback;
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" size_t vg_sparse_draft_workspace_bytes(int, int, int, int, int, int) { return 0; }

extern "C" vg_status vg_sparse_draft_attention(const vg_paged_kv* kv, const void* q,
                                               const int32_t* indices, const int32_t* counts,
                                               int per_head, int cap, const int32_t* tail_start,
                                               const int32_t* cur_len, int batch, int num_q_heads,
                                               int max_tail, float softmax_scale, void* out,
                                               void* /*workspace*/, size_t /*workspace_bytes*/,
                                               int32_t* error_flag, cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (!q || !counts || !tail_start || !cur_len || !out || batch <= 0 || num_q_heads <= 0 ||
      cap < 0 || max_tail < 0 || cap + max_tail <= 0 || !(softmax_scale == softmax_scale))
    return VG_ERR_INVALID_ARGUMENT;
  if (cap > 0 && !indices) return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads % kv->num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / kv->num_kv_heads;
  if (g > 8) return VG_ERR_UNSUPPORTED;
  if (ceil_div(cap + max_tail, kChunk) > kMaxDraftCluster * kMaxRounds) return VG_ERR_UNSUPPORTED;
  DraftParams p;
  p.k_pages = static_cast<const __nv_bfloat16*>(kv->k_pages);
  p.v_pages = static_cast<const __nv_bfloat16*>(kv->v_pages);
  p.page_table = kv->page_table;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.indices = indices;
  p.counts = counts;
  p.tail_start = tail_start;
  p.cur_len = cur_len;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.error_flag = error_flag;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = kv->num_kv_heads;
  p.group = g;
  p.per_head = per_head ? 1 : 0;
  p.cap = cap;
  p.max_tail = max_tail;
  p.num_pages = kv->num_pages;
  p.max_pages_per_seq = kv->max_pages_per_seq;
  p.pt_cap = std::min(kPtMax, (kv->max_pages_per_seq + 3) / 4 * 4);
  p.scale_log2 = softmax_scale * kLog2e;
  // cluster size per (shape, device), cached: the occupancy query is not free
  struct Entry { int dev, hd, entries, clusters, pt_cap, C; };
  static Entry cache[32];
  static int n_cache = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  const int clusters = batch * kv->num_kv_heads;
  int C = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cache; ++i)
      if (cache[i].dev == dev && cache[i].hd == kv->head_dim && cache[i].entries == cap + max_tail &&
          cache[i].clusters == clusters && cache[i].pt_cap == p.pt_cap)
        C = cache[i].C;
  }
  if (C == 0) {
    if (kv->head_dim == 128 ? launch_draft_attrs<128>() : launch_draft_attrs<64>()) return VG_ERR_LAUNCH;
    C = kv->head_dim == 128 ? draft_cluster_size<128>(cap + max_tail, clusters, p)
                            : draft_cluster_size<64>(cap + max_tail, clusters, p);
    std::lock_guard<std::mutex> lock(mu);
    cache[n_cache % 32] = Entry{dev, kv->head_dim, cap + max_tail, clusters, p.pt_cap, C};
    ++n_cache;
  }
  p.rounds = ceil_div(ceil_div(cap + max_tail, kChunk), C);
  if (p.rounds > kMaxRounds) return VG_ERR_UNSUPPORTED;
  p.ring = std::min(kRing, p.rounds);
  const cudaError_t e = kv->head_dim == 128 ? launch_draft<128>(p, C, stream)
                                             : launch_draft<64>(p, C, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
