// Sparse draft attention over the selected KV entries plus the dense tail
// (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" and Figure 1: while drafting, each draft token attends only the
// KV entries picked from the previous verification; A Sparse Glimpse of the
// Whole, "What carries the argument": the dense cache is kept, the index is a
// view into it.
//
// Design: one CTA per 64-entry chunk of the attended list (the selection,
// then the tail [tail_start, cur_len)), per (KV head, sequence); all chunks of
// a step are resident at once.
//  * The chunk's selected positions, the sequence's page-table row (one bulk
//    copy into shared memory when short), the query rows and the lengths are
//    loaded together, so a row's address costs one round trip.
//  * The chunk's K and V rows (256 bytes each at head_dim 128) are then
//    gathered with 16-byte cp.async pieces, consecutive threads on
//    consecutive pieces of a row, into a row-padded tile (row stride
//    head_dim * 2 + 16 bytes, so ldmatrix rows fall in distinct bank groups).
//  * The g query heads of the KV head are the rows of a 16-row bf16
//    mma.sync tile (zero padded); warp w takes positions [16w, 16w + 16),
//    and P is reused as the A operand of P.V.
//  * Each CTA writes an fp32 partial (m, l, O) to the workspace; a small
//    merge kernel, chained with programmatic dependent launch, combines the
//    chunks of each (sequence, KV head, query head).
#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kChunk = 64;  // attended entries per CTA
constexpr int kDraftWarps = 4;
constexpr int kDraftThreads = kDraftWarps * 32;
constexpr int kPtMax = 2048;  // page-table entries staged in shared memory (8 KB)
constexpr int kMaxChunks = 1024;

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
  float* part_o;   // [B][Hkv][chunks][g][HD]
  float* part_ml;  // [B][Hkv][chunks][g][2]
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq, chunks, pt_cap;
  float scale_log2;
};

template <int HD>
struct DraftLayout {
  static constexpr int kRowBytes = HD * 2 + 16;             // padded K / V / Q row
  static constexpr int kTileBytes = kChunk * kRowBytes;     // one of K / V
  static constexpr int kQBytes = 16 * kRowBytes;
  static constexpr int kOStride = 2 * 32 + 8;               // floats per (warp, n-tile) stash
  static constexpr size_t kBytes = 1024 + 2 * (size_t)kTileBytes + kQBytes + (size_t)kPtMax * 4 + 64;
  static_assert((size_t)kDraftWarps * (HD / 8) * kOStride * 4 <= 2 * (size_t)kTileBytes,
                "the O stash reuses the K/V tiles");
};

// Sequence-level checks shared by both kernels; false if the sequence is skipped.
__device__ __forceinline__ bool draft_lengths(const DraftParams& p, int b, int row, int rows,
                                              int* cnt, int* ts, int* cl) {
  *cnt = p.counts[(size_t)b * rows + row];
  *ts = p.tail_start[b];
  *cl = p.cur_len[b];
  if (*cnt < 0 || *cnt > p.cap) return false;
  if (*ts < 0 || *cl < *ts || *cl - *ts > p.max_tail || *cl <= 0 ||
      (*cl + kPageSize - 1) / kPageSize > p.max_pages_per_seq)
    return false;
  return true;
}

template <int HD>
__global__ void __launch_bounds__(kDraftThreads)
    sparse_draft_kernel(const DraftParams p) {
  using Lay = DraftLayout<HD>;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DN = HD / 8;   // O n-tiles
  constexpr int CH = HD / 8;   // 16-byte chunks per row

  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;
  // programmatic dependent launch: indices and counts come from the previous
  // kernel; the merge kernel may launch as soon as this grid has started
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int RB = Lay::kRowBytes;
  uint8_t* kt = smem;  // [64][RB]
  uint8_t* vt = kt + Lay::kTileBytes;
  uint8_t* qs = vt + Lay::kTileBytes;  // [16][RB]
  int32_t* pt_s = reinterpret_cast<int32_t*>(qs + Lay::kQBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pt_s + kPtMax);  // [0] page table
  __shared__ long long off_s[kChunk];
  __shared__ float wm_s[kDraftWarps][16], wl_s[kDraftWarps][16];

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // One round trip for everything the addresses depend on: this chunk's
  // selected positions (read speculatively; the index array holds cap
  // entries), the page-table row (one bulk copy when it is short), the
  // query rows and the lengths.
  const int e = chunk * kChunk + tid;
  int pos_sel = -1;
  if (tid < kChunk && e < p.cap) pos_sel = __ldg(p.indices + ((size_t)b * rows + row) * p.cap + e);
  const bool pt_in_smem = p.max_pages_per_seq <= p.pt_cap;
  if (pt_in_smem) {
    const int32_t* src = p.page_table + (size_t)b * p.max_pages_per_seq;
    const int n = p.max_pages_per_seq;
    const bool aligned = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    const int nb = aligned ? (n / 4) * 4 : 0;  // entries in the bulk copy (whole 16 bytes)
    if (tid == 0) {
      if (nb > 0) {
        mbar_arrive_expect_tx(&bars[0], nb * 4);
        bulk_load(pt_s, src, nb * 4, &bars[0]);
      } else {
        mbar_arrive(&bars[0]);
      }
    }
    for (int k = nb + tid; k < n; k += kDraftThreads) pt_s[k] = __ldg(src + k);
  } else if (tid == 0) {
    mbar_arrive(&bars[0]);
  }
  for (int idx = tid; idx < 16 * CH; idx += kDraftThreads) {  // query rows; rows >= g zero
    const int r = idx / CH, ch = idx - (idx / CH) * CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < g)
      v = *reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.num_q_heads + h * g + r) * HD + ch * 8);
    *reinterpret_cast<uint4*>(qs + r * RB + ch * 16) = v;
  }
  int cnt, ts, cl;
  const bool lengths_ok = draft_lengths(p, b, row, rows, &cnt, &ts, &cl);
  // the page-table copy must land before anything reads it or the CTA leaves
  if (!mbar_wait(&bars[0], 0)) flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
  if (!lengths_ok) {
    if (tid == 0 && chunk == 0)
      flag_error(p.error_flag, cnt < 0 || cnt > p.cap ? VG_DEVERR_COUNT : VG_DEVERR_LENGTH);
    return;
  }
  const int n_att = cnt + (cl - ts);
  const int ne = min(kChunk, n_att - chunk * kChunk);
  if (ne <= 0) return;  // past the end of this list: no partial
  __syncthreads();

  // resolve each entry's K/V row and issue its two bulk copies; rows without
  // an entry (past the list, bad index or page) are zero and masked below
  if (tid < kChunk) {
    long long off = -1;
    if (tid < ne) {
      int pos = -1;
      if (e < cnt) {
        pos = pos_sel;
        if (pos < 0 || pos >= ts) {
          flag_error(p.error_flag, VG_DEVERR_INDEX);
          pos = -1;
        }
      } else {
        pos = ts + (e - cnt);
      }
      if (pos >= 0) {
        const int phys =
            pt_in_smem ? pt_s[pos / kPageSize]
                       : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
        if (phys >= 0 && phys < p.num_pages)
          off = (((long long)phys * p.num_kv_heads + h) * kPageSize + (pos % kPageSize)) * HD;
        else
          flag_error(p.error_flag, VG_DEVERR_PAGE);
      }
    }
    off_s[tid] = off;
    if (off < 0) {
      uint8_t* kd = kt + tid * RB;
      uint8_t* vd = vt + tid * RB;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        *reinterpret_cast<uint4*>(kd + c * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vd + c * 16) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();  // every row's offset is known
  // gather: 16-byte cp.async pieces, consecutive threads on consecutive
  // pieces of a row (K rows, then V rows), all in flight at once
#pragma unroll 4
  for (int idx = tid; idx < 2 * kChunk * CH; idx += kDraftThreads) {
    const int t = idx / (kChunk * CH);
    const int rem = idx - t * (kChunk * CH);
    const int rr = rem / CH, ch = rem - rr * CH;
    const long long off = off_s[rr];
    if (off >= 0)
      cp_async_16((t ? vt : kt) + rr * RB + ch * 16, (t ? p.v_pages : p.k_pages) + off + ch * 8);
  }
  cp_async_commit();
  // Q fragments while the rows are in flight
  const uint32_t qs_u = smem_u32(qs);
  uint32_t qa[KS][4];
  {
    const int qrow = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(qs_u + qrow * RB + (2 * ks + (lane >> 4)) * 16, qa[ks][0], qa[ks][1], qa[ks][2],
              qa[ks][3]);
  }
  cp_async_wait<0>();
  __syncthreads();  // every thread's pieces have landed

  // warp w: positions [16w, 16w + 16) of the chunk
  const int r = lane >> 2, c = lane & 3;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
  if (warp * 16 < ne) {  // warp-uniform
    const uint32_t ku = smem_u32(kt), vu = smem_u32(vt);
    const int krow = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
    const int vrow = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(ku + krow * RB + (2 * ks + ((lane >> 3) & 1)) * 16, b0, b1, b2, b3);
      mma_16816(s[0], qa[ks], b0, b1);
      mma_16816(s[1], qa[ks], b2, b3);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = warp * 16 + nt * 8 + 2 * c + k;
        const bool valid = j < ne && off_s[j] >= 0;
        s[nt][k] = valid ? s[nt][k] * p.scale_log2 : -INFINITY;
        s[nt][2 + k] = valid ? s[nt][2 + k] * p.scale_log2 : -INFINITY;
        m0 = fmaxf(m0, s[nt][k]);
        m1 = fmaxf(m1, s[nt][2 + k]);
      }
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    const float ref0 = safe_ref(m0), ref1 = safe_ref(m1);
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
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int dp = 0; dp < DN / 2; ++dp) {
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vu + vrow * RB + (2 * dp + (lane >> 4)) * 16, v0, v1, v2, v3);
      mma_16816(acc[2 * dp], pa, v0, v1);
      mma_16816(acc[2 * dp + 1], pa, v2, v3);
    }
  }
  __syncthreads();  // K/V tiles are free: reuse them for the warp merge
  // O stash in the accumulator's own layout, rows 0..7 only (g <= 8):
  // (warp, n-tile dn, lane) -> 2 floats, rows r = lane / 4, columns
  // 8 dn + 2 (lane % 4) + {0, 1}; n-tiles padded to kOStride floats
  constexpr int OS = Lay::kOStride;
  float* sO = reinterpret_cast<float*>(kt);
  {
#pragma unroll
    for (int dn = 0; dn < DN; ++dn)
      *reinterpret_cast<float2*>(&sO[(warp * DN + dn) * OS + lane * 2]) =
          make_float2(acc[dn][0], acc[dn][1]);
    if (c == 0) {
      wm_s[warp][r] = m0;
      wl_s[warp][r] = l0;
      wm_s[warp][r + 8] = m1;
      wl_s[warp][r + 8] = l1;
    }
  }
  __syncthreads();
  // chunk partial: m, l and the unnormalised O relative to m, per query head
  const size_t slot = (((size_t)b * p.num_kv_heads + h) * p.chunks + chunk) * g;
  if (tid < g) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w) mx = fmaxf(mx, wm_s[w][tid]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w) {
      const float wt = ex2(wm_s[w][tid] - ref);
      wm_s[w][tid] = wt;  // the warp's weight from here on
      lt += wt * wl_s[w][tid];
    }
    p.part_ml[(slot + tid) * 2] = mx;
    p.part_ml[(slot + tid) * 2 + 1] = lt;
  }
  __syncthreads();
  for (int i = tid; i < g * HD; i += kDraftThreads) {
    const int qi = i / HD, d = i - (i / HD) * HD;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kDraftWarps; ++w)
      o += wm_s[w][qi] * sO[(w * DN + (d >> 3)) * OS + (qi * 4 + ((d & 7) >> 1)) * 2 + (d & 1)];
    p.part_o[slot * HD + i] = o;
  }
}

// Chunk merge: one CTA per (query head, KV head, sequence); chained with
// programmatic dependent launch.
template <int HD>
__global__ void __launch_bounds__(kMergeThreads) sparse_draft_merge_kernel(const DraftParams p) {
  __shared__ __align__(16) float smem_f[kMergeSmemFloats];
  const int qi = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = p.group;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  int cnt, ts, cl;
  if (!draft_lengths(p, b, row, rows, &cnt, &ts, &cl)) return;
  const int nch = (cnt + (cl - ts) + kChunk - 1) / kChunk;
  const size_t base = ((size_t)b * p.num_kv_heads + h) * p.chunks;
  merge_splits<HD>(p.part_o + (base * g + qi) * HD, (size_t)g * HD, p.part_ml + (base * g + qi) * 2,
                   (size_t)g * 2, nch, p.out + ((size_t)b * p.num_q_heads + h * g + qi) * HD, smem_f);
}

struct DraftPlan {
  int chunks;
  size_t off_ml, ws_bytes;
};

bool make_draft_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int cap,
                     int max_tail, DraftPlan* pl) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || cap < 0 || max_tail < 0 ||
      cap + max_tail <= 0 || num_q_heads % num_kv_heads)
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->chunks = ceil_div(cap + max_tail, kChunk);
  const size_t o_bytes = (size_t)batch * num_kv_heads * pl->chunks * g * head_dim * 4;
  const size_t ml_bytes = (size_t)batch * num_kv_heads * pl->chunks * g * 2 * 4;
  pl->off_ml = align_up(o_bytes, 256);
  pl->ws_bytes = pl->off_ml + align_up(ml_bytes, 256);
  return true;
}

template <int HD>
cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(sparse_draft_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)DraftLayout<HD>::kBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(p.chunks, p.num_kv_heads, p.batch);
  ccfg.blockDim = dim3(kDraftThreads, 1, 1);
  ccfg.dynamicSmemBytes = DraftLayout<HD>::kBytes;
  ccfg.stream = stream;
  ccfg.attrs = pdl;
  ccfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&ccfg, sparse_draft_kernel<HD>, p);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.group, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_draft_merge_kernel<HD>, p);
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" size_t vg_sparse_draft_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                                  int head_dim, int cap, int max_tail) {
  DraftPlan pl;
  if (!make_draft_plan(batch, num_q_heads, num_kv_heads, head_dim, cap, max_tail, &pl)) return 0;
  return pl.ws_bytes;
}

extern "C" vg_status vg_sparse_draft_attention(const vg_paged_kv* kv, const void* q,
                                               const int32_t* indices, const int32_t* counts,
                                               int per_head, int cap, const int32_t* tail_start,
                                               const int32_t* cur_len, int batch, int num_q_heads,
                                               int max_tail, float softmax_scale, void* out,
                                               void* workspace, size_t workspace_bytes,
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
  DraftPlan pl;
  if (!make_draft_plan(batch, num_q_heads, kv->num_kv_heads, kv->head_dim, cap, max_tail, &pl))
    return VG_ERR_INVALID_ARGUMENT;
  if (pl.chunks > kMaxChunks) return VG_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < pl.ws_bytes) return VG_ERR_WORKSPACE_TOO_SMALL;
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
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float*>(ws + pl.off_ml);
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
  p.chunks = pl.chunks;
  p.pt_cap = kPtMax;
  p.scale_log2 = softmax_scale * kLog2e;
  const cudaError_t e = kv->head_dim == 128 ? launch_draft<128>(p, stream)
                                             : launch_draft<64>(p, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
