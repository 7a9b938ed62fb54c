// Sparse draft attention over the selected KV entries plus the dense tail
// (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" and Figure 1: while drafting, each draft token attends only the
// KV entries picked from the previous verification; A Sparse Glimpse of the
// Whole, "What carries the argument": the dense cache is kept, the index is a
// view into it.
//
// Design: one CTA per (chunk of the attended list, KV head, sequence).  The
// attended list is the selection followed by the tail [tail_start, cur_len).
// Each CTA resolves its entries' page addresses, gathers their K and V rows
// (16-byte cp.async, all in flight at once), computes the g query heads'
// logits with CUDA-core FMAs and shuffle reductions (one draft row is only
// ~4 flop/byte, far below the tensor-core break-even), a chunk softmax, and
// P.V.  Chunks are merged by the last CTA of each (sequence, KV head)
// (atomic ticket, no waiting).
#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kChunk = 64;        // attended entries per CTA
constexpr int kDraftThreads = 128;

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
  float* part_o;     // [B][Hkv][splits][g][HD]
  float* part_ml;    // [B][Hkv][splits][g][2]
  int32_t* tickets;  // [B][Hkv]
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq, splits;
  float scale_log2;
};

template <int HD, int GMAX>
__global__ void __launch_bounds__(kDraftThreads)
    sparse_draft_kernel(const DraftParams p) {
  constexpr int LPR = HD / 8;              // lanes per KV row (16 B each)
  constexpr int RPW = 32 / LPR;            // rows per warp step
  constexpr int NW = kDraftThreads / 32;
  constexpr int SLOTS = NW * RPW;          // row slots per CTA step

  __shared__ __align__(16) __nv_bfloat16 kv_s[2][kChunk][HD];   // K, V rows
  __shared__ long long off_s[kChunk];                          // element offset or -1
  __shared__ float logit_s[GMAX][kChunk];
  __shared__ float m_s[GMAX], l_s[GMAX];
  __shared__ int flag_s;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;

  int cnt = p.counts[(size_t)b * rows + row];
  const int ts = p.tail_start[b];
  const int cl = p.cur_len[b];
  bool ok = true;
  if (cnt < 0 || cnt > p.cap) {
    if (tid == 0 && split == 0) flag_error(p.error_flag, VG_DEVERR_COUNT);
    ok = false;
  }
  if (ts < 0 || cl < ts || cl - ts > p.max_tail || cl <= 0 ||
      (cl + kPageSize - 1) / kPageSize > p.max_pages_per_seq) {
    if (tid == 0 && split == 0 && h == 0) flag_error(p.error_flag, VG_DEVERR_LENGTH);
    ok = false;
  }
  if (!ok) return;  // uniform across the CTAs of this (b, h): no ticket taken

  const int n_att = cnt + (cl - ts);
  const int e0 = split * kChunk;
  const int ne = max(0, min(n_att - e0, kChunk));

  // resolve the entries' row addresses
  if (tid < ne) {
    const int e = e0 + tid;
    int pos;
    bool valid = true;
    if (e < cnt) {
      pos = p.indices[((size_t)b * rows + row) * p.cap + e];
      if (pos < 0 || pos >= ts) {
        flag_error(p.error_flag, VG_DEVERR_INDEX);
        valid = false;
      }
    } else {
      pos = ts + (e - cnt);
    }
    long long off = -1;
    if (valid) {
      const int phys = p.page_table[(size_t)b * p.max_pages_per_seq + pos / kPageSize];
      if (phys >= 0 && phys < p.num_pages)
        off = (((long long)phys * p.num_kv_heads + h) * kPageSize + (pos % kPageSize)) * HD;
      else
        flag_error(p.error_flag, VG_DEVERR_PAGE);
    }
    off_s[tid] = off;
  }
  // the g query vectors, this lane's 8-element chunk, in fp32
  const int ch = lane % LPR;
  float qr[GMAX][8];
#pragma unroll
  for (int qi = 0; qi < GMAX; ++qi) {
    if (qi < g) {
      const uint4 raw = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)b * p.num_q_heads + h * g + qi) * HD + ch * 8);
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(v2[t]);
        qr[qi][2 * t] = f.x;
        qr[qi][2 * t + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int t = 0; t < 8; ++t) qr[qi][t] = 0.f;
    }
  }
  __syncthreads();

  // gather: K rows (group 0), then V rows (group 1)
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const __nv_bfloat16* pool = kv ? p.v_pages : p.k_pages;
    for (int idx = tid; idx < ne * LPR; idx += kDraftThreads) {
      const int e = idx / LPR, c = idx - (idx / LPR) * LPR;
      const long long off = off_s[e];
      if (off >= 0)
        cp_async_16(&kv_s[kv][e][c * 8], pool + off + c * 8);
      else
        *reinterpret_cast<uint4*>(&kv_s[kv][e][c * 8]) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  }
  cp_async_wait<1>();
  __syncthreads();

  // logits: row slot = warp * RPW + lane / LPR.  The trip count is uniform
  // across the warp (rows past ne are predicated off) because the loop body
  // shuffles with a full mask.
  const int slot = warp * RPW + lane / LPR;
  for (int base = warp * RPW; base < ne; base += SLOTS) {
    const int e = base + lane / LPR;
    const bool ev = e < ne;
    const uint4 raw = ev ? *reinterpret_cast<const uint4*>(&kv_s[0][e][ch * 8])
                         : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float kf[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __bfloat1622float2(k2[t]);
      kf[2 * t] = f.x;
      kf[2 * t + 1] = f.y;
    }
    float dot[GMAX];
#pragma unroll
    for (int qi = 0; qi < GMAX; ++qi) {
      float a = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) a = fmaf(qr[qi][t], kf[t], a);
      dot[qi] = a;
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)
#pragma unroll
      for (int qi = 0; qi < GMAX; ++qi) dot[qi] += __shfl_xor_sync(0xffffffffu, dot[qi], o);
    if (ev && ch == 0) {
      const bool valid = off_s[e] >= 0;
#pragma unroll
      for (int qi = 0; qi < GMAX; ++qi)
        if (qi < g) logit_s[qi][e] = valid ? dot[qi] * p.scale_log2 : -INFINITY;
    }
  }
  __syncthreads();

  // chunk softmax per query head (base 2)
  for (int qi = warp; qi < g; qi += NW) {
    float mx = -INFINITY;
    for (int e = lane; e < ne; e += 32) mx = fmaxf(mx, logit_s[qi][e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ref = safe_ref(mx);
    float sum = 0.f;
    for (int e = lane; e < ne; e += 32) {
      const float pe = ex2(logit_s[qi][e] - ref);
      logit_s[qi][e] = pe;
      sum += pe;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      m_s[qi] = mx;
      l_s[qi] = sum;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // P V
  float acc[GMAX][8];
#pragma unroll
  for (int qi = 0; qi < GMAX; ++qi)
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[qi][t] = 0.f;
  for (int e = slot; e < ne; e += SLOTS) {
    const uint4 raw = *reinterpret_cast<const uint4*>(&kv_s[1][e][ch * 8]);
    const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float vf[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __bfloat1622float2(v2[t]);
      vf[2 * t] = f.x;
      vf[2 * t + 1] = f.y;
    }
#pragma unroll
    for (int qi = 0; qi < GMAX; ++qi) {
      if (qi < g) {
        const float pe = logit_s[qi][e];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[qi][t] = fmaf(pe, vf[t], acc[qi][t]);
      }
    }
  }
  // fold the warp's RPW row slots (lanes with the same chunk) together
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int qi = 0; qi < GMAX; ++qi)
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[qi][t] += __shfl_xor_sync(0xffffffffu, acc[qi][t], o);
  __syncthreads();  // kv_s is free: reuse it for the cross-warp reduction
  float* red = reinterpret_cast<float*>(&kv_s[0][0][0]);  // [NW][g][HD]
  if (lane < LPR) {
#pragma unroll
    for (int qi = 0; qi < GMAX; ++qi) {
      if (qi < g) {
        float4* dst = reinterpret_cast<float4*>(&red[((size_t)warp * g + qi) * HD + ch * 8]);
        dst[0] = make_float4(acc[qi][0], acc[qi][1], acc[qi][2], acc[qi][3]);
        dst[1] = make_float4(acc[qi][4], acc[qi][5], acc[qi][6], acc[qi][7]);
      }
    }
  }
  __syncthreads();

  const size_t bh = (size_t)b * p.num_kv_heads + h;
  if (p.splits == 1) {
    for (int i = tid; i < g * HD; i += kDraftThreads) {
      const int qi = i / HD, d = i - (i / HD) * HD;
      float o = 0.f;
      for (int s = 0; s < NW; ++s) o += red[((size_t)s * g + qi) * HD + d];
      const float l = l_s[qi];
      p.out[((size_t)b * p.num_q_heads + h * g + qi) * HD + d] =
          __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
    }
    return;
  }
  float* po = p.part_o + ((bh * p.splits + split) * g) * HD;
  float* pml = p.part_ml + (bh * p.splits + split) * g * 2;
  for (int i = tid; i < g * HD; i += kDraftThreads) {
    const int qi = i / HD, d = i - (i / HD) * HD;
    float o = 0.f;
    for (int s = 0; s < NW; ++s) o += red[((size_t)s * g + qi) * HD + d];
    po[i] = o;
  }
  if (tid < g) {
    pml[tid * 2] = m_s[tid];
    pml[tid * 2 + 1] = l_s[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) flag_s = (atomicAdd(&p.tickets[bh], 1) == p.splits - 1);
  __syncthreads();
  if (!flag_s) return;
  __threadfence();

  float* w_s = reinterpret_cast<float*>(&kv_s[0][0][0]);  // [splits][g] weights
  const float* mlb = p.part_ml + bh * p.splits * g * 2;
  for (int qi = warp; qi < g; qi += NW) {
    float mx = -INFINITY;
    for (int s = lane; s < p.splits; s += 32) mx = fmaxf(mx, __ldcg(&mlb[(s * g + qi) * 2]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ref = safe_ref(mx);
    float lt = 0.f;
    for (int s = lane; s < p.splits; s += 32) {
      const float w = ex2(__ldcg(&mlb[(s * g + qi) * 2]) - ref);
      w_s[s * g + qi] = w;
      lt += w * __ldcg(&mlb[(s * g + qi) * 2 + 1]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    for (int s = lane; s < p.splits; s += 32) w_s[s * g + qi] *= inv;
  }
  __syncthreads();
  const float* pob = p.part_o + bh * p.splits * g * HD;
  for (int i = tid; i < g * HD; i += kDraftThreads) {
    const int qi = i / HD;
    float o = 0.f;
    for (int s = 0; s < p.splits; ++s) o += w_s[s * g + qi] * __ldcg(&pob[(size_t)s * g * HD + i]);
    p.out[((size_t)b * p.num_q_heads + h * g) * HD + i] = __float2bfloat16_rn(o);
  }
  if (tid == 0) p.tickets[bh] = 0;
}

struct DraftPlan {
  int splits;
  size_t off_ml, off_tickets, ws_bytes;
};

bool make_draft_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int cap,
                     int max_tail, DraftPlan* pl) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || cap < 0 || max_tail < 0 ||
      cap + max_tail <= 0)
    return false;
  // a fixed chunk of the attended list per CTA: the split count is the chunk count
  pl->splits = ceil_div(cap + max_tail, kChunk);
  const int g = num_q_heads / num_kv_heads;
  const size_t o_bytes = (size_t)batch * num_kv_heads * pl->splits * g * head_dim * 4;
  const size_t ml_bytes = (size_t)batch * num_kv_heads * pl->splits * g * 2 * 4;
  pl->off_ml = align_up(o_bytes, 256);
  pl->off_tickets = pl->off_ml + align_up(ml_bytes, 256);
  pl->ws_bytes = pl->splits > 1 ? pl->off_tickets + align_up((size_t)batch * num_kv_heads * 4, 256)
                                : 0;
  return true;
}

template <int HD, int GMAX>
cudaError_t launch_draft(const DraftParams& p, dim3 grid, cudaStream_t stream) {
  sparse_draft_kernel<HD, GMAX><<<grid, kDraftThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" size_t vg_sparse_draft_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                                  int head_dim, int cap, int max_tail) {
  DraftPlan pl;
  if (!make_draft_plan(batch, num_q_heads, num_kv_heads, head_dim, cap, max_tail, &pl))
    return 0;
  return pl.ws_bytes;
}

extern "C" vg_status vg_sparse_draft_attention(const vg_paged_kv* kv, const void* q,
                                               const int32_t* indices, const int32_t* counts,
                                               int per_head, int cap, const int32_t* tail_start,
                                               const int32_t* cur_len, int batch, int num_q_heads,
                                               int max_tail, float softmax_scale, void* out,
                                               void* workspace,
                                               size_t workspace_bytes, int32_t* error_flag,
                                               cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (!q || !counts || !tail_start || !cur_len || !out || batch <= 0 || num_q_heads <= 0 ||
      cap < 0 || max_tail < 0 || cap + max_tail <= 0 ||
      !(softmax_scale == softmax_scale))
    return VG_ERR_INVALID_ARGUMENT;
  if (cap > 0 && !indices) return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads % kv->num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / kv->num_kv_heads;
  if (g > 8) return VG_ERR_UNSUPPORTED;
  DraftPlan pl;
  if (!make_draft_plan(batch, num_q_heads, kv->num_kv_heads, kv->head_dim, cap, max_tail, &pl))
    return VG_ERR_INVALID_ARGUMENT;
  // the split merge keeps splits x g weights in the CTA's reused K/V buffer
  if ((size_t)pl.splits * g > (size_t)kChunk * kv->head_dim) return VG_ERR_UNSUPPORTED;
  if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes))
    return VG_ERR_WORKSPACE_TOO_SMALL;
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
  p.part_o = pl.ws_bytes ? reinterpret_cast<float*>(ws) : nullptr;
  p.part_ml = pl.ws_bytes ? reinterpret_cast<float*>(ws + pl.off_ml) : nullptr;
  p.tickets = pl.ws_bytes ? reinterpret_cast<int32_t*>(ws + pl.off_tickets) : nullptr;
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
  p.splits = pl.splits;
  p.scale_log2 = softmax_scale * kLog2e;
  dim3 grid(pl.splits, kv->num_kv_heads, batch);
  cudaError_t e;
  const int gm = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
  if (kv->head_dim == 128) {
    switch (gm) {
      case 1: e = launch_draft<128, 1>(p, grid, stream); break;
      case 2: e = launch_draft<128, 2>(p, grid, stream); break;
      case 4: e = launch_draft<128, 4>(p, grid, stream); break;
      default: e = launch_draft<128, 8>(p, grid, stream); break;
    }
  } else {
    switch (gm) {
      case 1: e = launch_draft<64, 1>(p, grid, stream); break;
      case 2: e = launch_draft<64, 2>(p, grid, stream); break;
      case 4: e = launch_draft<64, 4>(p, grid, stream); break;
      default: e = launch_draft<64, 8>(p, grid, stream); break;
    }
  }
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
