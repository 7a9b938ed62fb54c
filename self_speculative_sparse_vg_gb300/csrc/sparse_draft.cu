// Sparse draft attention over the selected KV entries plus the dense tail
// (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" and Figure 1: while drafting, each draft token attends only the
// KV entries picked from the previous verification; A Sparse Glimpse of the
// Whole, "What carries the argument": the dense cache is kept, the index is a
// view into it.
//
// Design: one kernel per draft step.  One CTA per CH-entry chunk of the
// attended list (the selection, then the tail [tail_start, cur_len)), per
// (KV head, sequence); all chunks of a step are resident at once.
//  * Addresses cost one round trip.  With the cache slots the selector wrote
//    beside the positions (physical page * 16 + offset, translated once per
//    selection), a chunk loads its slots, its positions (checked against the
//    prefix), the query rows and the lengths together.  Without slots the
//    sequence's page-table row is staged in shared memory in the same round
//    trip (one bulk copy when it is short).  Only the few tail entries look
//    their page up after the lengths are known.
//  * The chunk's K and V rows (256 bytes each at head_dim 128) are gathered
//    with 16-byte cp.async pieces, consecutive threads on consecutive pieces
//    of a row, into row-padded tiles (row stride head_dim * 2 + 16 bytes, so
//    ldmatrix rows fall in distinct bank groups).
//  * The g query heads of the KV head are the rows of a 16-row bf16 mma.sync
//    tile (zero padded); warp w takes positions [16w, 16w + 16), and P is
//    reused as the A operand of P.V.
//  * A list of one chunk writes the output directly.  Otherwise each CTA
//    writes an fp32 record (m, l, unnormalised O per query head) to the
//    workspace and takes a ticket from a per-(sequence, KV head) counter; the
//    CTA that draws the last ticket merges every record by log-sum-exp,
//    writes the output and puts the counter back to zero.  No CTA waits for
//    another and no second kernel is launched.
#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kChunk = 128;          // attended entries per CTA
constexpr int kMaxEntries = 65536;   // cap + max_tail
constexpr int kPtMax = 2048;         // page-table entries staged in shared memory (no slots)
constexpr int kRecHead = 16;         // floats before O in a chunk record: m[8], l[8]

struct DraftParams {
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int32_t* page_table;
  const __nv_bfloat16* q;
  const int32_t* indices;
  const int32_t* slots;    // NULL: translate positions through the page table
  const int32_t* counts;
  const int32_t* tail_start;
  const int32_t* cur_len;
  __nv_bfloat16* out;
  float* records;          // [B][Hkv][chunks][rec_floats]
  int32_t* tickets;        // [B][Hkv], zero between calls
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq, chunks, rec_floats;
  float scale_log2;
};

template <int HD, int CH>
struct DraftLayout {
  static constexpr int kWarps = CH / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowBytes = HD * 2 + 16;             // padded K / V / Q row
  static constexpr int kTileBytes = CH * kRowBytes;         // one of K / V
  static constexpr int kQBytes = 16 * kRowBytes;
  static constexpr int kOStride = 2 * 32 + 8;               // floats per (warp, n-tile) stash
  static constexpr int kMergeBytes = 2 * kTileBytes;        // K/V tiles, reused by the merge
  static constexpr size_t bytes(bool slots) {
    return 128 + (size_t)kMergeBytes + kQBytes + (slots ? 0 : (size_t)kPtMax * 4) + 64;
  }
  static_assert((size_t)kWarps * (HD / 8) * kOStride * 4 <= (size_t)kMergeBytes,
                "the O stash reuses the K/V tiles");
};

// Sequence-level checks; false if the sequence is skipped.
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

// Log-sum-exp merge of the nch chunk records of one (sequence, KV head) by
// the CTA that drew the last ticket.  Records are staged through shared
// memory a batch at a time (every load of a batch in flight together); warp
// w forms the batch weights of query heads w, w + NW, ...; thread t then
// accumulates float4 column (t mod HD/4) of head t / (HD/4), and more items
// when there are fewer threads than g * HD / 4.
template <int HD, int NT>
__device__ __forceinline__ void merge_records(const DraftParams& p, const float* src, int nch,
                                              __nv_bfloat16* dst, uint8_t* area, int area_bytes,
                                              float* mrun_s, float* lrun_s, float* corr_s) {
  constexpr int C4 = HD / 4;
  constexpr int NW = NT / 32;
  constexpr int IPT = (8 * C4 + NT - 1) / NT;  // items per thread at g = 8
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group, RF = p.rec_floats;
  const int cpb = (area_bytes - 64) / (RF * 4 + 32);  // chunks per batch (w_s: 8 floats each)
  float* recs = reinterpret_cast<float*>(area);
  float* w_s = recs + (size_t)cpb * RF;
  if (tid < 8) {
    mrun_s[tid] = -INFINITY;
    lrun_s[tid] = 0.f;
  }
  float4 acc[IPT];
#pragma unroll
  for (int i = 0; i < IPT; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += cpb) {
    const int nb = min(cpb, nch - c0);
    const int n4 = nb * RF / 4;
    const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)c0 * RF);
    float4* d4 = reinterpret_cast<float4*>(recs);
    for (int base = 0; base < n4; base += NT * 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = base + k * NT + tid;
        v[k] = i < n4 ? __ldcg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = base + k * NT + tid;
        if (i < n4) d4[i] = v[k];
      }
    }
    __syncthreads();
    for (int qi = warp; qi < g; qi += NW) {
      float mb = -INFINITY;
      for (int c = lane; c < nb; c += 32) mb = fmaxf(mb, recs[(size_t)c * RF + qi]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_old = mrun_s[qi];
      const float m_new = fmaxf(m_old, mb);
      const float ref = safe_ref(m_new);
      float lb = 0.f;
      for (int c = lane; c < nb; c += 32) {
        const float w = ex2(recs[(size_t)c * RF + qi] - ref);  // 0 for an empty chunk
        w_s[c * 8 + qi] = w;
        lb += w * recs[(size_t)c * RF + 8 + qi];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, o);
      if (lane == 0) {
        const float corr = ex2(m_old - ref);  // 0 while nothing was accumulated
        corr_s[qi] = corr;
        mrun_s[qi] = m_new;
        lrun_s[qi] = lrun_s[qi] * corr + lb;
      }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < IPT; ++it) {
      const int i = tid + it * NT;
      if (i < g * C4) {
        const int qi = i / C4, col = i - (i / C4) * C4;
        const float corr = corr_s[qi];
        float4 a = acc[it];
        a.x *= corr;
        a.y *= corr;
        a.z *= corr;
        a.w *= corr;
        for (int c = 0; c < nb; ++c) {
          const float w = w_s[c * 8 + qi];
          const float4 o =
              *reinterpret_cast<const float4*>(recs + (size_t)c * RF + kRecHead + qi * HD + col * 4);
          a.x += w * o.x;
          a.y += w * o.y;
          a.z += w * o.z;
          a.w += w * o.w;
        }
        acc[it] = a;
      }
    }
    __syncthreads();  // the staging area is rewritten by the next batch
  }
#pragma unroll
  for (int it = 0; it < IPT; ++it) {
    const int i = tid + it * NT;
    if (i < g * C4) {
      const int qi = i / C4, col = i - (i / C4) * C4;
      const float lt = lrun_s[qi];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float4 a = acc[it];
      uint2 w;
      w.x = pack_bf16(a.x * inv, a.y * inv);
      w.y = pack_bf16(a.z * inv, a.w * inv);
      *reinterpret_cast<uint2*>(dst + (size_t)qi * HD + col * 4) = w;
    }
  }
}

template <int HD, int CH, bool SLOTS>
__global__ void __launch_bounds__(DraftLayout<HD, CH>::kThreads, 2)
    sparse_draft_kernel(const DraftParams p) {
  using Lay = DraftLayout<HD, CH>;
  constexpr int NT = Lay::kThreads, NW = Lay::kWarps;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DN = HD / 8;   // O n-tiles
  constexpr int PC = HD / 8;   // 16-byte pieces per row
  constexpr int RB = Lay::kRowBytes;

  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;
  // programmatic dependent launch: indices, slots and counts come from the
  // previous kernel; the next kernel may launch as soon as this grid runs
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  uint8_t* kt = smem;  // [CH][RB]
  uint8_t* vt = kt + Lay::kTileBytes;
  uint8_t* qs = vt + Lay::kTileBytes;  // [16][RB]
  int32_t* pt_s = reinterpret_cast<int32_t*>(qs + Lay::kQBytes);  // no slots: page-table row
  uint64_t* bars = reinterpret_cast<uint64_t*>(pt_s + (SLOTS ? 0 : kPtMax));
  __shared__ long long off_s[CH];
  __shared__ float wm_s[NW][16], wl_s[NW][16];
  __shared__ float mrun_s[8], lrun_s[8], corr_s[8];
  __shared__ int last_s;

  if (!SLOTS) {
    if (tid == 0) {
      mbar_init(&bars[0], 1);
      fence_barrier_init();
    }
    __syncthreads();
  }

  // One round trip for everything the addresses depend on: this chunk's
  // selected positions and slots (read speculatively; the arrays hold cap
  // entries), the query rows and the lengths (and, without slots, the
  // page-table row).
  const int e = chunk * CH + tid;
  const size_t lrow = ((size_t)b * rows + row) * p.cap;
  int pos_sel = -1, slot_sel = -1;
  if (tid < CH && e < p.cap) {
    pos_sel = __ldg(p.indices + lrow + e);
    if (SLOTS) slot_sel = __ldg(p.slots + lrow + e);
  }
  const bool pt_in_smem = !SLOTS && p.max_pages_per_seq <= kPtMax;
  if (!SLOTS) {
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
      for (int k = nb + tid; k < n; k += NT) pt_s[k] = __ldg(src + k);
    } else if (tid == 0) {
      mbar_arrive(&bars[0]);
    }
  }
  for (int idx = tid; idx < 16 * PC; idx += NT) {  // query rows; rows >= g zero
    const int r = idx / PC, ch = idx - (idx / PC) * PC;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < g)
      v = *reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.num_q_heads + h * g + r) * HD + ch * 8);
    *reinterpret_cast<uint4*>(qs + r * RB + ch * 16) = v;
  }
  int cnt, ts, cl;
  const bool lengths_ok = draft_lengths(p, b, row, rows, &cnt, &ts, &cl);
  if (!SLOTS) {
    // the page-table copy must land before anything reads it or the CTA
    // leaves; a wait that gives up is reported and waited out once more
    if (!mbar_wait(&bars[0], 0)) {
      flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
      mbar_wait(&bars[0], 0);
    }
  }
  __nv_bfloat16* out_bh = p.out + ((size_t)b * p.num_q_heads + h * g) * HD;
  if (!lengths_ok) {
    if (tid == 0 && chunk == 0)
      flag_error(p.error_flag, cnt < 0 || cnt > p.cap ? VG_DEVERR_COUNT : VG_DEVERR_LENGTH);
    return;
  }
  const int n_att = cnt + (cl - ts);
  const int nch = (n_att + CH - 1) / CH;
  if (n_att == 0) {  // nothing attended: the output is zero
    if (chunk == 0)
      for (int i = tid; i < g * HD / 2; i += NT)
        reinterpret_cast<uint32_t*>(out_bh)[i] = 0u;
    return;
  }
  const int ne = min(CH, n_att - chunk * CH);
  if (ne <= 0) return;  // past the end of this list: no record, no ticket
  __syncthreads();      // the page-table entries other threads copied are visible

  // resolve each entry's K/V row; rows without an entry (past the list, bad
  // index, slot or page) are zero and masked below
  if (tid < CH) {
    long long off = -1;
    if (tid < ne) {
      int phys = -1, sl = 0;
      if (e < cnt) {
        const int pos = pos_sel;
        // a slot must address the position's own offset within its page
        const bool ok = pos >= 0 && pos < ts &&
                        !(SLOTS && slot_sel >= 0 && (slot_sel & 15) != (pos & 15));
        if (!ok) {
          flag_error(p.error_flag, VG_DEVERR_INDEX);
        } else {
          if (SLOTS) {
            phys = slot_sel < 0 ? -1 : slot_sel >> 4;
            sl = slot_sel & 15;
          } else {
            phys = pt_in_smem
                       ? pt_s[pos / kPageSize]
                       : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
            sl = pos % kPageSize;
          }
          if (phys < 0 || phys >= p.num_pages) flag_error(p.error_flag, VG_DEVERR_PAGE);
        }
      } else {
        const int pos = ts + (e - cnt);  // tail: its page is looked up now
        phys = pt_in_smem ? pt_s[pos / kPageSize]
                          : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
        sl = pos % kPageSize;
        if (phys < 0 || phys >= p.num_pages) flag_error(p.error_flag, VG_DEVERR_PAGE);
      }
      if (phys >= 0 && phys < p.num_pages)
        off = (((long long)phys * p.num_kv_heads + h) * kPageSize + sl) * HD;
    }
    off_s[tid] = off;
    if (off < 0) {
      uint8_t* kd = kt + tid * RB;
      uint8_t* vd = vt + tid * RB;
#pragma unroll
      for (int c = 0; c < PC; ++c) {
        *reinterpret_cast<uint4*>(kd + c * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vd + c * 16) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();  // every row's offset is known, the query rows are staged
  // gather: 16-byte cp.async pieces, consecutive threads on consecutive
  // pieces of a row (K rows, then V rows), all in flight at once
  const int nrow = ((ne + 15) / 16) * 16;  // rows the warps read (zero past ne)
#pragma unroll 4
  for (int idx = tid; idx < 2 * nrow * PC; idx += NT) {
    const int t = idx / (nrow * PC);
    const int rem = idx - t * (nrow * PC);
    const int rr = rem / PC, ch = rem - rr * PC;
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
  // chunk result per query head: m, l and the unnormalised O relative to m
  float* rec = p.records + (((size_t)b * p.num_kv_heads + h) * p.chunks + chunk) * p.rec_floats;
  if (tid < g) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, wm_s[w][tid]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float wt = ex2(wm_s[w][tid] - ref);
      wm_s[w][tid] = wt;  // the warp's weight from here on
      lt += wt * wl_s[w][tid];
    }
    wl_s[0][tid] = lt;   // read below, after the barrier (warp 0's l is no longer needed)
    if (nch > 1) {
      rec[tid] = mx;
      rec[8 + tid] = lt;
    }
  }
  __syncthreads();
  for (int i = tid; i < g * HD; i += NT) {
    const int qi = i / HD, d = i - (i / HD) * HD;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      o += wm_s[w][qi] * sO[(w * DN + (d >> 3)) * OS + (qi * 4 + ((d & 7) >> 1)) * 2 + (d & 1)];
    if (nch == 1) {  // the whole list: normalise and write the output
      const float lt = wl_s[0][qi];
      out_bh[i] = __float2bfloat16_rn(lt > 0.f ? o / lt : 0.f);
    } else {
      rec[kRecHead + i] = o;
    }
  }
  if (nch == 1) return;

  // ticket: the CTA that completes the set of chunk records merges them
  __syncthreads();  // every record write of this CTA is issued
  if (tid == 0) {
    __threadfence();
    int32_t* tk = p.tickets + (size_t)b * p.num_kv_heads + h;
    const int old = atomicAdd(tk, 1);
    const int last = old == nch - 1;
    if (last) *tk = 0;  // every chunk has arrived: ready for the next call
    last_s = last;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  merge_records<HD, NT>(p, p.records + ((size_t)b * p.num_kv_heads + h) * p.chunks * p.rec_floats,
                        nch, out_bh, kt, Lay::kMergeBytes, mrun_s, lrun_s, corr_s);
}

struct DraftPlan {
  int chunks, rec_floats;
  size_t off_rec, ws_bytes;
};

bool make_draft_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int cap,
                     int max_tail, DraftPlan* pl) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || cap < 0 || max_tail < 0 ||
      cap + max_tail <= 0 || num_q_heads % num_kv_heads)
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->chunks = ceil_div(cap + max_tail, kChunk);
  pl->rec_floats = kRecHead + g * head_dim;
  pl->off_rec = align_up((size_t)batch * num_kv_heads * 4, 256);
  pl->ws_bytes =
      pl->off_rec + align_up((size_t)batch * num_kv_heads * pl->chunks * pl->rec_floats * 4, 256);
  return true;
}

template <int HD, bool SLOTS>
cudaError_t launch_draft_impl(const DraftParams& p, cudaStream_t stream) {
  using Lay = DraftLayout<HD, kChunk>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(sparse_draft_kernel<HD, kChunk, SLOTS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes(SLOTS));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.chunks, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(Lay::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Lay::bytes(SLOTS);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_draft_kernel<HD, kChunk, SLOTS>, p);
}

template <int HD>
cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream) {
  return p.slots ? launch_draft_impl<HD, true>(p, stream) : launch_draft_impl<HD, false>(p, stream);
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
                                               const int32_t* indices, const int32_t* slots,
                                               const int32_t* counts, int per_head, int cap,
                                               const int32_t* tail_start, const int32_t* cur_len,
                                               int batch, int num_q_heads, int max_tail,
                                               float softmax_scale, void* out, void* workspace,
                                               size_t workspace_bytes, int32_t* error_flag,
                                               cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (!q || !counts || !tail_start || !cur_len || !out || batch <= 0 || num_q_heads <= 0 ||
      cap < 0 || max_tail < 0 || cap + max_tail <= 0 || !(softmax_scale == softmax_scale))
    return VG_ERR_INVALID_ARGUMENT;
  if (cap > 0 && !indices) return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads % kv->num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / kv->num_kv_heads;
  if (g > 8) return VG_ERR_UNSUPPORTED;
  if ((long long)cap + max_tail > kMaxEntries) return VG_ERR_UNSUPPORTED;
  DraftPlan pl;
  if (!make_draft_plan(batch, num_q_heads, kv->num_kv_heads, kv->head_dim, cap, max_tail, &pl))
    return VG_ERR_INVALID_ARGUMENT;
  if (!workspace || workspace_bytes < pl.ws_bytes) return VG_ERR_WORKSPACE_TOO_SMALL;
  DraftParams p;
  p.k_pages = static_cast<const __nv_bfloat16*>(kv->k_pages);
  p.v_pages = static_cast<const __nv_bfloat16*>(kv->v_pages);
  p.page_table = kv->page_table;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.indices = indices;
  p.slots = cap > 0 ? slots : nullptr;
  p.counts = counts;
  p.tail_start = tail_start;
  p.cur_len = cur_len;
  p.out = static_cast<__nv_bfloat16*>(out);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.tickets = reinterpret_cast<int32_t*>(ws);
  p.records = reinterpret_cast<float*>(ws + pl.off_rec);
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
  p.rec_floats = pl.rec_floats;
  p.scale_log2 = softmax_scale * kLog2e;
  const cudaError_t e = kv->head_dim == 128 ? launch_draft<128>(p, stream)
                                             : launch_draft<64>(p, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
