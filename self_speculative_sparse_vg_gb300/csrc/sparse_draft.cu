// Sparse draft attention over the selected KV entries plus the dense tail
// (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" and Figure 1: while drafting, each draft token attends only the
// KV entries picked from the previous verification; A Sparse Glimpse of the
// Whole, "What carries the argument": the dense cache is kept, the index is a
// view into it.
//
// Design: one kernel per draft step.  The attended list of a (sequence, KV
// head) -- the selection, then the tail [tail_start, cur_len) -- is cut into
// 64-entry chunks, and the chunks into S segments of `cpc` consecutive chunks;
// one CTA per (segment, KV head, sequence).  S and cpc are planned on the host
// so that every CTA of a step is resident at once and each walks at least
// two chunks.
//  * Addresses cost one round trip.  With the cache slots the selector wrote
//    beside the positions (physical page * 16 + offset, translated once per
//    selection) a chunk loads its slots and positions (the positions are
//    checked against the prefix); without slots the sequence's page-table row
//    is staged in shared memory with one bulk copy when it is short.  Only
//    the few tail entries look their page up after the lengths are known.
//  * A CTA streams its chunks through a two-stage ring: the K and V rows of
//    chunk j + 2 are gathered while chunk j is computed, one bulk copy per
//    row (256 bytes at head_dim 128) issued by the row's thread and counted
//    on the stage's mbarrier.  Rows are padded to head_dim * 2 + 16 bytes,
//    so the eight rows an ldmatrix reads fall in eight distinct bank groups;
//    rows without an entry are zero-filled.
//  * The g query heads of the KV head are the rows of a 16-row bf16 mma.sync
//    tile (zero padded); warp w takes positions [16w, 16w + 16) of every
//    chunk and keeps a running softmax (row maximum, sum and O accumulators
//    in registers) over the CTA's chunks; P is reused as the A operand of
//    P.V.  The warps are merged once at the end through shared memory.
//  * A list that fits one segment writes the output directly.  Otherwise
//    each CTA writes an fp32 record (m, l, unnormalised O per query head) and
//    takes a ticket from a per-(sequence, KV head) counter; the CTA that draws
//    the last ticket stages every record of its pair into shared memory with
//    one batch of cp.async copies, merges them by log-sum-exp, writes the
//    output and puts the counter back to zero.  No CTA waits for another.
#include <mutex>

#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kChunk = 64;           // attended entries per chunk
constexpr int kWarps = kChunk / 16;  // one warp per 16 entries
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;           // chunks in flight per CTA
constexpr int kMaxEntries = 65536;   // cap + max_tail
constexpr int kMaxSegments = 32;     // records per (sequence, KV head)
constexpr int kPtMax = 2048;         // page-table entries staged in shared memory (no slots)
constexpr int kRecHead = 16;         // floats before O in a record: m[8], l[8]

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
  float* records;          // [B][Hkv][segments][rec_floats]
  int32_t* tickets;        // [B][Hkv], zero between calls
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq, segments, cpc, rec_floats;
  uint64_t wait_ns;        // a wait longer than this reports VG_DEVERR_TIMEOUT (and goes on)
  float scale_log2;
};

template <int HD>
struct DraftLayout {
  static constexpr int kRowBytes = HD * 2 + 16;            // padded K / V row
  static constexpr int kTileBytes = kChunk * kRowBytes;    // one of K / V of a chunk
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes; // reused by the merges
  static constexpr int kOStride = 2 * 32 + 8;              // floats per (warp, n-tile) stash
  static constexpr size_t bytes(bool slots) {
    return 128 + (size_t)kRingBytes + (slots ? 0 : (size_t)kPtMax * 4) + 64;
  }
  static_assert((size_t)kWarps * (HD / 8) * kOStride * 4 <= (size_t)kRingBytes,
                "the O stash reuses the ring");
  static_assert(kRowBytes % 16 == 0 && kTileBytes % 16 == 0, "16-byte bulk-copy destinations");
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

// Row of list entry e's K/V in the pools viewed as [pages * heads * 16]
// rows of head_dim elements, or -1 (entry past the list, or a bad index, slot
// or page: the error is flagged).
template <bool SLOTS>
__device__ __forceinline__ int entry_row(const DraftParams& p, const int32_t* pt_s,
                                                  bool pt_in_smem, int b, int h, int e, int n_att,
                                                  int cnt, int ts, int pos_sel, int slot_sel) {
  if (e >= n_att) return -1;
  int phys = -1, sl = 0;
  if (e < cnt) {
    const int pos = pos_sel;
    // a slot must address the position's own offset within its page
    const bool ok = pos >= 0 && pos < ts &&
                    !(SLOTS && slot_sel >= 0 && (slot_sel & 15) != (pos & 15));
    if (!ok) {
      flag_error(p.error_flag, VG_DEVERR_INDEX);
      return -1;
    }
    if (SLOTS) {
      phys = slot_sel < 0 ? -1 : slot_sel >> 4;
      sl = slot_sel & 15;
    } else {
      phys = pt_in_smem ? pt_s[pos / kPageSize]
                        : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
      sl = pos % kPageSize;
    }
  } else {
    const int pos = ts + (e - cnt);  // tail: its page is looked up now
    phys = pt_in_smem ? pt_s[pos / kPageSize]
                      : __ldg(p.page_table + (size_t)b * p.max_pages_per_seq + pos / kPageSize);
    sl = pos % kPageSize;
  }
  if (phys < 0 || phys >= p.num_pages) {
    flag_error(p.error_flag, VG_DEVERR_PAGE);
    return -1;
  }
  return (phys * p.num_kv_heads + h) * kPageSize + sl;
}

// Resolve the rows of one chunk and gather them into a ring stage: thread
// t < kChunk owns entry t, writes its row to row_s, zero-fills its K and V
// rows when it has none, and otherwise issues two bulk copies (K, V) counted
// on `bar`.  Thread 0 sets the stage's expected byte count first.  Ends with
// the stage's rows in flight and row_s visible to the CTA.
template <int HD>
__device__ __forceinline__ void gather_chunk(const DraftParams& p, int row, int* row_s,
                                             uint8_t* stage, uint64_t* bar) {
  using Lay = DraftLayout<HD>;
  constexpr int RB = Lay::kRowBytes;
  const int t = threadIdx.x;
  const bool mine = t < kChunk;
  if (mine) {
    row_s[t] = row;
    if (row < 0) {
#pragma unroll
      for (int c = 0; c < HD / 8; ++c) {
        *reinterpret_cast<uint4*>(stage + t * RB + c * 16) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(stage + Lay::kTileBytes + t * RB + c * 16) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  const int nvalid = __syncthreads_count(mine && row >= 0);
  if (t == 0) mbar_arrive_expect_tx(bar, (uint32_t)nvalid * 2u * HD * 2u);
  __syncthreads();  // the expected count precedes every copy's completion
  if (mine && row >= 0) {
    bulk_load(stage + t * RB, p.k_pages + (size_t)row * HD, HD * 2, bar);
    bulk_load(stage + Lay::kTileBytes + t * RB, p.v_pages + (size_t)row * HD, HD * 2, bar);
  }
}

// Wait for a ring stage.  A slow wait is reported and goes on; one that
// gives up even so is waited out once more (bounded), so that no load is
// left writing into shared memory when the CTA leaves.
__device__ __forceinline__ void wait_stage(const DraftParams& p, uint64_t* bar, uint32_t parity) {
  if (!mbar_wait_checked(bar, parity, p.wait_ns, p.error_flag)) mbar_wait(bar, parity);
}

// Log-sum-exp merge of the nseg segment records of one (sequence, KV head)
// by the CTA that drew the last ticket.  The records are staged into shared
// memory a batch at a time with cp.async (every copy of a batch in flight
// together); warp w forms the batch weights of query heads w, w + 4, ...;
// then each thread accumulates float4 columns of the heads' O.
template <int HD>
__device__ __forceinline__ void merge_records(const DraftParams& p, const float* src, int nseg,
                                              __nv_bfloat16* dst, uint8_t* area, int area_bytes,
                                              float* mrun_s, float* lrun_s, float* corr_s) {
  constexpr int C4 = HD / 4;
  constexpr int IPT = (8 * C4 + kThreads - 1) / kThreads;  // items per thread at g = 8
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group, RF = p.rec_floats;
  const int cpb = (area_bytes - 64) / (RF * 4 + 32);  // records per batch (w_s: 8 floats each)
  float* recs = reinterpret_cast<float*>(area);
  float* w_s = recs + (size_t)cpb * RF;
  if (tid < 8) {
    mrun_s[tid] = -INFINITY;
    lrun_s[tid] = 0.f;
  }
  float4 acc[IPT];
#pragma unroll
  for (int i = 0; i < IPT; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nseg; c0 += cpb) {
    const int nb = min(cpb, nseg - c0);
    const int n4 = nb * RF / 4;
    const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)c0 * RF);
    for (int i = tid; i < n4; i += kThreads) cp_async_16(recs + (size_t)i * 4, s4 + i);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int qi = warp; qi < g; qi += kWarps) {
      float mb = -INFINITY;
      for (int c = lane; c < nb; c += 32) mb = fmaxf(mb, recs[(size_t)c * RF + qi]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_old = mrun_s[qi];
      const float m_new = fmaxf(m_old, mb);
      const float ref = safe_ref(m_new);
      float lb = 0.f;
      for (int c = lane; c < nb; c += 32) {
        const float w = ex2(recs[(size_t)c * RF + qi] - ref);  // 0 for an empty segment
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
      const int i = tid + it * kThreads;
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
    const int i = tid + it * kThreads;
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

template <int HD, bool SLOTS>
__global__ void __launch_bounds__(kThreads) sparse_draft_kernel(const DraftParams p) {
  using Lay = DraftLayout<HD>;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DN = HD / 8;   // O n-tiles
  constexpr int RB = Lay::kRowBytes;

  const int seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
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
  uint8_t* ring = smem;                     // [kStages][K tile, V tile]
  int32_t* pt_s = reinterpret_cast<int32_t*>(ring + Lay::kRingBytes);  // no slots: page-table row
  uint64_t* bars = reinterpret_cast<uint64_t*>(pt_s + (SLOTS ? 0 : kPtMax));  // [0] page table
  __shared__ int row_s[kStages][kChunk];
  __shared__ __align__(8) uint64_t stage_bar[kStages];
  __shared__ float wm_s[kWarps][16], wl_s[kWarps][16];
  __shared__ float mrun_s[8], lrun_s[8], corr_s[8];
  __shared__ int last_s;

  if (tid == 0) {
    if (!SLOTS) mbar_init(&bars[0], 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&stage_bar[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // One round trip for everything the first chunks' addresses depend on:
  // their selected positions and slots (read speculatively; the arrays hold
  // cap entries), the query rows and the lengths (and, without slots, the
  // page-table row).
  const int c_first = seg * p.cpc;
  const size_t lrow = ((size_t)b * rows + row) * p.cap;
  int pos_n[kStages], slot_n[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    const int e = (c_first + s) * kChunk + tid;
    pos_n[s] = -1;
    slot_n[s] = -1;
    if (tid < kChunk && e < p.cap && s < p.cpc) {
      pos_n[s] = __ldg(p.indices + lrow + e);
      if (SLOTS) slot_n[s] = __ldg(p.slots + lrow + e);
    }
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
      for (int k = nb + tid; k < n; k += kThreads) pt_s[k] = __ldg(src + k);
    } else if (tid == 0) {
      mbar_arrive(&bars[0]);
    }
  }
  // Q as the A fragments of the 16-row tile (rows >= g zero), straight from
  // global memory: lane (r, c) holds Q[r][16 ks + 2c, +1] and Q[r][16 ks + 2c
  // + 8, +1] of k-step ks; rows r + 8 are padding
  const int r = lane >> 2, c4 = lane & 3;
  uint32_t qa[KS][4];
  {
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(p.q + ((size_t)b * p.num_q_heads + h * g + r) * HD);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = r < g ? __ldg(qrow + ks * 8 + c4) : 0u;
      qa[ks][2] = r < g ? __ldg(qrow + ks * 8 + 4 + c4) : 0u;
      qa[ks][1] = 0u;
      qa[ks][3] = 0u;
    }
  }
  int cnt, ts, cl;
  const bool lengths_ok = draft_lengths(p, b, row, rows, &cnt, &ts, &cl);
  if (!SLOTS) {
    // the page-table copy must land before anything reads it or the CTA
    // leaves; a wait that gives up is reported and waited out once more
    if (!mbar_wait_checked(&bars[0], 0, p.wait_ns, p.error_flag)) mbar_wait(&bars[0], 0);
  }
  __nv_bfloat16* out_bh = p.out + ((size_t)b * p.num_q_heads + h * g) * HD;
  if (!lengths_ok) {
    if (tid == 0 && seg == 0)
      flag_error(p.error_flag, cnt < 0 || cnt > p.cap ? VG_DEVERR_COUNT : VG_DEVERR_LENGTH);
    return;
  }
  const int n_att = cnt + (cl - ts);
  const int nch = (n_att + kChunk - 1) / kChunk;       // chunks of the list
  const int nseg = (nch + p.cpc - 1) / p.cpc;          // segments with work
  if (n_att == 0) {  // nothing attended: the output is zero
    if (seg == 0)
      for (int i = tid; i < g * HD / 2; i += kThreads) reinterpret_cast<uint32_t*>(out_bh)[i] = 0u;
    return;
  }
  const int c_end = min(c_first + p.cpc, nch);
  if (c_first >= c_end) return;  // past the end of this list: no record, no ticket
  __syncthreads();  // the page-table entries other threads copied are visible

  // ---- prologue: the first kStages chunks in flight
#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    const int c = c_first + s;
    if (c < c_end) {
      const int row = tid < kChunk ? entry_row<SLOTS>(p, pt_s, pt_in_smem, b, h, c * kChunk + tid,
                                                      n_att, cnt, ts, pos_n[s], slot_n[s])
                                   : -1;
      gather_chunk<HD>(p, row, row_s[s], ring + s * Lay::kStageBytes, &stage_bar[s]);
    }
  }

  // ---- main loop: running softmax of this warp's rows over the chunks
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
  for (int c = c_first; c < c_end; ++c) {
    const int st = (c - c_first) % kStages;
    // positions of chunk c + kStages, loaded while this chunk is computed
    const int cn = c + kStages;
    int pos_nx = -1, slot_nx = -1;
    if (cn < c_end && tid < kChunk) {
      const int e = cn * kChunk + tid;
      if (e < p.cap) {
        pos_nx = __ldg(p.indices + lrow + e);
        if (SLOTS) slot_nx = __ldg(p.slots + lrow + e);
      }
    }
    wait_stage(p, &stage_bar[st], ((c - c_first) / kStages) & 1);  // this chunk's rows landed
    const int ne = min(kChunk, n_att - c * kChunk);
    if (warp * 16 < ne) {  // warp-uniform
      const uint32_t ku = smem_u32(ring + st * Lay::kStageBytes);
      const uint32_t vu = ku + Lay::kTileBytes;
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
      float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = warp * 16 + nt * 8 + 2 * c4 + k;
          const bool valid = j < ne && row_s[st][j] >= 0;
          s[nt][k] = valid ? s[nt][k] * p.scale_log2 : -INFINITY;
          s[nt][2 + k] = valid ? s[nt][2 + k] * p.scale_log2 : -INFINITY;
          cm0 = fmaxf(cm0, s[nt][k]);
          cm1 = fmaxf(cm1, s[nt][2 + k]);
        }
      }
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 1));
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, 2));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 1));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, 2));
      // move the running reference up when this chunk's maximum is larger
      const float n0 = fmaxf(m0, cm0), n1 = fmaxf(m1, cm1);
      const float ref0 = safe_ref(n0), ref1 = safe_ref(n1);
      const float k0 = ex2(m0 - ref0), k1 = ex2(m1 - ref1);  // 0 while nothing was accumulated
      m0 = n0;
      m1 = n1;
      l0 *= k0;
      l1 *= k1;
#pragma unroll
      for (int dn = 0; dn < DN; ++dn) {
        acc[dn][0] *= k0;
        acc[dn][1] *= k0;
        acc[dn][2] *= k1;
        acc[dn][3] *= k1;
      }
      uint32_t pa[4];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p00 = ex2(s[nt][0] - ref0), p01 = ex2(s[nt][1] - ref0);
        const float p10 = ex2(s[nt][2] - ref1), p11 = ex2(s[nt][3] - ref1);
        ls0 += p00 + p01;
        ls1 += p10 + p11;
        pa[nt * 2 + 0] = pack_bf16(p00, p01);
        pa[nt * 2 + 1] = pack_bf16(p10, p11);
      }
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
      l0 += ls0;
      l1 += ls1;
#pragma unroll
      for (int dp = 0; dp < DN / 2; ++dp) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vu + vrow * RB + (2 * dp + (lane >> 4)) * 16, v0, v1, v2, v3);
        mma_16816(acc[2 * dp], pa, v0, v1);
        mma_16816(acc[2 * dp + 1], pa, v2, v3);
      }
    }
    fence_proxy_async_smem();  // this thread's reads of the stage precede the next loads
    __syncthreads();           // the stage is free
    if (cn < c_end) {
      const int row = tid < kChunk ? entry_row<SLOTS>(p, pt_s, pt_in_smem, b, h, cn * kChunk + tid,
                                                      n_att, cnt, ts, pos_nx, slot_nx)
                                   : -1;
      gather_chunk<HD>(p, row, row_s[st], ring + st * Lay::kStageBytes, &stage_bar[st]);
    }
  }
  __syncthreads();  // every stage has landed and been read: reuse the ring for the warp merge

  // O stash in the accumulator's own layout, rows 0..7 only (g <= 8):
  // (warp, n-tile dn, lane) -> 2 floats, rows r = lane / 4, columns
  // 8 dn + 2 (lane % 4) + {0, 1}; n-tiles padded to kOStride floats
  constexpr int OS = Lay::kOStride;
  float* sO = reinterpret_cast<float*>(ring);
  {
#pragma unroll
    for (int dn = 0; dn < DN; ++dn)
      *reinterpret_cast<float2*>(&sO[(warp * DN + dn) * OS + lane * 2]) =
          make_float2(acc[dn][0], acc[dn][1]);
    if (c4 == 0) {
      wm_s[warp][r] = m0;
      wl_s[warp][r] = l0;
      wm_s[warp][r + 8] = m1;
      wl_s[warp][r + 8] = l1;
    }
  }
  __syncthreads();
  // segment result per query head: m, l and the unnormalised O relative to m
  float* rec = p.records + (((size_t)b * p.num_kv_heads + h) * p.segments + seg) * p.rec_floats;
  if (tid < g) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, wm_s[w][tid]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = ex2(wm_s[w][tid] - ref);
      wm_s[w][tid] = wt;  // the warp's weight from here on
      lt += wt * wl_s[w][tid];
    }
    wl_s[0][tid] = lt;    // read below, after the barrier
    if (nseg > 1) {
      rec[tid] = mx;
      rec[8 + tid] = lt;
    }
  }
  __syncthreads();
  for (int i = tid; i < g * HD; i += kThreads) {
    const int qi = i / HD, d = i - (i / HD) * HD;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      o += wm_s[w][qi] * sO[(w * DN + (d >> 3)) * OS + (qi * 4 + ((d & 7) >> 1)) * 2 + (d & 1)];
    if (nseg == 1) {  // the whole list: normalise and write the output
      const float lt = wl_s[0][qi];
      out_bh[i] = __float2bfloat16_rn(lt > 0.f ? o / lt : 0.f);
    } else {
      rec[kRecHead + i] = o;
    }
  }
  if (nseg == 1) return;

  // ticket: the CTA that completes the set of records merges them.  The
  // acquire-release add publishes this CTA's record (ordered before it by the
  // barrier) and, for the last CTA, makes every other record visible.
  __syncthreads();  // every record write of this CTA is issued
  if (tid == 0) {
    int32_t* tkt = p.tickets + (size_t)b * p.num_kv_heads + h;
    const int old = atomic_add_acq_rel_gpu(tkt, 1);
    const int last = old == nseg - 1;
    if (last) *tkt = 0;  // every segment has arrived: ready for the next call
    last_s = last;
  }
  __syncthreads();
  if (!last_s) return;
  merge_records<HD>(p, p.records + ((size_t)b * p.num_kv_heads + h) * p.segments * p.rec_floats,
                    nseg, out_bh, ring, Lay::kRingBytes, mrun_s, lrun_s, corr_s);
}

// CTAs of the draft kernel resident per SM (cached per device and variant);
// also sets the kernel's dynamic shared-memory limit once per device.
template <int HD, bool SLOTS>
int draft_occupancy() {
  static int cached[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    const int bytes = (int)DraftLayout<HD>::bytes(SLOTS);
    if (cudaFuncSetAttribute(sparse_draft_kernel<HD, SLOTS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sparse_draft_kernel<HD, SLOTS>, kThreads,
                                                      bytes) != cudaSuccess ||
        n <= 0)
      n = -1;
    cached[dev] = n;
  }
  return cached[dev];
}

struct DraftPlan {
  int chunks, cpc, segments, rec_floats;
  size_t off_rec, ws_bytes;
};

// Segments of a (sequence, KV head) list: every CTA of the step resident at
// once (SMs x occupancy), at least two chunks per CTA, at most kMaxSegments
// records to merge.  The plan depends only on the sizes and the device, so
// that the workspace query and the call agree.
bool make_draft_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int cap,
                     int max_tail, DraftPlan* pl) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || cap < 0 || max_tail < 0 ||
      cap + max_tail <= 0 || num_q_heads % num_kv_heads || (head_dim != 64 && head_dim != 128))
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->chunks = ceil_div(cap + max_tail, kChunk);
  const int o1 = head_dim == 128 ? draft_occupancy<128, true>() : draft_occupancy<64, true>();
  const int o2 = head_dim == 128 ? draft_occupancy<128, false>() : draft_occupancy<64, false>();
  const int occ = std::max(1, std::min(o1, o2));
  const long long resident = (long long)device_sm_count() * occ;
  const long long total = (long long)batch * num_kv_heads * pl->chunks;
  int cpc = (int)std::max<long long>(2, (total + resident - 1) / resident);
  cpc = std::max(cpc, ceil_div(pl->chunks, kMaxSegments));
  pl->cpc = std::min(cpc, pl->chunks);
  pl->segments = ceil_div(pl->chunks, pl->cpc);
  pl->rec_floats = kRecHead + g * head_dim;
  pl->off_rec = align_up((size_t)batch * num_kv_heads * 4, 256);
  pl->ws_bytes =
      pl->off_rec + align_up((size_t)batch * num_kv_heads * pl->segments * pl->rec_floats * 4, 256);
  return true;
}

template <int HD, bool SLOTS>
cudaError_t launch_draft_impl(const DraftParams& p, cudaStream_t stream) {
  if (draft_occupancy<HD, SLOTS>() <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.segments, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = DraftLayout<HD>::bytes(SLOTS);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_draft_kernel<HD, SLOTS>, p);
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
  if ((long long)kv->num_pages * kv->num_kv_heads * kPageSize >= (1ll << 31))
    return VG_ERR_UNSUPPORTED;  // row numbers are 32-bit
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
  p.segments = pl.segments;
  p.cpc = pl.cpc;
  p.rec_floats = pl.rec_floats;
  p.wait_ns = wait_report_ns();
  p.scale_log2 = softmax_scale * kLog2e;
  const cudaError_t e = kv->head_dim == 128 ? launch_draft<128>(p, stream)
                                             : launch_draft<64>(p, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
