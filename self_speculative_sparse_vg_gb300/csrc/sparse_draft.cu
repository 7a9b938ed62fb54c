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
// chunks of 16 W entries (W = 4 or 8 warps per CTA), and the chunks into S
// segments; one CTA per (segment, KV head, sequence), and the S CTAs of a
// (sequence, KV head) form one thread-block cluster (S <= 16).  W, S and the
// ring depth are planned on the host per launch so that the step's CTAs are
// resident at once; segment 0 (the cluster's leader) takes half a share of
// the chunks, the others a full share each.
//  * Addresses cost one round trip.  With the cache slots the selector wrote
//    beside the positions (physical page * 16 + offset, translated once per
//    selection) a chunk loads its slots and positions (the positions are
//    checked against the prefix); without slots the sequence's page-table row
//    is staged in shared memory with one bulk copy when it is short.  Only
//    the few tail entries look their page up after the lengths are known.
//  * A CTA streams its chunks through a ring of 2 to 6 stages (planned so
//    that, where shared memory allows, all of a CTA's chunks are requested
//    at once): the K and V rows of chunk j + stages are gathered while
//    chunk j is computed, in 16-byte cp.async pieces spread over all the
//    CTA's threads (per SM this sustains several times the rate of one bulk
//    copy per row, which the copy engine serves one at a time).  Rows are
//    padded to head_dim * 2 + 16 bytes, so the eight rows an ldmatrix reads
//    fall in eight distinct bank groups; rows without an entry are
//    zero-filled.
//  * The g query heads of the KV head are the rows of a 16-row bf16 mma.sync
//    tile (zero padded); warp w takes positions [16w, 16w + 16) of every
//    chunk and keeps a running softmax (row maximum, sum and O accumulators
//    in registers) over the CTA's chunks; P is reused as the A operand of
//    P.V.  The warps are merged once at the end through shared memory.
//  * Segments are merged inside the cluster, through distributed shared
//    memory: once its own chunks are done the leader arrives on every other
//    working CTA's "ready" mbarrier; each of them then pushes its fp32
//    record (m, l, unnormalised O per query head) into the leader's idle
//    ring with st.async, counted on the leader's mbarrier.  The leader merges
//    the records with its own registers by log-sum-exp and writes the output.
//    No global memory round trip and no workspace.  A list that fits the
//    leader's share is written directly.
#include <mutex>

#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

// A CTA has W warps (4 or 8, planned per launch) and takes chunks of 16 W
// attended entries: warp w computes entries [16w, 16w + 16) of each chunk.
constexpr int kMinStages = 2;        // chunks in flight per CTA: 2 .. kMaxStages, planned
constexpr int kMaxStages = 6;
constexpr int kMaxEntries = 65536;   // cap + max_tail
constexpr int kMaxSegments = 16;     // CTAs of a cluster (non-portable size above 8)
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
  int32_t* error_flag;
  int batch, num_q_heads, num_kv_heads, group, per_head, cap, max_tail;
  int num_pages, max_pages_per_seq;
  int segments;            // S: CTAs (cluster size) per (sequence, KV head)
  int stages;              // ring stages (chunks in flight) per CTA
  int chunks;              // chunks of the longest list, cut into the S segments
  uint64_t wait_ns;        // a wait longer than this reports VG_DEVERR_TIMEOUT (and goes on)
  float scale_log2;
};

template <int HD, int W>
struct DraftLayout {
  static constexpr int kChunk = 16 * W;                    // attended entries per chunk
  static constexpr int kThreads = 32 * W;
  static constexpr int kRowBytes = HD * 2 + 16;            // padded K / V row
  static constexpr int kTileBytes = kChunk * kRowBytes;    // one of K / V of a chunk
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMinRing = kMinStages * kStageBytes; // the ring is reused by the merges
  static constexpr int kOStride = 2 * 32 + 8;              // floats per (warp, n-tile) stash
  static constexpr size_t bytes(bool slots, int stages) {
    return 128 + (size_t)stages * kStageBytes + (slots ? 0 : (size_t)kPtMax * 4) + 64;
  }
  static constexpr int kRecBytes = (kRecHead + 8 * HD) * 4;  // one record at g = 8
  // deepest ring that fits 227 KB with the page-table row and static memory
  static constexpr int kStagesFit =
      (227 * 1024 - 6 * 1024 - 192 - kPtMax * 4) / kStageBytes < kMaxStages
          ? (227 * 1024 - 6 * 1024 - 192 - kPtMax * 4) / kStageBytes
          : kMaxStages;
  static_assert(kStagesFit >= kMinStages, "two stages fit");
  static_assert((size_t)W * (HD / 8) * kOStride * 4 <= (size_t)kMinRing,
                "the O stash reuses the ring");
  static_assert((size_t)(kMaxSegments - 1) * kRecBytes <= (size_t)kMinRing,
                "the leader receives the other segments' records in its ring");
  static_assert(kRowBytes % 16 == 0 && kTileBytes % 16 == 0, "16-byte copy destinations");
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
// t < kChunk owns entry t and publishes its row (or -1) in row_s; then every
// thread of the CTA copies a share of the chunk's K and V rows in 16-byte
// cp.async pieces, consecutive lanes on consecutive pieces of a row.  A row
// without an entry is zero-filled (source size 0).  The pieces form one
// cp.async group per chunk.
template <int HD, int W>
__device__ __forceinline__ void gather_chunk(const DraftParams& p, int row, int* row_s,
                                             uint8_t* stage) {
  using Lay = DraftLayout<HD, W>;
  constexpr int kChunk = Lay::kChunk, kThreads = Lay::kThreads;
  constexpr int RB = Lay::kRowBytes;
  constexpr int PR = HD * 2 / 16;  // pieces per row
  const int t = threadIdx.x;
  if (t < kChunk) row_s[t] = row;
  __syncthreads();
#pragma unroll 4
  for (int i = t; i < 2 * kChunk * PR; i += kThreads) {
    const int kv = i / (kChunk * PR);  // 0: K, 1: V
    const int rem = i - kv * kChunk * PR;
    const int rr = rem / PR, pc = rem - rr * PR;
    const int rw = row_s[rr];
    const __nv_bfloat16* base = kv ? p.v_pages : p.k_pages;
    cp_async_16_zfill(stage + kv * Lay::kTileBytes + rr * RB + pc * 16,
                      rw >= 0 ? base + (size_t)rw * HD + pc * 8 : base, rw >= 0);
  }
  cp_async_commit();
}

// First chunk of segment r of S over `chunks` chunks: the leader (r = 0)
// has weight 1, every other segment weight 2 (bounds rounded down).  With
// S <= chunks every segment but the leader's is non-empty.
__device__ __forceinline__ int seg_bound(int r, int S, int chunks) {
  const int w = r == 0 ? 0 : 2 * r - 1;
  return (int)(((long long)chunks * w) / (2 * S - 1));
}

template <int HD, bool SLOTS, int W>
__global__ void __launch_bounds__(32 * W) sparse_draft_kernel(const DraftParams p) {
  using Lay = DraftLayout<HD, W>;
  constexpr int kChunk = Lay::kChunk, kThreads = Lay::kThreads, kWarps = W;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DN = HD / 8;   // O n-tiles
  constexpr int RB = Lay::kRowBytes;
  constexpr int IT = (8 * HD / 4 + kThreads - 1) / kThreads;  // float4 columns of O per thread

  const int seg = blockIdx.x, h = blockIdx.y, b = blockIdx.z;  // seg = rank in the cluster
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = p.group, S = p.segments;
  const int row = p.per_head ? h : 0;
  const int rows = p.per_head ? p.num_kv_heads : 1;
  const int RF = kRecHead + g * HD;  // floats of one record
  // programmatic dependent launch: indices, slots and counts come from the
  // previous kernel; the next kernel may launch as soon as this grid runs
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  const int stages = p.stages;
  uint8_t* ring = smem;  // [stages][K tile, V tile]; then the O stash; leader: the records
  int32_t* pt_s = reinterpret_cast<int32_t*>(ring + (size_t)stages * Lay::kStageBytes);  // no slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(pt_s + (SLOTS ? 0 : kPtMax));  // [0] page table
  __shared__ int row_s[kMaxStages][kChunk];
  __shared__ __align__(8) uint64_t recv_bar;   // leader: the other segments' records landed
  __shared__ __align__(8) uint64_t ready_bar;  // other segments: the leader's ring is free
  __shared__ float wm_s[kWarps][16], wl_s[kWarps][16];
  __shared__ float segw_s[kMaxSegments][8];    // leader: merge weight of (segment, head)
  __shared__ float linv_s[8];

  if (tid == 0) {
    if (!SLOTS) mbar_init(&bars[0], 1);
    mbar_init(&recv_bar, 1);
    mbar_init(&ready_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // once this cluster barrier phase completes every CTA's mbarriers are
  // initialised; its wait comes just before the first remote access
  cluster_arrive_relaxed();

  // One round trip for everything the first chunks' addresses depend on:
  // their selected positions and slots (read speculatively; the arrays hold
  // cap entries), the query rows and the lengths (and, without slots, the
  // page-table row).
  const int c_first = seg_bound(seg, S, p.chunks);
  const int c_last = seg < S - 1 ? seg_bound(seg + 1, S, p.chunks) : p.chunks;
  const size_t lrow = ((size_t)b * rows + row) * p.cap;
  int pos_n[kMaxStages], slot_n[kMaxStages];
#pragma unroll
  for (int s = 0; s < kMaxStages; ++s) {
    const int e = (c_first + s) * kChunk + tid;
    pos_n[s] = -1;
    slot_n[s] = -1;
    if (tid < kChunk && e < p.cap && s < stages && c_first + s < c_last) {
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
  const int n_att = lengths_ok ? cnt + (cl - ts) : 0;
  const int nch = (n_att + kChunk - 1) / kChunk;  // chunks of this list
  const int c_end = min(c_last, nch);
  const bool work = c_first < c_end;
  // segments 1 .. n_send have work (their bounds increase with the rank)
  int n_send = 0;
  for (int q = 1; q < S; ++q) n_send += seg_bound(q, S, p.chunks) < nch;
  if (seg == 0 && tid == 0 && !lengths_ok)
    flag_error(p.error_flag, cnt < 0 || cnt > p.cap ? VG_DEVERR_COUNT : VG_DEVERR_LENGTH);
  if (seg == 0 && lengths_ok && n_att == 0)  // nothing attended: the output is zero
    for (int i = tid; i < g * HD / 2; i += kThreads) reinterpret_cast<uint32_t*>(out_bh)[i] = 0u;

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
  if (work) {
    __syncthreads();  // the page-table entries other threads copied are visible

    // ---- prologue: the first `stages` chunks in flight
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) {
      const int c = c_first + s;
      if (s < stages && c < c_end) {
        const int rw = tid < kChunk ? entry_row<SLOTS>(p, pt_s, pt_in_smem, b, h, c * kChunk + tid,
                                                       n_att, cnt, ts, pos_n[s], slot_n[s])
                                    : -1;
        gather_chunk<HD, W>(p, rw, row_s[s], ring + s * Lay::kStageBytes);
      } else if (s < stages) {
        cp_async_commit();  // an empty group: every chunk has stages - 1 groups after its own
      }
    }

    // ---- main loop: running softmax of this warp's rows over the chunks
    for (int c = c_first; c < c_end; ++c) {
      const int st = (c - c_first) % stages;
      // positions of chunk c + stages, loaded while this chunk is computed
      const int cn = c + stages;
      int pos_nx = -1, slot_nx = -1;
      if (cn < c_end && tid < kChunk) {
        const int e = cn * kChunk + tid;
        if (e < p.cap) {
          pos_nx = __ldg(p.indices + lrow + e);
          if (SLOTS) slot_nx = __ldg(p.slots + lrow + e);
        }
      }
      cp_async_wait_dyn(stages - 1);  // this thread's pieces of chunk c have landed
      __syncthreads();                // and every other thread's
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
      __syncthreads();  // the stage is free
      if (cn < c_end) {
        const int rw = tid < kChunk ? entry_row<SLOTS>(p, pt_s, pt_in_smem, b, h, cn * kChunk + tid,
                                                       n_att, cnt, ts, pos_nx, slot_nx)
                                    : -1;
        gather_chunk<HD, W>(p, rw, row_s[st], ring + st * Lay::kStageBytes);
      } else {
        cp_async_commit();
      }
    }
    __syncthreads();  // every stage has landed and been read: reuse the ring for the warp merge
  }

  // ---- this segment's record: m, l and the unnormalised O (relative to m)
  // per query head, the warps merged through an O stash in the accumulator's
  // own layout, rows 0..7 only (g <= 8): (warp, n-tile dn, lane) -> 2 floats,
  // rows r = lane / 4, columns 8 dn + 2 (lane % 4) + {0, 1}; n-tiles padded to
  // kOStride floats.  Thread t holds columns 4 (t + it * kThreads) of the
  // heads' concatenated O.
  constexpr int OS = Lay::kOStride;
  float* sO = reinterpret_cast<float*>(ring);
  float4 o4[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) o4[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (work) {
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
    __syncthreads();
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
      wl_s[0][tid] = lt;    // the segment's m and l, read below after the barrier
      wl_s[1][tid] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int i4 = tid + it * kThreads;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (i4 < g * HD / 4) {
        const int qi = (i4 * 4) / HD, d0 = i4 * 4 - qi * HD;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = d0 + k;
#pragma unroll
          for (int w = 0; w < kWarps; ++w)
            v[k] += wm_s[w][qi] * sO[(w * DN + (d >> 3)) * OS + (qi * 4 + ((d & 7) >> 1)) * 2 + (d & 1)];
        }
      }
      o4[it] = make_float4(v[0], v[1], v[2], v[3]);
    }
  }

  const uint32_t fill_bytes = (uint32_t)n_send * (uint32_t)RF * 4u;
  if (seg == 0 && work && n_send == 0) {  // the whole list is the leader's: write it
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int i4 = tid + it * kThreads;
      if (i4 < g * HD / 4) {
        const int qi = (i4 * 4) / HD;
        const float lt = wl_s[0][qi];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        uint2 w;
        w.x = pack_bf16(o4[it].x * inv, o4[it].y * inv);
        w.y = pack_bf16(o4[it].z * inv, o4[it].w * inv);
        *reinterpret_cast<uint2*>(out_bh + i4 * 4) = w;
      }
    }
  }
  cluster_wait_acquire();  // every CTA's mbarriers are initialised
  if (seg == 0 && n_send > 0) {
    // the ring is idle: arm the record count, then tell the senders
    __syncthreads();  // the O stash has been read
    fence_proxy_async_smem();
    if (tid == 0) mbar_arrive_expect_tx(&recv_bar, fill_bytes);
    __syncthreads();
    if (tid < n_send) mbar_arrive_remote(mapa_shared(smem_u32(&ready_bar), tid + 1));
  } else if (seg > 0 && work) {
    // push the record into slot seg - 1 of the leader's ring once it is free
    if (mbar_wait_checked<true>(&ready_bar, 0, p.wait_ns, p.error_flag)) {
      const uint32_t dst = mapa_shared(smem_u32(ring + (size_t)(seg - 1) * RF * 4), 0);
      const uint32_t rb = mapa_shared(smem_u32(&recv_bar), 0);
      if (tid < 4) {  // header: m[8], l[8] (heads >= g: m = -inf, l = 0)
        float hv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int qi = (tid & 1) * 4 + k;
          hv[k] = tid < 2 ? (qi < g ? wl_s[1][qi] : -INFINITY) : (qi < g ? wl_s[0][qi] : 0.f);
        }
        st_async_v4(dst + tid * 16,
                    make_uint4(__float_as_uint(hv[0]), __float_as_uint(hv[1]),
                               __float_as_uint(hv[2]), __float_as_uint(hv[3])),
                    rb);
      }
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int i4 = tid + it * kThreads;
        if (i4 < g * HD / 4)
          st_async_v4(dst + kRecHead * 4 + i4 * 16,
                      make_uint4(__float_as_uint(o4[it].x), __float_as_uint(o4[it].y),
                                 __float_as_uint(o4[it].z), __float_as_uint(o4[it].w)),
                      rb);
      }
    }
  }
  if (seg == 0 && n_send > 0) {
    // ---- leader: log-sum-exp merge of its own record (registers) and the
    // n_send pushed ones (ring slots 0 .. n_send - 1)
    const bool got =
        __syncthreads_and(mbar_wait_checked<true>(&recv_bar, 0, p.wait_ns, p.error_flag));
    cluster_arrive_release();  // the records have landed: the senders may leave
    if (got) {
      const float* recs = reinterpret_cast<const float*>(ring);
      // weights: warp w takes query heads w, w + W, ...; lane q < n_send
      // holds pushed record q, lane 16 the leader's own (m = -inf without work)
      for (int qi = warp; qi < g; qi += kWarps) {
        float mq = -INFINITY, lq = 0.f;
        if (lane < n_send) {
          mq = recs[(size_t)lane * RF + qi];
          lq = recs[(size_t)lane * RF + 8 + qi];
        } else if (lane == 16 && work) {
          mq = wl_s[1][qi];
          lq = wl_s[0][qi];
        }
        float mx = mq;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float w = ex2(mq - safe_ref(mx));  // 0 for an empty slot
        float lt = w * lq;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
        if (lane < n_send) segw_s[lane + 1][qi] = w;
        if (lane == 16) segw_s[0][qi] = w;
        if (lane == 0) linv_s[qi] = lt > 0.f ? 1.f / lt : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int i4 = tid + it * kThreads;
        if (i4 < g * HD / 4) {
          const int qi = (i4 * 4) / HD;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          if (work) {
            const float w0 = segw_s[0][qi];
            a = make_float4(w0 * o4[it].x, w0 * o4[it].y, w0 * o4[it].z, w0 * o4[it].w);
          }
          for (int q = 0; q < n_send; ++q) {
            const float w = segw_s[q + 1][qi];
            const float4 o =
                *reinterpret_cast<const float4*>(recs + (size_t)q * RF + kRecHead + i4 * 4);
            a.x += w * o.x;
            a.y += w * o.y;
            a.z += w * o.z;
            a.w += w * o.w;
          }
          const float inv = linv_s[qi];
          uint2 wv;
          wv.x = pack_bf16(a.x * inv, a.y * inv);
          wv.y = pack_bf16(a.z * inv, a.w * inv);
          *reinterpret_cast<uint2*>(out_bh + i4 * 4) = wv;
        }
      }
    }
  } else {
    cluster_arrive_release();
  }
  cluster_wait_acquire();  // senders stay until the leader holds their records
}

// CTAs of the draft kernel resident per SM with a ring of `stages` stages
// (cached per device, variant and stages; -1 when the ring does not fit);
// also sets the kernel's dynamic shared-memory limit and allows clusters of
// up to 16 CTAs, once per device.
template <int HD, bool SLOTS, int W>
int draft_occupancy(int stages) {
  using Lay = DraftLayout<HD, W>;
  static int cached[64][kMaxStages + 1] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || stages < kMinStages ||
      stages > Lay::kStagesFit)
    return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][0] == 0) {
    const bool ok =
        cudaFuncSetAttribute(sparse_draft_kernel<HD, SLOTS, W>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Lay::bytes(SLOTS, Lay::kStagesFit)) == cudaSuccess &&
        cudaFuncSetAttribute(sparse_draft_kernel<HD, SLOTS, W>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    cached[dev][0] = ok ? 1 : -1;
  }
  if (cached[dev][0] < 0) return -1;
  if (cached[dev][stages] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sparse_draft_kernel<HD, SLOTS, W>,
                                                      Lay::kThreads,
                                                      Lay::bytes(SLOTS, stages)) != cudaSuccess ||
        n <= 0)
      n = -1;
    cached[dev][stages] = n;
  }
  return cached[dev][stages];
}

// Clusters of S draft CTAs (ring of `stages` stages) the device holds at
// once (cached per device, variant, S and stages).
template <int HD, bool SLOTS, int W>
int draft_max_clusters(int S, int stages) {
  using Lay = DraftLayout<HD, W>;
  static int cached[64][kMaxSegments + 1][kMaxStages + 1] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || S < 1 || S > kMaxSegments ||
      stages < kMinStages || stages > Lay::kStagesFit)
    return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cached[dev][S][stages];
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(Lay::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Lay::bytes(SLOTS, stages);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_draft_kernel<HD, SLOTS, W>, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    c = n > 0 ? n : -1;
  }
  return c;
}

struct DraftPlan {
  int chunks, segments, stages;
};

// Segments and ring depth of a step with W-warp CTAs.  For each ring depth:
// as many segments as keep every CTA of the step resident at once, at most
// kMaxSegments (one cluster) and at most (chunks + 1) / 2 (two chunks a
// segment, one for the leader's half share), fewer while the device cannot
// hold all the step's clusters at once.  A CTA then needs ceil(chunks of
// its segment / stages) rounds of requests; the plan takes the depth with
// the fewest rounds (the shallowest of equals, which keeps most CTAs
// resident).
template <int HD, bool SLOTS, int W>
bool make_draft_plan(int batch, int num_kv_heads, int cap, int max_tail, DraftPlan* pl) {
  using Lay = DraftLayout<HD, W>;
  pl->chunks = ceil_div(cap + max_tail, Lay::kChunk);
  const long long units = (long long)batch * num_kv_heads;
  long long best_rounds = -1;
  for (int st = kMinStages; st <= Lay::kStagesFit; ++st) {
    const int occ = draft_occupancy<HD, SLOTS, W>(st);
    if (occ <= 0) continue;
    const long long resident = (long long)device_sm_count() * occ;
    long long S = std::max<long long>(1, resident / units);
    S = std::min<long long>(S, kMaxSegments);
    S = std::min<long long>(S, std::max(1, (pl->chunks + 1) / 2));
    while (S > 1 && draft_max_clusters<HD, SLOTS, W>((int)S, st) < units) --S;
    if (draft_max_clusters<HD, SLOTS, W>((int)S, st) <= 0) continue;
    const long long share = (2LL * pl->chunks + 2 * S - 2) / (2 * S - 1);  // chunks of a segment
    const long long rounds = (share + st - 1) / st;
    if (best_rounds < 0 || rounds < best_rounds) {
      best_rounds = rounds;
      pl->segments = (int)S;
      pl->stages = st;
    }
  }
  return best_rounds > 0;
}

template <int HD, bool SLOTS, int W>
cudaError_t launch_draft_w(DraftParams p, const DraftPlan& pl, cudaStream_t stream) {
  p.segments = pl.segments;
  p.chunks = pl.chunks;
  p.stages = pl.stages;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.segments;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.segments, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(DraftLayout<HD, W>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = DraftLayout<HD, W>::bytes(SLOTS, pl.stages);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sparse_draft_kernel<HD, SLOTS, W>, p);
}

// CTAs of 4 warps when the step has CTAs to spare for every SM (many
// (sequence, KV head) pairs); otherwise CTAs of 8 warps, whose gathers
// draw twice the threads per SM on the few SMs the step occupies.
template <int HD, bool SLOTS>
cudaError_t launch_draft_impl(const DraftParams& p, cudaStream_t stream) {
  DraftPlan p4, p8;
  const bool ok4 = make_draft_plan<HD, SLOTS, 4>(p.batch, p.num_kv_heads, p.cap, p.max_tail, &p4);
  const bool ok8 = make_draft_plan<HD, SLOTS, 8>(p.batch, p.num_kv_heads, p.cap, p.max_tail, &p8);
  const long long ctas4 = ok4 ? (long long)p.batch * p.num_kv_heads * p4.segments : 0;
  if (ok8 && (!ok4 || ctas4 <= device_sm_count())) return launch_draft_w<HD, SLOTS, 8>(p, p8, stream);
  if (ok4) return launch_draft_w<HD, SLOTS, 4>(p, p4, stream);
  return cudaErrorInvalidConfiguration;
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
  (void)batch, (void)num_q_heads, (void)num_kv_heads, (void)head_dim, (void)cap, (void)max_tail;
  return 0;  // segments merge inside their cluster
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
  if (kv->head_dim != 64 && kv->head_dim != 128) return VG_ERR_UNSUPPORTED;
  (void)workspace, (void)workspace_bytes;  // none needed
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
  p.segments = 0;  // planned at launch
  p.chunks = 0;
  p.stages = 0;
  p.wait_ns = wait_report_ns();
  p.scale_log2 = softmax_scale * kLog2e;
  const cudaError_t e = kv->head_dim == 128 ? launch_draft<128>(p, stream)
                                             : launch_draft<64>(p, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
