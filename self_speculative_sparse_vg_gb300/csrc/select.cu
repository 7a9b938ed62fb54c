// Verification-guided KV selection: sink + recent + top-k (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim": combine the captured first-draft and bonus logit rows across
// the query heads and keep the top-k prefix positions.  A Sparse Glimpse of
// the Whole, "What carries the argument": sink and recent tokens are always
// kept; per-head index variant.
//
// Design: one thread-block cluster of C (<= 16) CTAs per selection row; CTA c
// owns a contiguous slice of positions.  Each position's fp32 score is formed
// in the documented order and turned into an order-preserving 32-bit key:
// for the per-KV-head sum captures, when a CTA's share is at most 32K loads,
// by the cluster's CTAs themselves, straight into shared memory; otherwise
// (longer prefixes, raw-row and attention-weight captures) by a score kernel
// spread over many CTAs, through the workspace.  Clusters are halved (longer
// slices) while a batch's clusters would not all be resident at once: a
// second wave of clusters costs as much as the first.  The cluster then runs an
// MSB-first 8-bit radix select (at most 4 passes, fewer once the whole
// boundary bin is kept): every CTA pushes its 256-bin histogram into every
// CTA's shared memory with st.async, each CTA waits on a local mbarrier for
// the C histograms and sums them itself (no cluster barrier per pass).  That
// yields the exact top_k-th key T.  Keys > T are all kept; keys == T are kept
// by ascending position, using per-CTA counts pushed the same way; each CTA
// then writes its kept positions in order straight into their final slots.
// The result is deterministic and equals a stable sort by (score desc,
// position asc).
#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <tuple>

#include "vg_device.cuh"
#include "vg_host.h"

namespace cg = cooperative_groups;

namespace vg {
namespace {

// CTAs of the selection cluster have NT = 1024 threads, or 512 (two CTAs per
// SM) when a batch's clusters would not all be resident otherwise.
constexpr int kMaxCluster = 16;
constexpr int kTargetSlice = 2048;
constexpr int kMaxSlice = 16384;  // keys per CTA (64 KB of shared memory)
static_assert(kMaxSlice / 512 <= 32, "a lane's keys fit one 32-bit mask");
constexpr int kFusedLoads = 32768;  // capture loads per CTA up to which the cluster scores

struct SelectParams {
  const float* capture;
  int fused;          // keys formed in the select kernel (per-KV-head sum captures)
  uint32_t* keys_ws;  // [B][rows][max_prefix] order-preserving score keys
  const int32_t* prefix_lens;
  int32_t* indices;
  int32_t* counts;
  int32_t* slots;              // NULL, or cache slots beside the indices
  const int32_t* page_table;   // with slots: [batch][max_pages_per_seq]
  int max_pages_per_seq, num_pages;
  int32_t* error_flag;
  int capture_mode, batch, num_q_heads, num_kv_heads, group, max_prefix;
  int top_k, n_sink, n_recent, per_head, cap, rows, slice;
  int n_rows;         // VG_CAPTURE_ALL_ROWS: verify rows per head
  size_t lse_offset;  // VG_CAPTURE_ALL_ROWS: floats before the per-row normalisers
  uint64_t wait_ns;   // a wait longer than this reports VG_DEVERR_TIMEOUT (and goes on)
};

// Order-preserving map float -> uint32 (larger float -> larger key), -0 as +0.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Writes kept position `pos` to list slot `k` and, when slots are asked for,
// its cache slot (physical page * 16 + offset) from the CTA's staged
// page-table entries pt_s (logical pages pt0, pt0 + 1, ...).
__device__ __forceinline__ void put_kept(const SelectParams& p, int32_t* out, int32_t* sout,
                                         const int32_t* pt_s, int pt0, int k, int pos) {
  out[k] = pos;
  if (sout) {
    const int phys = pt_s[pos / 16 - pt0];
    int v = -1;
    if (phys >= 0 && phys < p.num_pages)
      v = phys * 16 + (pos & 15);
    else
      flag_error(p.error_flag, VG_DEVERR_PAGE);
    sout[k] = v;
  }
}

// Score of prefix position j for selection row `row` of sequence b, summed in
// the order documented in vg.h (plain fp32 adds, no reassociation).  The loads
// of one position are all issued before the first add (batches of 16), so a
// score costs one memory round trip per batch rather than one per term.
constexpr int kLoadBatch = 16;

// Per-KV-head sum capture: the row's own KV head, or the sum over KV heads.
__device__ __forceinline__ float group_sum_score(const SelectParams& p, int b, int row, int j) {
  const size_t L = p.max_prefix;
  const float* G = p.capture + (size_t)b * p.num_kv_heads * L + j;
  if (p.per_head) return __ldg(G + (size_t)row * L);
  float acc = 0.f;
  for (int h0 = 0; h0 < p.num_kv_heads; h0 += kLoadBatch) {
    float v[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      v[u] = (h0 + u < p.num_kv_heads) ? __ldg(G + (size_t)(h0 + u) * L) : 0.f;
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (h0 + u < p.num_kv_heads) acc = (h0 + u == 0) ? v[u] : acc + v[u];
  }
  return acc;
}

__device__ __forceinline__ float row_score(const SelectParams& p, int b, int row, int j) {
  const size_t L = p.max_prefix;
  if (p.capture_mode == VG_CAPTURE_ALL_ROWS) {
    // sum of post-softmax weights exp(s - lse) over the rows and query heads
    // of the selection row, in the order (KV head, query head, verify row)
    const int g = p.group, R = p.n_rows;
    const int h0 = p.per_head ? row : 0, h1 = p.per_head ? row + 1 : p.num_kv_heads;
    float acc = 0.f;
    bool first = true;
    for (int q = h0 * g; q < h1 * g; ++q) {
      const size_t base = ((size_t)b * p.num_q_heads + q) * R;
      for (int i0 = 0; i0 < R; i0 += kLoadBatch) {
        float s[kLoadBatch], z[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {  // every load of the batch before any use
          const bool ok = i0 + u < R;
          s[u] = ok ? __ldg(p.capture + (base + i0 + u) * L + j) : 0.f;
          z[u] = ok ? __ldg(p.capture + p.lse_offset + base + i0 + u) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
          if (i0 + u < R) {
            const float w = expf(s[u] - z[u]);
            acc = first ? w : acc + w;
            first = false;
          }
        }
      }
    }
    return acc;
  }
  if (p.capture_mode == VG_CAPTURE_GROUP_SUM) return group_sum_score(p, b, row, j);
  const float* Rw = p.capture + (size_t)b * p.num_q_heads * 2 * L + j;  // [q][2][L]
  const int g = p.group;  // <= 8, so one KV head's 2g terms fit one batch
  const int h0 = p.per_head ? row : 0, h1 = p.per_head ? row + 1 : p.num_kv_heads;
  float acc = 0.f;
  for (int h = h0; h < h1; ++h) {
    float v[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      v[u] = (u < 2 * g) ? __ldg(Rw + (size_t)(2 * h * g + u) * L) : 0.f;
    float G = v[0] + v[1];
#pragma unroll
    for (int qi = 1; qi < kLoadBatch / 2; ++qi)
      if (qi < g) G = G + (v[2 * qi] + v[2 * qi + 1]);
    acc = (h == h0) ? G : acc + G;
  }
  return acc;
}

// Score pass, spread over many CTAs (one position per thread): the fixed-order
// fp32 score of every prefix position, stored as its order-preserving key.
constexpr int kScoreThreads = 256;

__global__ void __launch_bounds__(kScoreThreads) select_score_kernel(const SelectParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int row = blockIdx.y, b = blockIdx.z;
  const int L = p.prefix_lens[b];
  const int j = blockIdx.x * kScoreThreads + threadIdx.x;
  if (L < 0 || L > p.max_prefix || L <= p.n_sink + p.n_recent + p.top_k || j >= L) return;
  p.keys_ws[((size_t)b * p.rows + row) * p.max_prefix + j] = score_key(row_score(p, b, row, j));
}

template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) select_kernel(const SelectParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;

  __shared__ __align__(16) uint32_t hist[2][256];
  __shared__ uint32_t tot_s[256];
  __shared__ int cnt[2];    // this CTA's candidate keys > T and == T
  __shared__ int ctl[5];    // digit, remaining k, gt_before, eq_before, boundary-bin count
  __shared__ int wb[160];
  // dynamic: keys [slice], then the histograms pushed by the cluster's CTAs
  // [pass][CTA][256], the counts they push [CTA] (uint4), and 5 mbarriers
  // counting the pushed bytes (one per pass, one for the counts)
  extern __shared__ __align__(16) uint8_t sel_smem[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel_smem);
  uint32_t* recv = reinterpret_cast<uint32_t*>(sel_smem + ((p.slice * 4 + 15) & ~15));
  uint4* crecv = reinterpret_cast<uint4*>(recv + 4 * kMaxCluster * 256);
  uint64_t* mb = reinterpret_cast<uint64_t*>(crecv + kMaxCluster);
  int32_t* pt_s = reinterpret_cast<int32_t*>(mb + 6);  // page-table entries of the slice

  // programmatic dependent launch: the capture comes from the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lo = rank * p.slice;
  // the slice's page-table entries, for the cache slots of kept positions
  // (loaded while the length is in flight; pages past the row are not read)
  const int pt0 = lo / 16;
  if (p.slots) {
    const int npt = min((lo + p.slice - 1) / 16, p.max_pages_per_seq - 1) - pt0 + 1;
    const int32_t* ptr = p.page_table + (size_t)b * p.max_pages_per_seq + pt0;
    for (int i = tid; i < npt; i += blockDim.x) pt_s[i] = __ldg(ptr + i);
  }
  const int L = p.prefix_lens[b];
  int32_t* out = p.indices + ((size_t)b * p.rows + row) * p.cap;
  int32_t* sout = p.slots ? p.slots + ((size_t)b * p.rows + row) * p.cap : nullptr;
  if (L < 0 || L > p.max_prefix) {  // same decision in every CTA of the cluster
    if (tid == 0 && rank == 0) flag_error(p.error_flag, VG_DEVERR_LENGTH);
    return;
  }
  const int budget = p.n_sink + p.n_recent + p.top_k;
  const int n_loc = max(0, min(lo + p.slice, L) - lo);

  if (L <= budget) {  // every prefix position is kept
    __syncthreads();  // the staged page-table entries are visible
    for (int j = tid; j < n_loc; j += blockDim.x) put_kept(p, out, sout, pt_s, pt0, lo + j, lo + j);
    if (rank == 0) {
      for (int j = L + tid; j < p.cap; j += blockDim.x) {
        out[j] = -1;
        if (sout) sout[j] = -1;
      }
      if (tid == 0) p.counts[(size_t)b * p.rows + row] = L;
    }
    return;
  }
  const int c_lo = p.n_sink, c_hi = L - p.n_recent;  // candidates [c_lo, c_hi)

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&mb[i], 1);
    fence_barrier_init();
    for (int i = 0; i < 4; ++i) mbar_arrive_expect_tx(&mb[i], (uint32_t)C * 1024u);
    mbar_arrive_expect_tx(&mb[4], (uint32_t)C * 16u);
  }
  __syncthreads();
  // once this barrier completes, every CTA's mbarriers are initialised and
  // may receive pushes; its wait comes just before the first push
  cluster_arrive_relaxed();
  bool peers_ready = false;

  if (tid < 256) hist[0][tid] = 0;  // the first pass's histogram
  const int terms = p.per_head ? 1 : p.num_kv_heads;
  if (p.fused && terms <= 8) {
    // four positions per thread at a time (coalesced across the threads),
    // every capture load of the four issued before the first add
    const size_t Lm = p.max_prefix;
    const float* G = p.capture + (size_t)b * p.num_kv_heads * Lm + (p.per_head ? (size_t)row * Lm : 0);
    for (int j0 = tid; j0 < n_loc; j0 += 4 * NT) {
      float v[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
#pragma unroll
        for (int t = 0; t < 8; ++t)
          v[u][t] = (t < terms && j < n_loc) ? __ldg(G + (size_t)t * Lm + lo + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
        float acc = v[u][0];
#pragma unroll
        for (int t = 1; t < 8; ++t)
          if (t < terms) acc = acc + v[u][t];
        if (j < n_loc) keys[j] = score_key(acc);
      }
    }
  } else if (p.fused) {
#pragma unroll 2
    for (int j = tid; j < n_loc; j += blockDim.x)
      keys[j] = score_key(group_sum_score(p, b, row, lo + j));
  } else {
    const uint32_t* kw = p.keys_ws + ((size_t)b * p.rows + row) * p.max_prefix + lo;
#pragma unroll 4
    for (int j = tid; j < n_loc; j += blockDim.x) keys[j] = __ldcg(kw + j);
  }
  __syncthreads();

  // ---- exact top_k-th largest candidate key: 4 passes of 8 bits, MSB first
  uint32_t prefix = 0, mask = 0;
  int krem = p.top_k;
  const int iters = (n_loc + blockDim.x - 1) / blockDim.x;
  if (p.top_k > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* hb = hist[pass & 1];  // zeroed, with a barrier since
      for (int it = 0; it < iters; ++it) {
        const int j = it * blockDim.x + tid;
        const int pos = lo + j;
        const bool in = j < n_loc && pos >= c_lo && pos < c_hi;
        const uint32_t key = in ? keys[j] : 0u;
        const bool v = in && ((key & mask) == prefix);
        const int dig = v ? (int)((key >> shift) & 255u) : -1;
        // lane 0's digit is counted with one ballot (keys crowd into few
        // bins, the first pass's into one or two), the others one by one
        const int d0 = __shfl_sync(0xffffffffu, dig, 0);
        const unsigned same = __ballot_sync(0xffffffffu, dig == d0);
        if (lane == 0 && d0 >= 0) atomicAdd(&hb[d0], (uint32_t)__popc(same));
        if (v && dig != d0) atomicAdd(&hb[dig], 1u);
      }
      __syncthreads();
      if (!peers_ready) {
        cluster_wait_acquire();
        peers_ready = true;
      }
      // push this CTA's histogram (64 pieces of 16 bytes) into slot `rank` of
      // every CTA's region for this pass
      uint32_t* rp = recv + pass * kMaxCluster * 256;
      for (int i = tid; i < 64 * C; i += NT) {
        const int dst = i >> 6, piece = i & 63;
        const uint4 hv = reinterpret_cast<const uint4*>(hb)[piece];
        st_async_v4(mapa_shared(smem_u32(rp + rank * 256 + piece * 4), dst), hv,
                    mapa_shared(smem_u32(&mb[pass]), dst));
      }
      if (tid < 256) {
        mbar_wait_checked(&mb[pass], 0, p.wait_ns, p.error_flag);
        uint32_t v[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) v[c] = c < C ? rp[c * 256 + tid] : 0u;
        uint32_t t = 0;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) t += v[c];
        tot_s[tid] = t;
        hist[(pass + 1) & 1][tid] = 0;  // the next pass's histogram (pushed a pass ago)
      }
      __syncthreads();
      if (tid < 32) {
        // lane owns digits [8 lane, 8 lane + 8); suffix sums run from digit 255 down
        uint32_t own = 0;
#pragma unroll
        for (int d = 0; d < 8; ++d) own += tot_s[8 * lane + d];
        uint32_t incl = own;  // sum over lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
          if (lane + o < 32) incl += t;
        }
        uint32_t above = incl - own;  // keys with a digit above this lane's range
        for (int d = 8 * lane + 7; d >= 8 * lane; --d) {
          const uint32_t t = tot_s[d];
          if (above < (uint32_t)krem && above + t >= (uint32_t)krem) {
            ctl[0] = d;
            ctl[1] = krem - (int)above;
            ctl[4] = (int)t;
          }
          above += t;
        }
      }
      __syncthreads();
      prefix |= (uint32_t)ctl[0] << shift;
      mask |= 255u << shift;
      krem = ctl[1];
      const bool whole_bin = (ctl[4] == krem);  // every key of the boundary bin is kept
      // no barrier here: ctl and tot_s are next written after the next
      // pass's first barrier
      if (whole_bin) break;  // same decision in every CTA (same cluster-wide histogram)
    }
  }
  // Keys are compared on the bits fixed so far (all 32 unless the search
  // stopped early because the whole boundary bin is kept): (key & mask) > T
  // is kept, and krem of the (key & mask) == T keys are kept, lowest
  // positions first.
  const uint32_t T = prefix;

  // ---- kept keys: every (key & mask) > T, and the first krem with
  // (key & mask) == T in position order, written to their sorted slots.
  // Warp w owns the contiguous key range [w * 32 * per, (w + 1) * 32 * per)
  // of this CTA's slice, read 32 at a time; counts go through ballots, and
  // the warps are ordered by one exclusive scan per quantity.
  const int per = (n_loc + NT - 1) / NT;  // keys per lane
  constexpr int kWarps = NT / 32;
  const int wid = tid >> 5;
  const int wbase = wid * 32 * per;
  const unsigned lt_mask = (1u << lane) - 1u;
  int gt_w = 0, eq_w = 0;
  if (p.top_k > 0) {
    for (int i = 0; i < per; ++i) {
      const int j = wbase + i * 32 + lane;
      const int pos = lo + j;
      const bool in = j < n_loc && pos >= c_lo && pos < c_hi;
      const uint32_t k = in ? (keys[j] & mask) : 0u;
      gt_w += __popc(__ballot_sync(0xffffffffu, in && k > T));
      eq_w += __popc(__ballot_sync(0xffffffffu, in && k == T));
    }
  }
  if (lane == 0) {
    wb[wid] = eq_w;
    wb[32 + wid] = gt_w;
  }
  __syncthreads();
  if (wid == 0) {  // exclusive scan of the per-warp == T counts, totals
    const int e = lane < kWarps ? wb[lane] : 0, gtv = lane < kWarps ? wb[32 + lane] : 0;
    int incl = e, gsum = gtv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
      gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
    }
    wb[64 + lane] = incl - e;
    if (lane == 31) {
      cnt[0] = gsum;
      cnt[1] = incl;
    }
  }
  __syncthreads();
  if (!peers_ready) {
    cluster_wait_acquire();
    peers_ready = true;
  }
  if (tid < C)  // this CTA's totals into slot `rank` of CTA tid
    st_async_v4(mapa_shared(smem_u32(&crecv[rank]), tid),
                make_uint4((uint32_t)cnt[0], (uint32_t)cnt[1], 0u, 0u),
                mapa_shared(smem_u32(&mb[4]), tid));
  // every push of this CTA is issued; the wait at the end keeps every CTA
  // resident until all of them are
  cluster_arrive_release();
  if (tid < 32) {  // lane c takes CTA c's counts; sum over the lower ranks
    mbar_wait_checked(&mb[4], 0, p.wait_ns, p.error_flag);
    int gv = 0, ev = 0;
    if (lane < rank) {
      gv = (int)crecv[lane].x;
      ev = (int)crecv[lane].y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gv += __shfl_xor_sync(0xffffffffu, gv, o);
      ev += __shfl_xor_sync(0xffffffffu, ev, o);
    }
    if (lane == 0) {
      ctl[2] = gv;
      ctl[3] = ev;
    }
  }
  __syncthreads();

  if (p.top_k > 0) {
    const int gt_before = ctl[2], eq_before = ctl[3];
    const int eq_rank0 = eq_before + wb[64 + wid];  // rank of this warp's first == T key
    int sel_w = 0, eq_run = eq_rank0;
    uint32_t selbits = 0;  // bit i: this lane's key of round i is kept (per <= 32)
    for (int i = 0; i < per; ++i) {
      const int j = wbase + i * 32 + lane;
      const int pos = lo + j;
      const bool in = j < n_loc && pos >= c_lo && pos < c_hi;
      const uint32_t k = in ? (keys[j] & mask) : 0u;
      const bool is_eq = in && k == T;
      const unsigned eb = __ballot_sync(0xffffffffu, is_eq);
      const bool sel = (in && k > T) || (is_eq && eq_run + __popc(eb & lt_mask) < krem);
      selbits |= (uint32_t)sel << i;
      sel_w += __popc(__ballot_sync(0xffffffffu, sel));
      eq_run += __popc(eb);
    }
    if (lane == 0) wb[96 + wid] = sel_w;
    __syncthreads();
    if (wid == 0) {
      const int v = lane < kWarps ? wb[96 + lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      wb[128 + lane] = incl - v;
    }
    __syncthreads();
    const int slot0 = p.n_sink + gt_before + min(eq_before, krem) + wb[128 + wid];
    int sel_run = 0;
    for (int i = 0; i < per; ++i) {
      const bool sel = (selbits >> i) & 1u;
      const unsigned sbal = __ballot_sync(0xffffffffu, sel);
      if (sel)
        put_kept(p, out, sout, pt_s, pt0, slot0 + sel_run + __popc(sbal & lt_mask),
                 lo + wbase + i * 32 + lane);
      sel_run += __popc(sbal);
    }
  }
  // sink and recent positions, by the CTA whose slice holds them
  for (int j = tid; j < n_loc; j += blockDim.x) {
    const int pos = lo + j;
    if (pos < p.n_sink)
      put_kept(p, out, sout, pt_s, pt0, pos, pos);
    else if (pos >= L - p.n_recent)
      put_kept(p, out, sout, pt_s, pt0, p.n_sink + p.top_k + (pos - (L - p.n_recent)), pos);
  }
  if (rank == 0) {
    for (int j = budget + tid; j < p.cap; j += blockDim.x) {
      out[j] = -1;
      if (sout) sout[j] = -1;
    }
    if (tid == 0) p.counts[(size_t)b * p.rows + row] = budget;
  }
  cluster_wait_acquire();
}

size_t select_smem_bytes(int slice) {
  return align_up((size_t)slice * 4, 16) + 4 * kMaxCluster * 256 * 4 + kMaxCluster * 16 + 6 * 8 +
         align_up(((size_t)slice / 16 + 2) * 4, 16);
}

template <int NT>
bool set_select_attributes_nt() {
  return cudaFuncSetAttribute(select_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)select_smem_bytes(kMaxSlice)) == cudaSuccess &&
         cudaFuncSetAttribute(select_kernel<NT>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                              1) == cudaSuccess;
}

bool set_select_attributes() {
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return true;
  if (!set_select_attributes_nt<1024>() || !set_select_attributes_nt<512>()) return false;
  if (dev < 64) done[dev] = true;
  return true;
}

// Clusters of C CTAs of NT threads (slice of `slice` keys each) the device
// holds at once.
int select_max_clusters(int C, int slice, int NT) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, int> memo;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, C, slice, NT);
  {
    std::lock_guard<std::mutex> g(mu);
    const auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = select_smem_bytes(slice);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e =
      NT == 512 ? cudaOccupancyMaxActiveClusters(&n, select_kernel<512>, &cfg)
                : cudaOccupancyMaxActiveClusters(&n, select_kernel<1024>, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> g(mu);
  memo[key] = n;
  return n;
}

// Cluster size, keys per CTA and threads per CTA for `clusters` selection
// rows of max_prefix positions: slices of about kTargetSlice keys in
// clusters of up to kMaxCluster CTAs of 1024 threads.  While the rows'
// clusters would not all be resident at once (a second wave costs a whole
// selection): CTAs of 512 threads (two per SM), else clusters halved, as
// long as the slice still fits.
bool select_shape(int max_prefix, long long clusters, int* C, int* slice, int* nt) {
  int c = 1;
  while (c < kMaxCluster && ceil_div(max_prefix, c) > kTargetSlice) c *= 2;
  int s = align_up(ceil_div(max_prefix, c), 4);
  if (s > kMaxSlice) return false;
  int t = 1024;
  while (c > 1 && clusters > 1) {
    if (clusters <= select_max_clusters(c, s, 1024)) break;
    if (clusters <= select_max_clusters(c, s, 512)) {
      t = 512;
      break;
    }
    const int s2 = align_up(ceil_div(max_prefix, c / 2), 4);
    if (s2 > kMaxSlice) break;
    c /= 2;
    s = s2;
  }
  *C = c;
  *slice = s;
  *nt = t;
  return true;
}

// Whether the cluster forms the keys itself (no score kernel): per-KV-head sum
// captures whose CTAs have few loads to issue (up to kFusedLoads each);
// otherwise the score kernel spreads the loads over the whole device.
bool select_fused(int capture_mode, int per_head, int num_kv_heads, int slice) {
  return capture_mode == VG_CAPTURE_GROUP_SUM &&
         (long long)(per_head ? 1 : num_kv_heads) * slice <= kFusedLoads;
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" size_t vg_select_workspace_bytes(int batch, int num_kv_heads, int max_prefix,
                                            int per_head) {
  if (batch <= 0 || num_kv_heads <= 0 || max_prefix <= 0) return 0;
  const size_t rows = per_head ? num_kv_heads : 1;
  return align_up((size_t)batch * rows * max_prefix * 4, 256);
}

static vg_status select_impl(const float* capture, int capture_mode, int n_rows,
                             const int32_t* prefix_lens, int batch, int num_q_heads,
                             int num_kv_heads, int max_prefix, int top_k, int n_sink,
                             int n_recent, int per_head, int32_t* indices, int32_t* counts,
                             int cap, const vg_paged_kv* kv, int32_t* slots, void* workspace,
                             size_t workspace_bytes, int32_t* error_flag, cudaStream_t stream);

extern "C" int vg_select_launches(int capture_mode, int batch, int num_kv_heads, int max_prefix,
                                  int per_head) {
  if (batch <= 0 || num_kv_heads <= 0 || max_prefix <= 0) return 0;
  if (capture_mode == VG_CAPTURE_ALL_SUM) capture_mode = VG_CAPTURE_GROUP_SUM;
  if (capture_mode != VG_CAPTURE_GROUP_SUM && capture_mode != VG_CAPTURE_ROWS &&
      capture_mode != VG_CAPTURE_ALL_ROWS)
    return 0;
  int C, slice, nt;
  if (!select_shape(max_prefix, 1, &C, &slice, &nt) || !set_select_attributes()) return 0;
  select_shape(max_prefix, (long long)batch * (per_head ? num_kv_heads : 1), &C, &slice, &nt);
  return select_fused(capture_mode, per_head, num_kv_heads, slice) ? 1 : 2;
}

extern "C" vg_status vg_select_kv(const float* capture, int capture_mode,
                                  const int32_t* prefix_lens, int batch, int num_q_heads,
                                  int num_kv_heads, int max_prefix, int top_k, int n_sink,
                                  int n_recent, int per_head, int32_t* indices, int32_t* counts,
                                  int cap, const vg_paged_kv* kv, int32_t* slots,
                                  void* workspace, size_t workspace_bytes, int32_t* error_flag,
                                  cudaStream_t stream) {
  if (capture_mode == VG_CAPTURE_ALL_SUM) capture_mode = VG_CAPTURE_GROUP_SUM;  // same layout
  if (capture_mode != VG_CAPTURE_GROUP_SUM && capture_mode != VG_CAPTURE_ROWS)
    return VG_ERR_INVALID_ARGUMENT;
  return select_impl(capture, capture_mode, 0, prefix_lens, batch, num_q_heads, num_kv_heads,
                     max_prefix, top_k, n_sink, n_recent, per_head, indices, counts, cap, kv,
                     slots, workspace, workspace_bytes, error_flag, stream);
}

extern "C" vg_status vg_select_kv_weights(const float* capture, int n_rows,
                                          const int32_t* prefix_lens, int batch, int num_q_heads,
                                          int num_kv_heads, int max_prefix, int top_k, int n_sink,
                                          int n_recent, int per_head, int32_t* indices,
                                          int32_t* counts, int cap, const vg_paged_kv* kv,
                                          int32_t* slots, void* workspace,
                                          size_t workspace_bytes, int32_t* error_flag,
                                          cudaStream_t stream) {
  if (n_rows <= 0 || n_rows > 16) return VG_ERR_INVALID_ARGUMENT;
  return select_impl(capture, VG_CAPTURE_ALL_ROWS, n_rows, prefix_lens, batch, num_q_heads,
                     num_kv_heads, max_prefix, top_k, n_sink, n_recent, per_head, indices, counts,
                     cap, kv, slots, workspace, workspace_bytes, error_flag, stream);
}

static vg_status select_impl(const float* capture, int capture_mode, int n_rows,
                             const int32_t* prefix_lens, int batch, int num_q_heads,
                             int num_kv_heads, int max_prefix, int top_k, int n_sink,
                             int n_recent, int per_head, int32_t* indices, int32_t* counts,
                             int cap, const vg_paged_kv* kv, int32_t* slots, void* workspace,
                             size_t workspace_bytes, int32_t* error_flag, cudaStream_t stream) {
  if (!capture || !prefix_lens || !indices || !counts || batch <= 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || max_prefix <= 0 || top_k < 0 || n_sink < 0 || n_recent < 0 || cap <= 0)
    return VG_ERR_INVALID_ARGUMENT;
  if (slots) {  // cache slots need the page table of the cache the positions index
    const vg_status st = check_paged_kv(kv);
    if (st != VG_OK) return st;
    if (kv->num_kv_heads != num_kv_heads || ceil_div(max_prefix, kPageSize) > kv->max_pages_per_seq)
      return VG_ERR_INVALID_ARGUMENT;
  }
  if (num_q_heads % num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads / num_kv_heads > 8) return VG_ERR_UNSUPPORTED;
  const long long budget = (long long)n_sink + n_recent + top_k;
  if (cap < std::min<long long>(max_prefix, budget)) return VG_ERR_INVALID_ARGUMENT;
  int C, slice, nt;
  if (!select_shape(max_prefix, 1, &C, &slice, &nt)) return VG_ERR_UNSUPPORTED;
  const size_t ws_need = vg_select_workspace_bytes(batch, num_kv_heads, max_prefix, per_head);
  if (!workspace || workspace_bytes < ws_need) return VG_ERR_WORKSPACE_TOO_SMALL;
  if (!set_select_attributes()) return VG_ERR_LAUNCH;
  select_shape(max_prefix, (long long)batch * (per_head ? num_kv_heads : 1), &C, &slice, &nt);

  SelectParams p;
  p.capture = capture;
  p.keys_ws = static_cast<uint32_t*>(workspace);
  p.prefix_lens = prefix_lens;
  p.indices = indices;
  p.counts = counts;
  p.slots = slots;
  p.page_table = slots ? kv->page_table : nullptr;
  p.max_pages_per_seq = slots ? kv->max_pages_per_seq : 0;
  p.num_pages = slots ? kv->num_pages : 0;
  p.error_flag = error_flag;
  p.capture_mode = capture_mode;
  p.n_rows = n_rows;
  p.lse_offset = (size_t)batch * num_q_heads * (n_rows > 0 ? n_rows : 1) * max_prefix;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.max_prefix = max_prefix;
  p.top_k = top_k;
  p.n_sink = n_sink;
  p.n_recent = n_recent;
  p.per_head = per_head ? 1 : 0;
  p.cap = cap;
  p.wait_ns = wait_report_ns();
  p.rows = per_head ? num_kv_heads : 1;
  p.slice = slice;
  p.fused = select_fused(capture_mode, per_head, num_kv_heads, slice) ? 1 : 0;

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t scfg = {};
  scfg.gridDim = dim3(ceil_div(max_prefix, kScoreThreads), p.rows, batch);
  scfg.blockDim = dim3(kScoreThreads, 1, 1);
  scfg.stream = stream;
  scfg.attrs = pdl;
  scfg.numAttrs = 1;
  if (!p.fused && cudaLaunchKernelEx(&scfg, select_score_kernel, p) != cudaSuccess)
    return VG_ERR_LAUNCH;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, p.rows, batch);
  cfg.blockDim = dim3(nt, 1, 1);
  cfg.dynamicSmemBytes = select_smem_bytes(slice);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = nt == 512 ? cudaLaunchKernelEx(&cfg, select_kernel<512>, p)
                                  : cudaLaunchKernelEx(&cfg, select_kernel<1024>, p);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}
