// Verification attention with Collect-2-Query capture (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" / Figure 6: the verify pass is full attention of the k+1 block
// rows over the whole cache, and it writes only two pre-softmax logit rows
// (first draft token, bonus token) for the prefix positions.
//
// Design (a unit of work is one KV split of one KV head of one sequence; one
// CTA per unit, or, when the units outnumber the SMs, one persistent CTA per
// SM walking a unit list built on the device from the lengths):
//  * The g query heads x R verify rows of one KV head are packed into the M
//    dimension of 5th-generation tensor-core MMAs (tcgen05.mma, bf16 in, fp32
//    accumulators in tensor memory, M padded to 128), so every K/V page is
//    read from HBM once per KV head.  Row order in M: [row 0 of each
//    head][row k of each head][rows 1..k-1].
//  * A producer warp streams 128-position tiles (8 pages) of K and V into a
//    shared-memory ring with 4-D TMA loads (128-byte swizzle, evict-first L2
//    policy); the swizzled tiles are the tensor cores' K-major (K) and
//    MN-major (V) B operands as they land.  Q and P, the A operands, live in
//    tensor memory, so shared memory holds only the ring.
//  * One thread issues, whichever is ready first, S = Q K^T for the next tile
//    into one of two TMEM buffers, or O += P V for the oldest tile whose P is
//    written, into a TMEM accumulator; the tensor cores compute the next
//    scores during softmax and a ring stage is released as soon as its P V
//    has run.  Completion is signalled through tcgen05.commit on mbarriers;
//    every wait is bounded.
//  * Softmax warps hold one packed row per lane (tcgen05.ld), so row maxima
//    and sums need no shuffles; the exponent reference moves only when a row
//    maximum grows by more than 2^32, and O is then rescaled in TMEM.  P goes
//    back to tensor memory as bf16 pairs.
//  * Capture epilogue (from the softmax warps' registers): the Collect-2 rows
//    or their per-KV-head sum in a fixed order, or the Collect-All column
//    sums (butterfly over each warp's rows, then warps in order).
//  * Splits over the KV length write fp32 partials (O, m, l) to the
//    workspace; a small merge kernel, one CTA per (output row, KV head,
//    sequence), combines them.  It is chained with programmatic dependent
//    launch, so its launch overlaps the verify grid.
#include <climits>
#include <mutex>

#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kMaxSplits = 256;

struct VerifyParams {
  const __nv_bfloat16* q;
  const int32_t* prefix_lens;
  const int32_t* page_table;
  __nv_bfloat16* out;
  float* capture;
  float* part_o;      // [B][Hkv][splits][M][HD]
  float* part_ml;     // [B][Hkv][splits][M][2]
  int32_t* error_flag;
  int batch, n_rows, num_q_heads, num_kv_heads, group, m_rows, m_tiles;
  int max_prefix, max_pages_per_seq, num_pages;
  int capture_mode, splits, tiles_per_split, stages, groups;
  size_t lse_offset;  // VG_CAPTURE_ALL_ROWS: floats before the per-row normalisers
  // sparse verification: per sequence, the union of the rows' blocks
  int32_t* u_pages;    // [B][u_max] logical pages, ascending
  uint32_t* u_masks;   // [B][u_max] bit i: verify row i selected the page
  int32_t* u_count;    // [B]
  int u_max;
  int persistent;      // dense: CTAs walk a list of units (gridDim.x CTAs in all)
  uint64_t wait_ns;    // a wait longer than this reports VG_DEVERR_TIMEOUT (and goes on)
  float scale, scale_log2;
};

// Row m of the packed M dimension -> (verify row i, head within group qi).
__device__ __forceinline__ void row_of(int m, int g, int R, int& i, int& qi) {
  if (m < g) {
    i = 0;
    qi = m;
  } else if (m < 2 * g) {
    i = R - 1;
    qi = m - g;
  } else {
    const int r = m - 2 * g;
    i = 1 + r / g;
    qi = r - (r / g) * g;
  }
}

// Thread roles: warps 0..3 are softmax warps (warp w reads TMEM lanes
// [32 w, 32 w + 32)), warp 4 is the TMA producer, warp 5 issues the
// tensor-core MMAs and owns the tensor memory.
//
// Tiles are 128 positions (8 pages), so one S = Q K^T is 8 MMAs of N = 128
// and one O += P V is 8 MMAs of K = 16 positions: a single issuing thread
// keeps up with HBM.  P is written back into its own S buffer (bf16 pairs in
// the first 64 columns), which is reused by the next-but-one S only after
// that P V has completed.
//
// The packed rows are replicated into CS = 4 (M <= 32), 2 (M <= 64) or 1
// copies of the 128-row MMA tile (the padding is free): copy c occupies TMEM
// lanes [c * 128 / CS, ...), and its warps run an independent online softmax
// over columns [c * 128 / CS, (c + 1) * 128 / CS) of every tile, with P zero
// elsewhere.  Each copy accumulates its own (m, l, O) over a share of the
// positions and the copies are merged once at the end, so the per-tile
// softmax work of a warp shrinks by CS.
constexpr int kVTile = 128;            // positions per tile = 8 pages
constexpr int kVerifyThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kMPad = 128;             // UMMA M
// Tensor memory columns: S double buffer (2 x 128 fp32; P aliases its first
// 64 columns), O (<= 128 fp32), Q as the A operand (<= 64 bf16-pair columns).
constexpr int kTmemCols = 512;
constexpr int kSCol = 0, kOCol = 2 * kVTile, kQCol = kOCol + 128;
// Q is double-buffered (a persistent CTA writes the next unit's Q while the
// current unit's last scores are still being read): buffer i at kQCol + i *
// HD / 2 (bf16 pairs), which ends at column 512 for head_dim 128.
// O and l follow a new row maximum only past a 2^32 growth: until then P is
// taken relative to the older reference, so one entry of P is at most 2^32
// (exact range in bf16 and fp32, same relative precision) and l, O stay far
// below the fp32 range (<= 2^32 per position of a split).  A rescale must
// wait for the last P.V, so it is kept off the common path.
constexpr float kRescaleLog2 = 32.f;
constexpr int kChunk = 32;             // columns a softmax pass holds in registers
constexpr int kMaxPersistBatch = 64;   // sequences a persistent CTA's unit table holds
constexpr int kCapStride = kChunk + 4; // floats per staged capture row (16-byte rows, no bank conflicts)

template <int HD>
struct VerifyLayout {
  static constexpr int kTileBytes = kVTile * HD * 2;   // one of K / V: [HD/64][128 pos][128 B]
  static constexpr int kHalfBytes = kVTile * 128;      // one 64-dim half of a tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kCapFloats = 4 * 16 * kCapStride;  // per-warp Collect-2 staging
  static constexpr int kAllFloats = 2 * 4 * kVTile;       // Collect-All partials [slot][warp]
  static constexpr int kBars = 15;                        // besides the ring's 4 per stage
  static constexpr int kSliceMax = 1024;                  // sparse: union pages of one split
  static constexpr int kUnitTab = 4 * kMaxPersistBatch + 2; // persistent: per-sequence unit table
  static size_t bytes(int stages) {
    return 1024 + (size_t)stages * kStageBytes + (size_t)(kCapFloats + kAllFloats) * 4 +
           (size_t)kSliceMax * 8 + (4 * (size_t)stages + kBars) * 8 + 16 + kUnitTab * 4;
  }
};

struct VerifyBars {
  uint64_t *kfull, *vfull, *kempty, *empty, *s_full, *p_full, *capfull, *capfree, *drain, *qfull;
  int stages;
};

// Q rows of a unit for one softmax warp's 32 TMEM lanes (the A operand):
// lane c * RPC + m holds packed row m of copy c, every other lane zero (its
// logits are exactly zero).  load_q reads this lane's row into registers,
// store_q writes them to tensor-memory buffer `buf`.
template <int HD>
__device__ __forceinline__ void load_q(const VerifyParams& p, int b, int h, int warp, int lane,
                                       uint4 (&x)[HD / 8]) {
  const int M = p.m_rows;
  const int CS = M <= 32 ? 4 : (M <= 64 ? 2 : 1);
  const int RPC = kMPad / CS;
  const int row = 32 * warp + lane;
  const int cp = row / RPC, mm = row - cp * RPC;
  const uint4* src = nullptr;
  if (b >= 0 && cp < CS && mm < M) {
    int i, qi;
    row_of(mm, p.group, p.n_rows, i, qi);
    src = reinterpret_cast<const uint4*>(
        p.q + ((size_t)(b * p.n_rows + i) * p.num_q_heads + h * p.group + qi) * HD);
  }
#pragma unroll
  for (int k = 0; k < HD / 8; ++k) x[k] = src ? src[k] : make_uint4(0, 0, 0, 0);
}

template <int HD>
__device__ __forceinline__ void store_q(uint32_t tmem, int buf, int warp, const uint4 (&xq)[HD / 8]) {
  const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16) + kQCol + buf * (HD / 2);
#pragma unroll
  for (int half = 0; half < HD / 64; ++half) {
    uint4 x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = xq[half * 8 + k];
    uint32_t v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[4 * k] = x[k].x;
      v[4 * k + 1] = x[k].y;
      v[4 * k + 2] = x[k].z;
      v[4 * k + 3] = x[k].w;
    }
    tmem_st32u(trow + half * 32, v);
  }
  tmem_st_wait();
  tc_fence_before();
}

template <int HD>
__device__ __forceinline__ void write_q(const VerifyParams& p, uint32_t tmem, int buf, int b,
                                        int h, int warp, int lane) {
  uint4 x[HD / 8];
  load_q<HD>(p, b, h, warp, lane, x);
  store_q<HD>(tmem, buf, warp, x);
}

// Softmax warp of a copy for one unit of work (a split of one KV head of one
// sequence); COLS = 128 / CS columns of each tile, handled in chunks of 32
// (two passes over TMEM when COLS > 32: maximum, then P).  `tbase` is the
// CTA's count of tiles before this unit: ring stages, S/P buffers and their
// barrier phases follow that running count across units.  When the CTA has a
// next unit (nb >= 0), its Q goes to tensor-memory buffer qbuf_next (arrival
// on qfull[qbuf_next]) before this unit's epilogue, so that the tensor cores
// can start its scores meanwhile.  The copies' merge goes through `scratch`
// (the capture staging area, idle by then) one 32-column chunk at a time, or
// through the ring all at once when `ring` is given (a CTA's only unit: no
// load is in flight at its epilogue).
template <int HD, int COLS, int CM, bool SP>
__device__ __forceinline__ void verify_softmax(const VerifyParams& p, const VerifyBars& bars,
                                               float* scratch, float* ring, float* cap_s,
                                               float* all_s,
                                               const int32_t* sl_page, const uint32_t* sl_mask,
                                               int sl_n, uint32_t tmem, int b, int h, int split,
                                               int t0, int ntiles, int L, int tbase, int& hs,
                                               int nb, int nh, int qbuf_next, int warp, int lane) {
  constexpr int CS = kVTile / COLS;       // copies
  constexpr int QC = 4 / CS;              // warps (TMEM quadrants) per copy
  constexpr int RPC = 32 * QC;            // rows per copy
  constexpr int NCH = COLS / kChunk;      // chunks per tile
  const int g = p.group, R = p.n_rows, M = p.m_rows;
  const int NS = (M + 31) >> 5;
  const int c = warp / QC, wq = warp % QC;  // copy, warp within the copy
  const int nwc = (CS == 1) ? NS : QC;      // warps of this copy holding rows
  const int col0 = c * COLS;
  const int m = wq * 32 + lane;             // packed row of this lane
  int lim = -1, ri = 0, rq = 0;             // last attended position, verify row, head
  if (m < M) {
    row_of(m, g, R, ri, rq);
    lim = L + ri;
  }
  const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
  // capture mode CM is a template parameter: each mode is its own kernel
  const bool cap_two = wq == 0 && (CM == VG_CAPTURE_GROUP_SUM || CM == VG_CAPTURE_ROWS);
  constexpr bool cap_all = CM == VG_CAPTURE_ALL_SUM;
  constexpr bool cap_rows = CM == VG_CAPTURE_ALL_ROWS;
  const int s1 = (R > 1) ? g : 0;           // packed row of "row k, head 0"
  const int nrows = (R > 1) ? 2 * g : g;    // captured rows
  float* cap_w = cap_s + warp * 16 * kCapStride;
  const int stages = bars.stages;
  float m_used = -INFINITY, lsum = 0.f;
  bool live = true;

  for (int lt = 0; lt < ntiles; ++lt) {
    const int T = tbase + lt;  // the CTA's running tile index
    const int sb = T & 1, u = T >> 1;
    const int tile_pos = (t0 + lt) * kVTile;
    const uint32_t sbuf = trow + kSCol + sb * kVTile;
    if (live && !mbar_wait_checked(&bars.s_full[sb], u & 1, p.wait_ns, p.error_flag)) live = false;
    tc_fence_after();
    const int cpos = tile_pos + col0;  // position of this warp's first column
    const int rem = lim - cpos;        // last attended column of this row among the warp's
    // sparse: which of this warp's columns the row attends (one bit per column
    // of each 32-column chunk); the tile's 8 slots hold union pages
    uint32_t vbits[NCH];
    if constexpr (SP) {
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        uint32_t bits = 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int slot = lt * (kVTile / kPageSize) + (col0 + k * kChunk) / kPageSize + half;
          if (m < M && slot < sl_n && sl_page[slot] >= 0) {
            const int pos0 = sl_page[slot] * kPageSize;
            const bool sel = (sl_mask[slot] >> ri) & 1u;
#pragma unroll
            for (int c = 0; c < kPageSize; ++c) {
              const int pos = pos0 + c;
              if (pos < L ? sel : pos <= lim) bits |= 1u << (half * kPageSize + c);
            }
          }
        }
        vbits[k] = bits;
      }
    }

    // -------- pass 1: capture (prefix positions) and the row maximum
    // (dense: a tile whose columns every row of the warp attends skips the
    // per-column masks; padding lanes hold zero scores and are never read)
    const bool full_tile = !SP && __all_sync(0xffffffffu, m >= M || rem >= COLS - 1);
    float s[kChunk];
    float call[NCH];                   // Collect-All column sums of this lane
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      tmem_ld32(sbuf + col0 + k * kChunk, s);
      const int kpos = cpos + k * kChunk;
      if (kpos < L) {
        if (cap_rows && m < M) {  // every row, raw, for weight statistics
          float* dst = p.capture + (((size_t)b * p.num_q_heads + h * g + rq) * R + ri) * p.max_prefix + kpos;
          const int nj = min(kChunk, L - kpos);
          if (nj == kChunk && (p.max_prefix & 3) == 0) {
#pragma unroll
            for (int j = 0; j < kChunk; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(s[j] * p.scale, s[j + 1] * p.scale, s[j + 2] * p.scale, s[j + 3] * p.scale);
          } else {
#pragma unroll
            for (int j = 0; j < kChunk; ++j)
              if (j < nj) dst[j] = s[j] * p.scale;
          }
        }
        if (cap_two) {
          if (lane < nrows) {
#pragma unroll
            for (int j = 0; j < kChunk; j += 4)
              *reinterpret_cast<float4*>(cap_w + lane * kCapStride + j) =
                  make_float4(s[j] * p.scale, s[j + 1] * p.scale, s[j + 2] * p.scale, s[j + 3] * p.scale);
          }
          __syncwarp();
          if (kpos + lane < L) {
            if (CM == VG_CAPTURE_GROUP_SUM) {
              float G = cap_w[lane] + cap_w[s1 * kCapStride + lane];
              for (int qi = 1; qi < g; ++qi)
                G = G + (cap_w[qi * kCapStride + lane] + cap_w[(s1 + qi) * kCapStride + lane]);
              p.capture[((size_t)b * p.num_kv_heads + h) * p.max_prefix + kpos + lane] = G;
            } else {
              for (int rr = 0; rr < nrows; ++rr) {
                const int qi = rr < g ? rr : rr - g;
                const size_t base = ((size_t)b * p.num_q_heads + h * g + qi) * 2;
                const float v = cap_w[rr * kCapStride + lane];
                p.capture[(base + (rr < g ? 0 : 1)) * p.max_prefix + kpos + lane] = v;
                if (R == 1) p.capture[(base + 1) * p.max_prefix + kpos + lane] = v;
              }
            }
          }
          __syncwarp();
        }
        if (cap_all) {
          // column sums over this warp's 32 rows (rows >= M hold zeros) by
          // recursive halving: this lane ends with column `lane` of the chunk
          float cv[kChunk];
#pragma unroll
          for (int j = 0; j < kChunk; ++j) cv[j] = s[j] * p.scale;
#pragma unroll
          for (int step = 0; step < 5; ++step) {
            const int d = 16 >> step, w = (kChunk / 2) >> step;
            const bool up = (lane & d) != 0;
#pragma unroll
            for (int j = 0; j < w; ++j) {
              const float send = up ? cv[j] : cv[j + w];
              const float recv = __shfl_xor_sync(0xffffffffu, send, d);
              cv[j] = (up ? cv[j + w] : cv[j]) + recv;
            }
          }
          call[k] = cv[0];
        }
      }
      if (full_tile) {  // every column attended: a tree, no masks
        float t[kChunk / 2];
#pragma unroll
        for (int j = 0; j < kChunk / 2; ++j) t[j] = fmaxf(s[j], s[j + kChunk / 2]);
#pragma unroll
        for (int w = kChunk / 4; w > 0; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
        mx = fmaxf(mx, t[0]);
      } else {
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (SP ? ((vbits[k] >> j) & 1u) != 0 : k * kChunk + j <= rem) mx = fmaxf(mx, s[j]);
      }
    }
    if (cap_all && cpos < L) {
      // across the copy's warps, in order, through shared memory
      // hs counts this copy's handshakes in the CTA (tiles past the prefix
      // have none), so that the barrier phases hold across units
      const int slot = hs & 1;
      const int cb = c * 2 + slot;  // this copy's handshake barrier of the slot
      float* part = all_s + slot * 4 * kVTile;
      if (wq != 0) {
        if (hs >= 2 && live &&
            !mbar_wait_checked(&bars.capfree[cb], ((hs >> 1) - 1) & 1, p.wait_ns, p.error_flag))
          live = false;
#pragma unroll
        for (int k = 0; k < NCH; ++k) part[warp * kVTile + k * kChunk + lane] = call[k];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.capfull[cb]);
      } else {
        if (nwc > 1 && live &&
            !mbar_wait_checked(&bars.capfull[cb], (hs >> 1) & 1, p.wait_ns, p.error_flag))
          live = false;
        float* dst = p.capture + ((size_t)b * p.num_kv_heads + h) * p.max_prefix + cpos;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
          float a = call[k];
          for (int w2 = 1; w2 < nwc; ++w2) a = a + part[(warp + w2) * kVTile + k * kChunk + lane];
          if (cpos + k * kChunk + lane < L) dst[k * kChunk + lane] = a;
        }
        __syncwarp();
        if (nwc > 1 && lane == 0) mbar_arrive(&bars.capfree[cb]);
      }
      ++hs;
    }

    // -------- online softmax (base 2) with a lazily moved reference
    mx *= p.scale_log2;  // scale > 0: the max commutes with it; -inf stays -inf
    const bool need = mx > m_used + kRescaleLog2;
    if (__any_sync(0xffffffffu, need)) {
      const float mn = need ? mx : m_used;
      const float corr = (mn == -INFINITY) ? 1.f : ex2(m_used - mn);
      lsum *= corr;
      if (lt > 0) {  // O holds P(0..t-1) V: wait for the last P.V, then scale the row
        const int pst = (T - 1) % stages;
        if (live &&
            !mbar_wait_checked(&bars.empty[pst], ((T - 1) / stages) & 1, p.wait_ns, p.error_flag))
          live = false;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          tmem_ld32(trow + kOCol + cc * 32, o);
          float o16[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) o16[k] = o[k] * corr;
          tmem_st16(trow + kOCol + cc * 32, o16);
#pragma unroll
          for (int k = 0; k < 16; ++k) o16[k] = o[16 + k] * corr;
          tmem_st16(trow + kOCol + cc * 32 + 16, o16);
        }
        tmem_st_wait();
      }
      m_used = mn;
    }
    const float nref = -safe_ref(m_used);

    // -------- pass 2: P = 2^(s - m) as bf16 pairs into the first 64 columns
    // of this S buffer; the 16-column groups outside this warp's share are zero
    uint32_t pk[NCH][kChunk / 2];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      if (NCH > 1) tmem_ld32(sbuf + col0 + k * kChunk, s);
      if (full_tile) {  // no masks; the row sum as a tree
        float ps[kChunk / 2];
#pragma unroll
        for (int j = 0; j < kChunk / 2; ++j) {
          const float p0 = ex2(fmaf(s[2 * j], p.scale_log2, nref));
          const float p1 = ex2(fmaf(s[2 * j + 1], p.scale_log2, nref));
          ps[j] = p0 + p1;
          pk[k][j] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int w = kChunk / 4; w > 0; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) ps[j] += ps[j + w];
        lsum += ps[0];
      } else {
#pragma unroll
        for (int j = 0; j < kChunk / 2; ++j) {
          const int jj = k * kChunk + 2 * j;
          const bool v0 = SP ? ((vbits[k] >> (2 * j)) & 1u) != 0 : jj <= rem;
          const bool v1 = SP ? ((vbits[k] >> (2 * j + 1)) & 1u) != 0 : jj + 1 <= rem;
          const float p0 = v0 ? ex2(fmaf(s[2 * j], p.scale_log2, nref)) : 0.f;
          const float p1 = v1 ? ex2(fmaf(s[2 * j + 1], p.scale_log2, nref)) : 0.f;
          lsum += p0 + p1;
          pk[k][j] = pack_bf16(p0, p1);
        }
      }
    }
    tc_fence_before();  // every read of S precedes the P writes over it
    const uint32_t zero16[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    const int g0 = col0 / kChunk;  // this warp's first 16-column P group (32 positions each)
#pragma unroll
    for (int gg = 0; gg < kVTile / kChunk; ++gg)
      if (gg < g0 || gg >= g0 + NCH) tmem_st16u(sbuf + gg * 16, zero16);
#pragma unroll
    for (int k = 0; k < NCH; ++k) tmem_st16u(sbuf + (g0 + k) * 16, pk[k]);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.p_full[sb]);
  }
  // -------- the next unit's Q, so that its scores can start during this
  // unit's epilogue (the buffer's previous unit has had all its scores read)
  if (nb >= 0) {
    write_q<HD>(p, tmem, qbuf_next, nb, nh, warp, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.qfull[qbuf_next]);
  }

  // -------- epilogue: merge the copies, then this lane's row of O
  if (ntiles > 0)
    mbar_wait_checked(&bars.empty[(tbase + ntiles - 1) % stages],
                      ((tbase + ntiles - 1) / stages) & 1, p.wait_ns, p.error_flag);
  tc_fence_after();
  // scratch, column-major so that a warp's 32 rows are 32 consecutive
  // floats: sml[copy - 1][{m, l}][row], then W columns of O per copy
  // so[copy - 1][d][row] (W = 32, or all of head_dim through the ring)
  float* sml = scratch;
  const int per = ring ? HD / 32 : 1;  // 32-column chunks per hand-over
  float* so = ring ? ring : scratch + (CS > 1 ? (CS - 1) * 2 * RPC : 0);
  if (CS > 1 && c > 0) {
    sml[((c - 1) * 2) * RPC + m] = m_used;
    sml[((c - 1) * 2 + 1) * RPC + m] = lsum;
  }
  if (CS > 1) named_barrier_sync(1, 4 * 32);  // all four softmax warps
  // weights of the copies relative to the largest reference (copy 0's warps)
  float mxr = m_used;
  for (int c2 = 1; c2 < CS; ++c2) mxr = fmaxf(mxr, sml[((c2 - 1) * 2) * RPC + m]);
  const float ref = safe_ref(mxr);
  const float w0 = m_used == -INFINITY ? 0.f : ex2(m_used - ref);
  float wc[CS > 1 ? CS - 1 : 1];
  float lt_all = w0 * lsum;
#pragma unroll
  for (int c2 = 1; c2 < CS; ++c2) {
    const float mc = sml[((c2 - 1) * 2) * RPC + m];
    const float lc = sml[((c2 - 1) * 2 + 1) * RPC + m];
    wc[c2 - 1] = mc == -INFINITY ? 0.f : ex2(mc - ref);
    lt_all += wc[c2 - 1] * lc;
  }
  const size_t bh = (size_t)b * p.num_kv_heads + h;
  const float inv = lt_all > 0.f ? 1.f / lt_all : 0.f;
#pragma unroll 1
  for (int g0 = 0; g0 < HD / 32; g0 += per) {
    if (CS > 1) {  // copies 1.. hand their columns to copy 0
      if (c > 0) {
#pragma unroll 1
        for (int cc = g0; cc < g0 + per; ++cc) {
          float o[32];
          if (ntiles > 0) {
            tmem_ld32(trow + kOCol + cc * 32, o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0.f;
          }
          float* d = so + ((size_t)(c - 1) * per + (cc - g0)) * 32 * RPC + m;
#pragma unroll
          for (int k = 0; k < 32; ++k) d[k * RPC] = o[k];
        }
      }
      named_barrier_sync(1, 4 * 32);
    }
#pragma unroll 1
  for (int cc = g0; cc < g0 + per; ++cc) {
    float o[32];
    if (c == 0) {
      if (ntiles > 0) {
        tmem_ld32(trow + kOCol + cc * 32, o);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0.f;
      }
    }
    if (c == 0 && m < M) {
#pragma unroll
      for (int k = 0; k < 32; ++k) o[k] *= w0;
#pragma unroll
      for (int c2 = 1; c2 < CS; ++c2) {
        const float* src = so + ((size_t)(c2 - 1) * per + (cc - g0)) * 32 * RPC + m;
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] += wc[c2 - 1] * src[k * RPC];
      }
      if (p.splits == 1) {
        __nv_bfloat16* dst =
            p.out + ((size_t)(b * R + ri) * p.num_q_heads + h * g + rq) * HD + cc * 32;
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          uint4 w;
          w.x = pack_bf16(o[k] * inv, o[k + 1] * inv);
          w.y = pack_bf16(o[k + 2] * inv, o[k + 3] * inv);
          w.z = pack_bf16(o[k + 4] * inv, o[k + 5] * inv);
          w.w = pack_bf16(o[k + 6] * inv, o[k + 7] * inv);
          *reinterpret_cast<uint4*>(dst + k) = w;
        }
      } else {
        float* dst = p.part_o + ((bh * p.splits + split) * M + m) * HD + cc * 32;
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(dst + k) = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
      }
    }
  }
    // the columns are read before the next are written, and before any warp
    // goes on to the next unit (whose capture staging overlaps the scratch)
    if (CS > 1) named_barrier_sync(1, 4 * 32);
  }
  if (c > 0) return;
  if (m < M && p.splits > 1) {
    float* ml = p.part_ml + ((bh * p.splits + split) * M + m) * 2;
    ml[0] = mxr;
    ml[1] = lt_all;
  }
  if (m < M && p.splits == 1 && cap_rows)  // the row's normaliser: (m + log2 l) ln 2
    p.capture[p.lse_offset + ((size_t)b * p.num_q_heads + h * g + rq) * R + ri] =
        (mxr + __log2f(lt_all)) * 0.6931471805599453f;
}

template <int HD, int CM, bool SP>
__global__ void __launch_bounds__(kVerifyThreads, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const VerifyParams p) {
  using Lay = VerifyLayout<HD>;
  constexpr int KS = HD / 16;     // k-steps of Q K^T
  constexpr int kTileBytes = Lay::kTileBytes;
  constexpr int kStageBytes = Lay::kStageBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.n_rows, M = p.m_rows;
  const int NS = (M + 31) >> 5;
  const int CS = M <= 32 ? 4 : (M <= 64 ? 2 : 1);  // row copies
  const int NAW = CS == 1 ? NS : 4;                  // softmax warps at work
  const int stages = p.stages;

  uint8_t* ring = smem;
  float* cap_s = reinterpret_cast<float*>(ring + (size_t)stages * kStageBytes);
  float* all_s = cap_s + Lay::kCapFloats;
  int32_t* sl_page = reinterpret_cast<int32_t*>(all_s + Lay::kAllFloats);  // sparse: split's
  uint32_t* sl_mask = reinterpret_cast<uint32_t*>(sl_page + Lay::kSliceMax);  // union slice
  VerifyBars bars;
  bars.stages = stages;
  bars.kfull = reinterpret_cast<uint64_t*>(sl_mask + Lay::kSliceMax);  // K half landed
  bars.vfull = bars.kfull + stages;   // V half landed
  bars.kempty = bars.vfull + stages;  // Q K(t)^T done: K half free
  bars.empty = bars.kempty + stages;  // P(t) V(t) done: V half, S and P buffer free
  bars.s_full = bars.empty + stages;  // S of a buffer computed (tensor-core commit)
  bars.p_full = bars.s_full + 2;      // P of a buffer written by every softmax warp
  bars.capfull = bars.p_full + 2;     // [copy][slot]: Collect-All partials written
  bars.capfree = bars.capfull + 4;    // [copy][slot]: Collect-All slot read
  bars.drain = bars.capfree + 4;      // every tensor-core operation issued so far done
  bars.qfull = bars.drain + 1;        // [buffer]: a later unit's Q written (persistent CTAs)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars.qfull + 2);
  int* utab = reinterpret_cast<int*>(tmem_holder + 4);  // persistent: per-sequence unit table

  // the K/V tensor maps are kernel parameters, independent of earlier
  // kernels: fetch their descriptors before anything else so that the first
  // TMA does not wait for them
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  // programmatic dependent launch: inputs may come from the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kPagesPerTile = kVTile / kPageSize;  // 8

  // ---- the CTA's units of work.  One CTA per (split, KV head, sequence)
  // runs one unit.  A persistent CTA (dense only) takes every gridDim.x-th
  // unit of a list built from the device lengths: the full splits of every
  // (sequence, KV head) first, then the shorter last splits, so that the
  // round-robin keeps the CTAs balanced.
  const bool persistent = !SP && p.persistent;
  int n_units = 1;
  int pre_id = -1;  // page id of lane's page in the first unit's first window (one CTA per unit)
  if (persistent) {
    // utab: [0, B] prefix of full units, [B+1, 2B+1] prefix of last
    // (partial) units, [2B+2, 3B+1] tiles per sequence, [3B+2, 4B+1] lengths
    const int B = p.batch;
    if (threadIdx.x < B) {
      const int bb = threadIdx.x;
      const int L = p.prefix_lens[bb];
      const bool ok = L >= 1 && L <= p.max_prefix &&
                      (L + R + kPageSize - 1) / kPageSize <= p.max_pages_per_seq;
      if (!ok && blockIdx.x == 0) flag_error(p.error_flag, VG_DEVERR_LENGTH);
      const int tiles = ok ? (L + R + kVTile - 1) / kVTile : 0;
      utab[2 * B + 2 + bb] = tiles;
      utab[3 * B + 2 + bb] = L;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int f = 0, q = 0;
      for (int bb = 0; bb < B; ++bb) {
        utab[bb] = f;
        utab[B + 1 + bb] = q;
        const int tiles = utab[2 * B + 2 + bb];
        f += p.num_kv_heads * (tiles / p.tiles_per_split);
        q += p.num_kv_heads * (tiles % p.tiles_per_split != 0 ? 1 : 0);
      }
      utab[B] = f;
      utab[2 * B + 1] = q;
    }
    __syncthreads();
    const int total = utab[B] + utab[2 * B + 1];
    n_units = blockIdx.x < total ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  } else if (!SP && warp == kProducerWarp) {
    // the page ids of the first 4 tiles are read while the length is still
    // in flight (within the page-table row; ids past the sequence are dropped
    // once the length is known)
    const int lp = blockIdx.x * p.tiles_per_split * kPagesPerTile + lane;
    if (lp < p.max_pages_per_seq)
      pre_id = p.page_table[(size_t)blockIdx.z * p.max_pages_per_seq + lp];
  }
  // unit k of this CTA: (sequence, KV head, split), its first tile and tile
  // count, the sequence's length (a negative b: no such unit, or a skipped
  // sequence)
  auto unit_of = [&](int k, int& b, int& h, int& split, int& t0, int& ntiles, int& L) {
    b = -1;
    h = split = t0 = ntiles = L = 0;
    if (k >= n_units) return;
    if (!persistent) {
      b = blockIdx.z;
      h = blockIdx.y;
      split = blockIdx.x;
      L = p.prefix_lens[b];
      const int n_b = L + R;
      if (L < 1 || L > p.max_prefix || (n_b + kPageSize - 1) / kPageSize > p.max_pages_per_seq) {
        b = -1;
        return;
      }
      const int u_n = SP ? min(p.u_count[b], p.u_max) : 0;  // union pages of this sequence
      const int tiles_b = SP ? (u_n + kPagesPerTile - 1) / kPagesPerTile : (n_b + kVTile - 1) / kVTile;
      // Dense: split s streams tiles [s tps, (s + 1) tps).  Sparse: the
      // union's size is known only on the device, so split s takes tiles s,
      // s + S, ... and every split has work whatever the union's size.
      t0 = SP ? 0 : split * p.tiles_per_split;
      ntiles = SP ? (split < tiles_b ? min((tiles_b - split + p.splits - 1) / p.splits,
                                          p.tiles_per_split)
                                     : 0)
                  : max(0, min(t0 + p.tiles_per_split, tiles_b) - t0);
      return;
    }
    const int B = p.batch, tps = p.tiles_per_split;
    int i = blockIdx.x + k * gridDim.x;
    const bool full = i < utab[B];
    if (!full) i -= utab[B];
    const int* pre = full ? utab : utab + B + 1;
    int bb = 0;
    while (bb + 1 < B && pre[bb + 1] <= i) ++bb;
    const int j = i - pre[bb];
    const int tiles = utab[2 * B + 2 + bb];
    b = bb;
    L = utab[3 * B + 2 + bb];
    if (full) {
      const int nf = tiles / tps;
      h = j / nf;
      split = j - h * nf;
    } else {
      h = j;
      split = tiles / tps;
    }
    t0 = split * tps;
    ntiles = min(tps, tiles - t0);
  };

  int b0, h0, split0, t00, nt0, L0;
  unit_of(0, b0, h0, split0, t00, nt0, L0);
  if (persistent && warp == kProducerWarp && b0 >= 0) {
    const int lp = t00 * kPagesPerTile + lane;
    if (lp < (L0 + R + kPageSize - 1) / kPageSize)
      pre_id = p.page_table[(size_t)b0 * p.max_pages_per_seq + lp];
  }
  if (!persistent && b0 < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      flag_error(p.error_flag, VG_DEVERR_LENGTH);
    return;  // uniform for every CTA of this sequence
  }
  if (n_units == 0) return;  // a persistent CTA without work (uniform)
  int sl_n = 0;  // slots of this split's union slice (sparse; -1 past the union)
  if constexpr (SP) {
    const int u_n = min(p.u_count[b0], p.u_max);
    sl_n = min(nt0 * kPagesPerTile, Lay::kSliceMax);
    for (int i = threadIdx.x; i < sl_n; i += kVerifyThreads) {
      const int lt = i / kPagesPerTile;
      const int e = (split0 + lt * p.splits) * kPagesPerTile + (i - lt * kPagesPerTile);
      sl_page[i] = e < u_n ? p.u_pages[(size_t)b0 * p.u_max + e] : -1;
      sl_mask[i] = e < u_n ? p.u_masks[(size_t)b0 * p.u_max + e] : 0u;
    }
  }

  // the first unit's Q rows: loads issued now, written to tensor memory once
  // it is allocated
  uint4 qreg[HD / 8];
  if (warp < 4) load_q<HD>(p, b0, h0, warp, lane, qreg);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    const int nwc = CS == 1 ? NS : 4 / CS;  // warps per copy holding rows
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], NAW);
      mbar_init(&bars.qfull[s], NAW);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars.capfull[s], nwc > 1 ? nwc - 1 : 1);
      mbar_init(&bars.capfree[s], 1);
    }
    mbar_init(bars.drain, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_holder, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The first unit's Q (buffer 0) and zero rows in buffer 1 (rows that no
  // unit fills) are handed from the softmax warps to the MMA warp through
  // named barrier 2 (warps 0-3 and 5); later units' Q through qfull.
  constexpr int kQReadyBar = 2, kQReadyThreads = 5 * 32;
  if (warp < 4) {
    store_q<HD>(tmem, 0, warp, qreg);
    if (n_units > 1) write_q<HD>(p, tmem, 1, -1, 0, warp, lane);
    named_barrier_sync(kQReadyBar, kQReadyThreads);
  } else if (warp == kMmaWarp) {
    named_barrier_sync(kQReadyBar, kQReadyThreads);
    tc_fence_after();
  }

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------- producer
    // The K and V halves of a ring stage are filled and freed separately:
    // K(t) once Q K(t - stages)^T is done, V(t) once P(t - stages) V is done.
    // K is issued one tile ahead of V, so that the loads the next Q K^T
    // waits for are not held back by the softmax of older tiles.  The warp
    // fetches the page ids of 4 tiles (32 ids, one per lane) in one round
    // trip; each lane issues one TMA box (16 positions x 64 dims) of a half.
    // Across a persistent CTA's units the ring keeps streaming: the next
    // unit's first page ids are read while the current unit is loaded.
    const uint64_t pol = l2_policy_evict_first();
    constexpr int kHalfBoxes = kPagesPerTile * (HD / 64);  // boxes of one of K / V
    const int pi = lane / (HD / 64), dh = lane % (HD / 64);
    int k_armed = 0, v_armed = 0;  // K / V tile loads issued (the CTA's running count)
    bool aborted = false;
    int b = b0, h = h0, split = split0, t0 = t00, ntiles = nt0, L = L0;
    for (int k = 0; k < n_units && !aborted; ++k) {
      int nb, nh, nsplit, nt0n, nntiles, nL;
      unit_of(k + 1, nb, nh, nsplit, nt0n, nntiles, nL);
      int pre_next = -1;  // the next unit's first page ids, read ahead
      if (nb >= 0) {
        const int lp = nt0n * kPagesPerTile + lane;
        const int npg = (nL + R + kPageSize - 1) / kPageSize;
        if (lp < npg) pre_next = p.page_table[(size_t)nb * p.max_pages_per_seq + lp];
      }
      const int npages_b = (L + R + kPageSize - 1) / kPageSize;
      const int tbase = k_armed;
      // Page ids of tiles [4w, 4w + 4) for the window w of the K tile, and of
      // the window before it (V runs one tile behind).  The page-table entries
      // of window w + 1 are read when window w starts, so that the load's
      // latency is hidden behind four tiles of streaming.
      constexpr int kNoPage = INT_MIN;  // lane's slot lies outside the unit
      auto fetch = [&](int kt) -> int {
        const int lt_l = kt + (lane >> 3);
        const int slot = lt_l * kPagesPerTile + (lane & 7);
        const int lp = SP ? (slot < sl_n ? sl_page[slot] : -1)
                          : (t0 + lt_l) * kPagesPerTile + (lane & 7);
        if (lt_l < ntiles && lp >= 0 && lp < npages_b)
          return (kt == 0 && !SP) ? pre_id : p.page_table[(size_t)b * p.max_pages_per_seq + lp];
        return kNoPage;
      };
      int raw_now = fetch(0), raw_ahead = fetch(4);
      int id_cur = p.num_pages, id_prev = p.num_pages;
      for (int kt = 0; kt <= ntiles; ++kt) {
        const int vt = kt - 1;
        const bool new_window = kt < ntiles && (kt & 3) == 0;
        if (new_window) {
          id_prev = id_cur;
          if (kt > 0) {
            raw_now = raw_ahead;
            raw_ahead = fetch(kt + 4);
          }
          id_cur = p.num_pages;  // out of range: TMA fills zeros
          if (raw_now != kNoPage) {
            if (raw_now >= 0 && raw_now < p.num_pages)
              id_cur = raw_now;
            else
              flag_error(p.error_flag, VG_DEVERR_PAGE);
          }
        }
        if (kt < ntiles) {
          const int T = tbase + kt;
          const int st = T % stages;
          int go = 1;
          if (lane == 0 && T >= stages)
            go = mbar_wait_checked(&bars.kempty[st], ((T / stages) - 1) & 1, p.wait_ns,
                                   p.error_flag);
          go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) {  // the consumer is gone: stop, then drain what is in flight
            aborted = true;
            break;
          }
          const int id = __shfl_sync(0xffffffffu, id_cur, (kt & 3) * 8 + (pi & 7));
          if (lane == 0) mbar_arrive_expect_tx(&bars.kfull[st], kTileBytes);
          __syncwarp();
          if (lane < kHalfBoxes)
            tma_load_4d(ring + st * kStageBytes + dh * Lay::kHalfBytes + pi * kPageSize * 128, &tmk,
                        &bars.kfull[st], dh * 64, 0, h, id, pol);
          __syncwarp();
          ++k_armed;
        }
        if (vt >= 0) {
          const int T = tbase + vt;
          const int st = T % stages;
          int go = 1;
          if (lane == 0 && T >= stages)
            go = mbar_wait_checked(&bars.empty[st], ((T / stages) - 1) & 1, p.wait_ns,
                                   p.error_flag);
          go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) {
            aborted = true;
            break;
          }
          const int idv = new_window ? id_prev : id_cur;  // V's tile is in the window before
          const int id = __shfl_sync(0xffffffffu, idv, (vt & 3) * 8 + (pi & 7));
          if (lane == 0) mbar_arrive_expect_tx(&bars.vfull[st], kTileBytes);
          __syncwarp();
          if (lane < kHalfBoxes)
            tma_load_4d(ring + st * kStageBytes + kTileBytes + dh * Lay::kHalfBytes +
                            pi * kPageSize * 128,
                        &tmv, &bars.vfull[st], dh * 64, 0, h, id, pol);
          __syncwarp();
          ++v_armed;
        }
      }
      b = nb;
      h = nh;
      split = nsplit;
      t0 = nt0n;
      ntiles = nntiles;
      L = nL;
      pre_id = pre_next;
    }
    // After a normal run every load has been consumed.  After an abandoned
    // run, wait (bounded) for the last load armed on every stage, so that no
    // copy is still writing into shared memory when the CTA leaves.
    if (lane == 0 && aborted) {
      for (int s = 0; s < stages; ++s) {
        if (k_armed > s) mbar_wait(&bars.kfull[s], (((k_armed - 1 - s) / stages)) & 1);
        if (v_armed > s) mbar_wait(&bars.vfull[s], (((v_armed - 1 - s) / stages)) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t ring_u = smem_u32(ring);
      constexpr uint32_t id_qk = umma_idesc_bf16(kMPad, kVTile, 0, 0);
      constexpr uint32_t id_pv = umma_idesc_bf16(kMPad, HD, 0, 1);
      bool live = true, reported = false;
      int tbase = 0;
      uint64_t last = global_timer_ns();
      for (int k = 0; k < n_units && live; ++k) {
        int b, h, split, t0, ntiles, L;
        unit_of(k, b, h, split, t0, ntiles, L);
        const int qbuf = k & 1;
        // a later unit's Q is written by the softmax warps (qfull), the first
        // one was handed over before the roles split
        bool q_ready = k == 0;
        // Issue whichever is ready: S(t) = Q K(t)^T (needs tile t and P(t - 2)
        // V done, which frees its S buffer) or O += P(t) V(t) (needs P(t)).
        int nq = 0, np = 0;
        while (np < ntiles) {
          bool moved = false;
          if (!q_ready && mbar_test_wait(&bars.qfull[qbuf], ((k - 1) >> 1) & 1)) {
            tc_fence_after();
            q_ready = true;
          }
          if (q_ready && nq < ntiles) {
            const int T = tbase + nq;
            const int st = T % stages, sb = T & 1;
            if (mbar_test_wait(&bars.kfull[st], (T / stages) & 1) &&
                (T < 2 || mbar_test_wait(&bars.empty[(T - 2) % stages], ((T - 2) / stages) & 1))) {
              tc_fence_after();
              const uint32_t kb = ring_u + st * kStageBytes;
#pragma unroll
              for (int ks = 0; ks < KS; ++ks) {
                const uint64_t bd =
                    umma_smem_desc(kb + (ks >> 2) * Lay::kHalfBytes + (ks & 3) * 32, 16, 1024);
                umma_bf16_ts(tmem + kSCol + sb * kVTile, tmem + kQCol + qbuf * (HD / 2) + ks * 8,
                             bd, id_qk, ks > 0);
              }
              umma_commit(&bars.s_full[sb]);
              umma_commit(&bars.kempty[st]);  // K half of the stage free for the producer
              ++nq;
              moved = true;
            }
          }
          if (np < nq) {
            const int T = tbase + np;
            const int st = T % stages, sb = T & 1;
            if (mbar_test_wait(&bars.p_full[sb], (T >> 1) & 1) &&
                mbar_test_wait(&bars.vfull[st], (T / stages) & 1)) {
              tc_fence_after();
              const uint32_t vb = ring_u + st * kStageBytes + kTileBytes;
#pragma unroll
              for (int ks = 0; ks < kVTile / 16; ++ks) {
                // V is MN-major: 64-dim blocks one half-tile apart, 8-position groups 1 KB apart
                const uint64_t bd = umma_smem_desc(vb + ks * 16 * 128, Lay::kHalfBytes, 1024);
                umma_bf16_ts(tmem + kOCol, tmem + kSCol + sb * kVTile + ks * 8, bd, id_pv,
                             (np > 0 || ks > 0));
              }
              umma_commit(&bars.empty[st]);
              ++np;
              moved = true;
            }
          }
          if (moved) {
            last = global_timer_ns();
          } else {
            const uint64_t idle = global_timer_ns() - last;
            if (!reported && (idle > p.wait_ns || idle > kWaitLimitNs)) {
              flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
              reported = true;
            }
            if (idle > kWaitLimitNs) {
              live = false;
              break;
            }
          }
        }
        tbase += ntiles;
      }
      // the last P.V has finished before the tensor memory is released
      if (live && tbase > 0 &&
          !mbar_wait_checked(&bars.empty[(tbase - 1) % stages], ((tbase - 1) / stages) & 1,
                             p.wait_ns, p.error_flag))
        live = false;
      if (!live) {  // abandoned: wait (bounded) for every tensor-core operation issued
        umma_commit(bars.drain);
        mbar_wait(bars.drain, 0);
      }
    }
    __syncwarp();
  } else if (warp < NAW) {
    // ---------------------------------------------------------- softmax
    float* scratch = cap_s;  // the capture staging and slice area, idle in an epilogue
    // a CTA with one unit has an idle ring at its epilogue
    float* ring_f = n_units == 1 ? reinterpret_cast<float*>(ring) : nullptr;
    int tbase = 0, hs = 0;
    for (int k = 0; k < n_units; ++k) {
      int b, h, split, t0, ntiles, L;
      unit_of(k, b, h, split, t0, ntiles, L);
      int nb, nh, nsplit, nt0n, nntiles, nL;
      unit_of(k + 1, nb, nh, nsplit, nt0n, nntiles, nL);
      const int qn = (k + 1) & 1;
      if (CS == 4)
        verify_softmax<HD, 32, CM, SP>(p, bars, scratch, ring_f, cap_s, all_s, sl_page, sl_mask, sl_n, tmem, b, h, split, t0, ntiles, L, tbase, hs, nb, nh, qn, warp, lane);
      else if (CS == 2)
        verify_softmax<HD, 64, CM, SP>(p, bars, scratch, ring_f, cap_s, all_s, sl_page, sl_mask, sl_n, tmem, b, h, split, t0, ntiles, L, tbase, hs, nb, nh, qn, warp, lane);
      else
        verify_softmax<HD, 128, CM, SP>(p, bars, scratch, ring_f, cap_s, all_s, sl_page, sl_mask, sl_n, tmem, b, h, split, t0, ntiles, L, tbase, hs, nb, nh, qn, warp, lane);
      tbase += ntiles;
    }
  }
  tc_fence_before();
  __syncthreads();  // every TMEM access and every MMA of this CTA is done
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Split-K merge: one CTA per (output row m, KV head, sequence).  Thread t < splits
// reads split t's (m, l); each of the HD / 4 threads of a float4 column then
// sums the splits' partial rows with the log-sum-exp weights.  Launched with
// programmatic dependent launch: it waits for the verify grid (and its
// memory) before reading the partials.
template <int HD>
__global__ void __launch_bounds__(kMergeThreads) verify_merge_kernel(const VerifyParams p) {
  __shared__ __align__(16) float smem_f[kMergeSmemFloats];
  const int m = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  // The length and the union size are read before waiting for the verify
  // grid: this kernel's predecessor is always that grid, which writes
  // neither (it waits for its own predecessors before it lets this kernel
  // launch), so the read overlaps the verify tail instead of following it.
  const int L = p.prefix_lens[b];
  const int u_cnt = p.u_count ? p.u_count[b] : 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (L < 1 || L > p.max_prefix ||
      (L + p.n_rows + kPageSize - 1) / kPageSize > p.max_pages_per_seq)
    return;  // the verify kernel skipped this sequence (and flagged it)
  const int M = p.m_rows, S = p.splits;
  // splits with work: dense, split s streams tiles [s tps, (s + 1) tps) of
  // the sequence's; sparse, split s takes union tiles s, s + S, ...
  const int tiles_b = p.u_count ? (min(u_cnt, p.u_max) + kVTile / kPageSize - 1) / (kVTile / kPageSize)
                                : (L + p.n_rows + kVTile - 1) / kVTile;
  const int s_work = p.u_count ? min(S, tiles_b)
                               : min(S, (tiles_b + p.tiles_per_split - 1) / p.tiles_per_split);
  const size_t bh = (size_t)b * p.num_kv_heads + h;
  int i, qi;
  row_of(m, p.group, p.n_rows, i, qi);
  merge_splits<HD>(p.part_o + (bh * S * M + m) * HD, (size_t)M * HD, p.part_ml + (bh * S * M + m) * 2,
                   (size_t)M * 2, s_work,
                   p.out + ((size_t)(b * p.n_rows + i) * p.num_q_heads + h * p.group + qi) * HD, smem_f,
                   p.capture_mode == VG_CAPTURE_ALL_ROWS
                       ? p.capture + p.lse_offset +
                             ((size_t)b * p.num_q_heads + h * p.group + qi) * p.n_rows + i
                       : nullptr);
}

// Sparse verification, exact merged schedule (SSV: Sparse Speculative
// Verification, section 4.2 and Figures 2/4/5): the union of the verify rows'
// selected blocks (16-position pages) plus the pages of the verify block
// itself, ascending, with one bit per row that selected each page.  One CTA
// per sequence: page bits in shared memory, then an ordered compaction.
constexpr int kUnionThreads = 1024;

__global__ void __launch_bounds__(kUnionThreads)
    sparse_union_kernel(const VerifyParams p, const int32_t* blocks, const int32_t* block_counts,
                        int max_blocks) {
  extern __shared__ uint32_t pm[];  // [pages of the sequence] row bits
  __shared__ int wsum[32], woff[32], tot_s, base_s;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int R = p.n_rows;
  const int L = p.prefix_lens[b];
  if (L < 1 || L > p.max_prefix || (L + R + kPageSize - 1) / kPageSize > p.max_pages_per_seq) {
    if (tid == 0) p.u_count[b] = 0;  // the verify kernel skips and flags the sequence
    return;
  }
  const int npb = (L + R + kPageSize - 1) / kPageSize;  // pages up to the end of the block
  const int npl = (L + kPageSize - 1) / kPageSize;      // pages holding prefix positions
  for (int i = tid; i < npb; i += kUnionThreads) pm[i] = 0;
  __syncthreads();
  for (int e = tid; e < R * max_blocks; e += kUnionThreads) {
    const int i = e / max_blocks, k = e - i * max_blocks;
    const int cnt = block_counts[(size_t)b * R + i];
    if (cnt < 0 || cnt > max_blocks) {
      if (k == 0) flag_error(p.error_flag, VG_DEVERR_COUNT);
      continue;
    }
    if (k >= cnt) continue;
    const int blk = blocks[((size_t)b * R + i) * max_blocks + k];
    if (blk < 0 || blk >= npl) {
      flag_error(p.error_flag, VG_DEVERR_INDEX);
      continue;
    }
    atomicOr(&pm[blk], 1u << i);
  }
  for (int pg = L / kPageSize + tid; pg < npb; pg += kUnionThreads)
    atomicOr(&pm[pg], 1u << 31);  // the verify block's own pages are always streamed
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int c0 = 0; c0 < npb; c0 += kUnionThreads) {
    const int pg = c0 + tid;
    const bool f = pg < npb && pm[pg] != 0u;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wsum[wid] = __popc(bal);
    __syncthreads();
    if (wid == 0) {
      const int v = wsum[lane];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      woff[lane] = incl - v;
      if (lane == 31) tot_s = incl;
    }
    __syncthreads();
    if (f) {
      const int slot = base_s + woff[wid] + __popc(bal & ((1u << lane) - 1u));
      if (slot < p.u_max) {
        p.u_pages[(size_t)b * p.u_max + slot] = pg;
        p.u_masks[(size_t)b * p.u_max + slot] = pm[pg] & 0xffffu;
      }
    }
    __syncthreads();
    if (tid == 0) base_s += tot_s;
    __syncthreads();
  }
  if (tid == 0) p.u_count[b] = min(base_s, p.u_max);
}

struct VerifyPlan {
  int hd, m_rows, m_tiles, groups, splits, tiles_per_split, stages;
  int persistent, grid_x;  // dense: persistent CTAs walking the units, and their number
  size_t smem_bytes;
  size_t off_ml, ws_bytes;
};

bool make_verify_plan(int batch, int n_rows, int num_q_heads, int num_kv_heads, int head_dim,
                      int max_prefix, int num_splits, VerifyPlan* pl, bool sparse = false) {
  if (batch <= 0 || n_rows <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_prefix <= 0)
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->hd = head_dim;
  pl->m_rows = g * n_rows;
  pl->m_tiles = ceil_div(pl->m_rows, 16);
  pl->groups = 1;
  const int tiles = ceil_div(max_prefix + n_rows, kVTile);
  int tps;
  if (num_splits > 0) {
    tps = ceil_div(tiles, std::min(num_splits, tiles));
  } else {
    const int pairs = batch * num_kv_heads;
    const int sms = device_sm_count();
    int splits = std::max(1, sms / pairs);
    tps = ceil_div(tiles, splits);
    if (batch > 1) tps = std::min(tps, 24);  // ragged lengths: chunks small enough to balance SMs
    tps = std::max(tps, std::min(tiles, 2));
  }
  if (ceil_div(tiles, tps) > kMaxSplits) tps = ceil_div(tiles, kMaxSplits);
  pl->tiles_per_split = tps;
  pl->splits = ceil_div(tiles, tps);
  // More units than SMs (and a batch the unit table holds): persistent CTAs,
  // one per SM, each walking its share of the units, so that one unit's
  // prologue and epilogue overlap the streaming of the next.
  const long long units = (long long)batch * num_kv_heads * pl->splits;
  const int sms = device_sm_count();
  pl->persistent = !sparse && batch <= kMaxPersistBatch && units > sms ? 1 : 0;
  pl->grid_x = pl->persistent ? sms : pl->splits;
  auto smem_for = [&](int stages) {
    return head_dim == 128 ? VerifyLayout<128>::bytes(stages) : VerifyLayout<64>::bytes(stages);
  };
  int stages = (head_dim == 128 ? 3 : 6);
  while (stages > 2 && smem_for(stages) > 227 * 1024) --stages;
  pl->stages = stages;
  pl->smem_bytes = smem_for(stages);
  const size_t o_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * head_dim * 4;
  const size_t ml_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * 2 * 4;
  pl->off_ml = align_up(o_bytes, 256);
  pl->ws_bytes = pl->splits > 1 ? pl->off_ml + align_up(ml_bytes, 256) : 0;
  return true;
}

template <int HD, int CM, bool SP = false>
cudaError_t launch_verify_main(const VerifyPlan& pl, const CUtensorMap& tk, const CUtensorMap& tv,
                               const VerifyParams& p, dim3 grid, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<HD, CM, SP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t vcfg = {};
  vcfg.gridDim = grid;
  vcfg.blockDim = dim3(kVerifyThreads, 1, 1);
  vcfg.dynamicSmemBytes = pl.smem_bytes;
  vcfg.stream = stream;
  vcfg.attrs = pdl;
  vcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&vcfg, verify_kernel<HD, CM, SP>, tk, tv, p);
}

template <int HD>
cudaError_t launch_verify(const VerifyPlan& pl, const CUtensorMap& tk, const CUtensorMap& tv,
                          const VerifyParams& p, dim3 grid, cudaStream_t stream,
                          bool sparse = false) {
  cudaError_t e;
  if (sparse) {
    e = launch_verify_main<HD, VG_CAPTURE_NONE, true>(pl, tk, tv, p, grid, stream);
  } else switch (p.capture_mode) {
    case VG_CAPTURE_GROUP_SUM: e = launch_verify_main<HD, VG_CAPTURE_GROUP_SUM>(pl, tk, tv, p, grid, stream); break;
    case VG_CAPTURE_ROWS: e = launch_verify_main<HD, VG_CAPTURE_ROWS>(pl, tk, tv, p, grid, stream); break;
    case VG_CAPTURE_ALL_SUM: e = launch_verify_main<HD, VG_CAPTURE_ALL_SUM>(pl, tk, tv, p, grid, stream); break;
    case VG_CAPTURE_ALL_ROWS: e = launch_verify_main<HD, VG_CAPTURE_ALL_ROWS>(pl, tk, tv, p, grid, stream); break;
    default: e = launch_verify_main<HD, VG_CAPTURE_NONE>(pl, tk, tv, p, grid, stream); break;
  }
  if (e != cudaSuccess || pl.splits == 1) return e;
  // split merge, chained with programmatic dependent launch
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.m_rows, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_merge_kernel<HD>, p);
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" size_t vg_verify_workspace_bytes(int batch, int n_rows, int num_q_heads,
                                            int num_kv_heads, int head_dim, int max_prefix,
                                            int num_splits) {
  VerifyPlan pl;
  if (!make_verify_plan(batch, n_rows, num_q_heads, num_kv_heads, head_dim, max_prefix,
                        num_splits, &pl))
    return 0;
  return pl.ws_bytes;
}

extern "C" vg_status vg_verify_attention(const vg_paged_kv* kv, const void* q,
                                         const int32_t* prefix_lens, int batch, int n_rows,
                                         int num_q_heads, int max_prefix, float softmax_scale,
                                         void* out, int capture_mode, float* capture,
                                         int num_splits, void* workspace, size_t workspace_bytes,
                                         int32_t* error_flag, cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (!q || !prefix_lens || !out || batch <= 0 || n_rows <= 0 || num_q_heads <= 0 ||
      max_prefix <= 0 || num_splits < 0 || !(softmax_scale == softmax_scale))
    return VG_ERR_INVALID_ARGUMENT;
  if (capture_mode != VG_CAPTURE_NONE && capture_mode != VG_CAPTURE_GROUP_SUM &&
      capture_mode != VG_CAPTURE_ROWS && capture_mode != VG_CAPTURE_ALL_SUM &&
      capture_mode != VG_CAPTURE_ALL_ROWS)
    return VG_ERR_INVALID_ARGUMENT;
  if (capture_mode != VG_CAPTURE_NONE && !capture) return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads % kv->num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / kv->num_kv_heads;
  if (g > 8 || n_rows > 16 || g * n_rows > 96) return VG_ERR_UNSUPPORTED;
  if (ceil_div(max_prefix + n_rows, kPageSize) > kv->max_pages_per_seq)
    return VG_ERR_INVALID_ARGUMENT;
  VerifyPlan pl;
  if (!make_verify_plan(batch, n_rows, num_q_heads, kv->num_kv_heads, kv->head_dim, max_prefix,
                        num_splits, &pl))
    return VG_ERR_INVALID_ARGUMENT;
  if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes))
    return VG_ERR_WORKSPACE_TOO_SMALL;
  if (pl.smem_bytes > 227 * 1024) return VG_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if (!page_pool_tensor_map(kv->k_pages, kv->num_pages, kv->num_kv_heads, kv->head_dim, &tk) ||
      !page_pool_tensor_map(kv->v_pages, kv->num_pages, kv->num_kv_heads, kv->head_dim, &tv))
    return VG_ERR_LAUNCH;

  VerifyParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.prefix_lens = prefix_lens;
  p.page_table = kv->page_table;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.capture = capture;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = pl.ws_bytes ? reinterpret_cast<float*>(ws) : nullptr;
  p.part_ml = pl.ws_bytes ? reinterpret_cast<float*>(ws + pl.off_ml) : nullptr;
  p.error_flag = error_flag;
  p.batch = batch;
  p.n_rows = n_rows;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = kv->num_kv_heads;
  p.group = g;
  p.m_rows = pl.m_rows;
  p.m_tiles = pl.m_tiles;
  p.max_prefix = max_prefix;
  p.max_pages_per_seq = kv->max_pages_per_seq;
  p.num_pages = kv->num_pages;
  p.capture_mode = capture_mode;
  p.lse_offset = (size_t)batch * num_q_heads * n_rows * max_prefix;
  p.splits = pl.splits;
  p.tiles_per_split = pl.tiles_per_split;
  p.stages = pl.stages;
  p.groups = pl.groups;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * kLog2e;
  p.wait_ns = wait_report_ns();
  p.persistent = pl.persistent;
  const dim3 grid = pl.persistent ? dim3(pl.grid_x, 1, 1) : dim3(pl.splits, kv->num_kv_heads, batch);
  const cudaError_t e = kv->head_dim == 128 ? launch_verify<128>(pl, tk, tv, p, grid, stream)
                                             : launch_verify<64>(pl, tk, tv, p, grid, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Sparse verification (declared in vg.h).
namespace {

// Most union pages a sequence can have: every row's blocks distinct, plus the
// pages of the verify block, never more than the pages of the whole range.
int sparse_union_max(int max_prefix, int n_rows, int max_blocks) {
  const long long all = ceil_div(max_prefix + n_rows, kPageSize);
  const long long sel = (long long)n_rows * max_blocks + ceil_div(n_rows, kPageSize) + 1;
  return (int)std::min(all, sel);
}

struct SparseLayout {
  VerifyPlan pl;
  int u_max;
  size_t off_pages, off_masks, off_count, bytes;
};

bool make_sparse_layout(int batch, int n_rows, int num_q_heads, int num_kv_heads, int head_dim,
                        int max_prefix, int max_blocks, int num_splits, SparseLayout* sl) {
  if (max_blocks < 0 || max_prefix <= 0 || n_rows <= 0) return false;
  sl->u_max = std::max(1, sparse_union_max(max_prefix, n_rows, max_blocks));
  // plan the splits over the largest union, as if it were a dense range
  const int eff = std::max(1, sl->u_max * kPageSize - n_rows);
  if (!make_verify_plan(batch, n_rows, num_q_heads, num_kv_heads, head_dim, eff, num_splits,
                        &sl->pl, true))
    return false;
  // a split's union pages must fit its shared-memory slice
  constexpr int kMaxTps = VerifyLayout<128>::kSliceMax / (kVTile / kPageSize);
  if (sl->pl.tiles_per_split > kMaxTps) {
    const int tiles = ceil_div(eff + n_rows, kVTile);
    if (!make_verify_plan(batch, n_rows, num_q_heads, num_kv_heads, head_dim, eff,
                          std::max(num_splits, ceil_div(tiles, kMaxTps)), &sl->pl, true))
      return false;
    if (sl->pl.tiles_per_split > kMaxTps) return false;
  }
  sl->off_pages = align_up(sl->pl.ws_bytes, 256);
  sl->off_masks = sl->off_pages + align_up((size_t)batch * sl->u_max * 4, 256);
  sl->off_count = sl->off_masks + align_up((size_t)batch * sl->u_max * 4, 256);
  sl->bytes = sl->off_count + align_up((size_t)batch * 4, 256);
  return true;
}

}  // namespace

extern "C" size_t vg_sparse_verify_workspace_bytes(int batch, int n_rows, int num_q_heads,
                                                   int num_kv_heads, int head_dim, int max_prefix,
                                                   int max_blocks, int num_splits) {
  SparseLayout sl;
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      !make_sparse_layout(batch, n_rows, num_q_heads, num_kv_heads, head_dim, max_prefix,
                          max_blocks, num_splits, &sl))
    return 0;
  return sl.bytes;
}

extern "C" vg_status vg_sparse_verify_attention(
    const vg_paged_kv* kv, const void* q, const int32_t* prefix_lens, int batch, int n_rows,
    int num_q_heads, int max_prefix, float softmax_scale, const int32_t* blocks,
    const int32_t* block_counts, int max_blocks, void* out, int num_splits, void* workspace,
    size_t workspace_bytes, int32_t* error_flag, cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (!q || !prefix_lens || !out || !block_counts || batch <= 0 || n_rows <= 0 ||
      num_q_heads <= 0 || max_prefix <= 0 || num_splits < 0 || max_blocks < 0 ||
      !(softmax_scale == softmax_scale) || (max_blocks > 0 && !blocks))
    return VG_ERR_INVALID_ARGUMENT;
  if (num_q_heads % kv->num_kv_heads) return VG_ERR_INVALID_ARGUMENT;
  const int g = num_q_heads / kv->num_kv_heads;
  if (g > 8 || n_rows > 16 || g * n_rows > 96) return VG_ERR_UNSUPPORTED;
  if (ceil_div(max_prefix + n_rows, kPageSize) > kv->max_pages_per_seq)
    return VG_ERR_INVALID_ARGUMENT;
  if ((size_t)kv->max_pages_per_seq * 4 > 200 * 1024) return VG_ERR_UNSUPPORTED;
  SparseLayout sl;
  if (!make_sparse_layout(batch, n_rows, num_q_heads, kv->num_kv_heads, kv->head_dim, max_prefix,
                          max_blocks, num_splits, &sl))
    return VG_ERR_INVALID_ARGUMENT;
  if (!workspace || workspace_bytes < sl.bytes) return VG_ERR_WORKSPACE_TOO_SMALL;
  if (sl.pl.smem_bytes > 227 * 1024) return VG_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if (!page_pool_tensor_map(kv->k_pages, kv->num_pages, kv->num_kv_heads, kv->head_dim, &tk) ||
      !page_pool_tensor_map(kv->v_pages, kv->num_pages, kv->num_kv_heads, kv->head_dim, &tv))
    return VG_ERR_LAUNCH;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VerifyParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.prefix_lens = prefix_lens;
  p.page_table = kv->page_table;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.capture = nullptr;
  p.part_o = sl.pl.ws_bytes ? reinterpret_cast<float*>(ws) : nullptr;
  p.part_ml = sl.pl.ws_bytes ? reinterpret_cast<float*>(ws + sl.pl.off_ml) : nullptr;
  p.error_flag = error_flag;
  p.batch = batch;
  p.n_rows = n_rows;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = kv->num_kv_heads;
  p.group = g;
  p.m_rows = sl.pl.m_rows;
  p.m_tiles = sl.pl.m_tiles;
  p.max_prefix = max_prefix;
  p.max_pages_per_seq = kv->max_pages_per_seq;
  p.num_pages = kv->num_pages;
  p.capture_mode = VG_CAPTURE_NONE;
  p.lse_offset = 0;
  p.splits = sl.pl.splits;
  p.tiles_per_split = sl.pl.tiles_per_split;
  p.stages = sl.pl.stages;
  p.groups = sl.pl.groups;
  p.u_pages = reinterpret_cast<int32_t*>(ws + sl.off_pages);
  p.u_masks = reinterpret_cast<uint32_t*>(ws + sl.off_masks);
  p.u_count = reinterpret_cast<int32_t*>(ws + sl.off_count);
  p.u_max = sl.u_max;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * kLog2e;
  p.wait_ns = wait_report_ns();
  // the union pass, then the verify grid and its split merge (PDL chain)
  const size_t usmem = (size_t)kv->max_pages_per_seq * 4;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(sparse_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024) != cudaSuccess)
      return VG_ERR_LAUNCH;
    attr_done[dev] = true;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t ucfg = {};
  ucfg.gridDim = dim3(batch, 1, 1);
  ucfg.blockDim = dim3(kUnionThreads, 1, 1);
  ucfg.dynamicSmemBytes = usmem;
  ucfg.stream = stream;
  ucfg.attrs = pdl;
  ucfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&ucfg, sparse_union_kernel, p, blocks, block_counts, max_blocks) !=
      cudaSuccess)
    return VG_ERR_LAUNCH;
  dim3 grid(sl.pl.splits, kv->num_kv_heads, batch);
  const cudaError_t e = kv->head_dim == 128
                            ? launch_verify<128>(sl.pl, tk, tv, p, grid, stream, true)
                            : launch_verify<64>(sl.pl, tk, tv, p, grid, stream, true);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of vg_verify_attention (declared in vg.h).
//
// Its split partials live in one file-scope device array of
// fixed size instead of a caller-provided workspace.  The array exists once
// per GPU that loads this library and stays resident until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) uint8_t g_verify_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
void* noalloc_scratch_on_current_device() {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" size_t vg_verify_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" vg_status vg_verify_attention_noalloc(const vg_paged_kv* kv, const void* q,
                                                 const int32_t* prefix_lens, int batch,
                                                 int n_rows, int num_q_heads, int max_prefix,
                                                 float softmax_scale, void* out,
                                                 int capture_mode, float* capture,
                                                 int num_splits, int32_t* error_flag,
                                                 cudaStream_t stream) {
  vg_status st = check_paged_kv(kv);
  if (st != VG_OK) return st;
  if (batch <= 0 || n_rows <= 0 || num_q_heads <= 0 || max_prefix <= 0 || num_splits < 0 ||
      num_q_heads % kv->num_kv_heads)
    return VG_ERR_INVALID_ARGUMENT;
  VerifyPlan pl;
  if (!make_verify_plan(batch, n_rows, num_q_heads, kv->num_kv_heads, kv->head_dim, max_prefix,
                        num_splits, &pl))
    return VG_ERR_INVALID_ARGUMENT;
  if (pl.ws_bytes > kNoAllocScratchBytes) return VG_ERR_WORKSPACE_TOO_SMALL;
  // the scratch array used is the current device's: the stream must belong to it
  int cur = -1, sdev = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(stream, &sdev) != cudaSuccess)
    return VG_ERR_LAUNCH;
  if (cur != sdev) return VG_ERR_INVALID_ARGUMENT;
  uint8_t* scratch = static_cast<uint8_t*>(noalloc_scratch_on_current_device());
  if (!scratch) return VG_ERR_LAUNCH;
  // The array keeps the previous call's contents; nothing in it has to start
  // at zero: every partial is written before the merge reads it.
  return vg_verify_attention(kv, q, prefix_lens, batch, n_rows, num_q_heads, max_prefix,
                             softmax_scale, out, capture_mode, capture, num_splits, scratch,
                             kNoAllocScratchBytes, error_flag, stream);
}
