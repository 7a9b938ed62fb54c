// Verification attention with Collect-2-Query capture (sm_103a).
//
// Vegas: Self-Speculative Decoding with Verification-Guided Sparse Attention,
// "Core claim" / Figure 6: the verify pass is full attention of the k+1 block
// rows over the whole cache, and it writes only two pre-softmax logit rows
// (first draft token, bonus token) for the prefix positions.
//
// Design (one CTA per (KV split, KV head, sequence)):
//  * The g query heads x R verify rows of one KV head are packed into the
//    M dimension of warp-level bf16 tensor-core MMAs (m16n8k16, fp32
//    accumulate), so every K/V page is read from HBM once per KV head.
//    Row order in M: [row 0 of each head][row k of each head][rows 1..k-1],
//    which keeps the two captured rows inside the first 16-row tile.
//  * A producer warp streams 64-position tiles (4 pages) of K and V into a
//    shared-memory ring with 4-D TMA loads (128-byte swizzle, evict-first
//    L2 policy); consumers wait on mbarriers (bounded waits).
//  * Consumer warp (mt, grp) owns rows [16 mt, 16 mt + 16) of whole 64-position
//    tiles; the NG warp groups take alternating tiles, each keeping its own
//    online-softmax state (8 independent MMA accumulators per warp, softmax
//    reductions and rescales amortised over 64 positions).
//  * Capture epilogue: the first-row-tile warps stage their 16 x 64 logits
//    in shared memory and write either the raw two rows or their per-KV-head
//    sum in a fixed order, with coalesced stores.  Collect-All (every row)
//    reduces each row tile's 16 rows per column with a butterfly, hands the
//    partial column sums to the group's first warp through shared memory
//    (mbarrier handshakes with bounded waits), which adds them in row-tile
//    order and stores the per-KV-head sum.
//  * Splits over the KV length write fp32 partials (O, m, l) to the
//    workspace; a small merge kernel, one CTA per (output row, KV head,
//    sequence), combines them.  It is chained with programmatic dependent
//    launch, so its launch overlaps the verify grid.
#include <mutex>

#include "vg_device.cuh"
#include "vg_host.h"

namespace vg {
namespace {

constexpr int kTileN = 64;  // positions per pipeline stage = 4 pages
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

// Zero the bf16 halves of a packed pair whose positions are >= n.
__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int pos, int n) {
  if (pos >= n) v &= 0xffff0000u;
  if (pos + 1 >= n) v &= 0x0000ffffu;
  return v;
}

constexpr int kVerifyMaxThreads = 256;  // <= 7 consumer warps + 1 producer

template <int HD>
__global__ void __launch_bounds__(kVerifyMaxThreads, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const VerifyParams p) {
  constexpr int NT = kTileN / 8;  // S n-tiles per warp: a warp owns a whole 64-position tile
  constexpr int KS = HD / 16;     // k-steps of Q K^T
  constexpr int DN = HD / 8;      // O n-tiles
  constexpr int CH = HD / 8;      // 16-byte chunks per row
  constexpr int kTileBytes = kTileN * HD * 2;  // one of K / V
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kCapStride = 72;  // floats per row of a warp's capture staging tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, R = p.n_rows, M = p.m_rows;
  const int MT = p.m_tiles, NG = p.groups;
  const int n_cons = MT * NG;
  const int Mpad = MT * 16;
  const int stages = p.stages;

  uint8_t* ring = smem;
  uint8_t* qs = ring + stages * kStageBytes;
  float* cbuf = reinterpret_cast<float*>(qs + Mpad * HD * 2);
  float* cpart = cbuf + NG * 16 * kCapStride;  // Collect-All partials [NG][2][MT][64]
  uint64_t* full = reinterpret_cast<uint64_t*>(cpart + NG * 2 * MT * kTileN);
  uint64_t* empty = full + stages;
  uint64_t* capfull = empty + stages;  // [NG][2]: partials of a slot written
  uint64_t* capfree = capfull + 2 * NG;  // [NG][2]: a slot read by the group's first warp

  // programmatic dependent launch: inputs may come from the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int L = p.prefix_lens[b];
  const int n_b = L + R;
  if (L < 1 || L > p.max_prefix || (n_b + kPageSize - 1) / kPageSize > p.max_pages_per_seq) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(p.error_flag, VG_DEVERR_LENGTH);
    return;  // uniform for every CTA of this sequence
  }
  const int tiles_b = (n_b + kTileN - 1) / kTileN;
  const int t0 = split * p.tiles_per_split;
  const int ntiles = max(0, min(t0 + p.tiles_per_split, tiles_b) - t0);
  const int npages_b = (n_b + kPageSize - 1) / kPageSize;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MT);  // a tile is consumed by the MT warps of one group
    }
    for (int s = 0; s < 2 * NG; ++s) {
      mbar_init(&capfull[s], MT > 1 ? MT - 1 : 1);
      mbar_init(&capfree[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();  // barriers initialised: the producer may start at once

  float mrun0 = -INFINITY, mrun1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;

  if (warp == n_cons) {
    // ---------------------------------------------------------- producer
    // The warp fetches the page ids of 8 tiles (32 ids, one per lane) in one
    // round trip; lane 0 then issues the tiles' TMA loads as stages free up.
    if (ntiles > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
      }
      const uint64_t pol = l2_policy_evict_first();
      int my_id = p.num_pages;
      for (int lt = 0; lt < ntiles; ++lt) {
        if ((lt & 7) == 0) {
          const int lt_l = lt + (lane >> 2);
          const int lp = (t0 + lt_l) * (kTileN / kPageSize) + (lane & 3);
          my_id = p.num_pages;  // out of range: TMA fills zeros
          if (lt_l < ntiles && lp < npages_b) {
            const int e = p.page_table[(size_t)b * p.max_pages_per_seq + lp];
            if (e >= 0 && e < p.num_pages)
              my_id = e;
            else
              flag_error(p.error_flag, VG_DEVERR_PAGE);
          }
        }
        const int st = lt % stages;
        int go = 1;
        if (lane == 0 && lt >= stages) go = mbar_wait(&empty[st], ((lt / stages) - 1) & 1);
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          if (lane == 0) flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
          break;
        }
        // one TMA box (16 positions x 64 dims) per lane: page pi, half dh, K or V
        constexpr int kBoxes = (kTileN / kPageSize) * (HD / 64) * 2;
        const int pi = lane / ((HD / 64) * 2), dh = (lane >> 1) & (HD / 64 - 1), kv = lane & 1;
        const int id = __shfl_sync(0xffffffffu, my_id, (lt & 7) * 4 + (pi & 3));
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kStageBytes);
        __syncwarp();
        if (lane < kBoxes) {
          uint8_t* dst = ring + st * kStageBytes + kv * kTileBytes + dh * kTileN * 128 +
                         pi * kPageSize * 128;
          tma_load_4d(dst, kv ? &tmv : &tmk, &full[st], dh * 64, 0, h, id, pol);
        }
        __syncwarp();
      }
    }
  } else {
    // ---------------------------------------------------------- consumers
    // Q rows of this KV head -> shared (same swizzled layout as K), padding
    // zero; only the consumer warps wait for it (named barrier 1).
    for (int idx = threadIdx.x; idx < Mpad * CH; idx += n_cons * 32) {
      const int row = idx / CH, ch = idx - (idx / CH) * CH;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < M) {
        int i, qi;
        row_of(row, g, R, i, qi);
        const size_t off = ((size_t)(b * R + i) * p.num_q_heads + h * g + qi) * HD + ch * 8;
        v = *reinterpret_cast<const uint4*>(p.q + off);
      }
      *reinterpret_cast<uint4*>(qs + sw128_offset(row, ch, Mpad)) = v;
    }
    named_barrier_sync(1, n_cons * 32);
    // warp (mt, grp): rows [16 mt, 16 mt + 16) of tiles grp, grp + NG, ...
    // The ring depth is a multiple of NG, so a stage's previous phase was
    // consumed by this same group and a parity wait can never see it stale.
    const int mt = warp % MT, grp = warp / MT;
    const int r = lane >> 2, c = lane & 3;
    const int m0 = mt * 16 + r, m1 = m0 + 8;
    int lim0 = n_b - 1, lim1 = n_b - 1;  // last attended position of each row
    {
      int i, qi;
      if (m0 < M) { row_of(m0, g, R, i, qi); lim0 = L + i; }
      if (m1 < M) { row_of(m1, g, R, i, qi); lim1 = L + i; }
    }
    const uint32_t qs_u = smem_u32(qs);
    uint32_t qa[KS][4];
    const int qrow = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(qs_u + sw128_offset(qrow, 2 * ks + (lane >> 4), Mpad), qa[ks][0], qa[ks][1],
              qa[ks][2], qa[ks][3]);
    const bool cap_warp =
        (mt == 0) && (p.capture_mode == VG_CAPTURE_GROUP_SUM || p.capture_mode == VG_CAPTURE_ROWS);
    const bool cap_all = p.capture_mode == VG_CAPTURE_ALL_SUM;
    bool cap_live = true;  // false after a capture handshake timed out: wait no more
    float* cb = cbuf + grp * 16 * kCapStride;
    const uint32_t ring_u = smem_u32(ring);
    const int krow = (lane & 7) + ((lane >> 4) << 3);       // K ldmatrix row within 16
    const int kchk = (lane >> 3) & 1;                        // K ldmatrix chunk offset
    const int vrow = (lane & 7) + (((lane >> 3) & 1) << 3);  // V ldmatrix.trans row within 16
    const int vchk = lane >> 4;                              // V ldmatrix.trans chunk offset

    for (int lt = grp; lt < ntiles; lt += NG) {
      const int st = lt % stages;
      if (!mbar_wait(&full[st], (lt / stages) & 1)) {
        flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
        break;
      }
      const uint32_t kt = ring_u + st * kStageBytes, vt = kt + kTileBytes;
      const int tile_pos = (t0 + lt) * kTileN;

      // S = Q K^T for 16 rows x 64 positions: 8 independent accumulators
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt + sw128_offset(np * 16 + krow, 2 * ks + kchk, kTileN), b0, b1, b2, b3);
          mma_16816(s[2 * np], qa[ks], b0, b1);
          mma_16816(s[2 * np + 1], qa[ks], b2, b3);
        }
      }

      // Collect-2-Query capture (prefix positions only)
      if (cap_warp && tile_pos < L) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = nt * 8 + 2 * c;
          *reinterpret_cast<float2*>(&cb[r * kCapStride + col]) =
              make_float2(s[nt][0] * p.scale, s[nt][1] * p.scale);
          *reinterpret_cast<float2*>(&cb[(r + 8) * kCapStride + col]) =
              make_float2(s[nt][2] * p.scale, s[nt][3] * p.scale);
        }
        __syncwarp();
        const int s1 = (R > 1) ? g : 0;
#pragma unroll
        for (int jj = 0; jj < kTileN / 32; ++jj) {
          const int j = jj * 32 + lane;
          const int pos = tile_pos + j;
          if (pos < L) {
            if (p.capture_mode == VG_CAPTURE_GROUP_SUM) {
              float G = cb[j] + cb[s1 * kCapStride + j];
              for (int qi = 1; qi < g; ++qi)
                G = G + (cb[qi * kCapStride + j] + cb[(s1 + qi) * kCapStride + j]);
              p.capture[((size_t)b * p.num_kv_heads + h) * p.max_prefix + pos] = G;
            } else {
              for (int qi = 0; qi < g; ++qi) {
                const size_t base = ((size_t)b * p.num_q_heads + h * g + qi) * 2;
                p.capture[base * p.max_prefix + pos] = cb[qi * kCapStride + j];
                p.capture[(base + 1) * p.max_prefix + pos] = cb[(s1 + qi) * kCapStride + j];
              }
            }
          }
        }
        __syncwarp();
      }

      // Collect-All-Query capture: sum of every row of the tile's columns
      if (cap_all && tile_pos < L) {
        const int use_n = (lt - grp) / NG;  // this group's tile counter
        const int slot = use_n & 1, use = use_n >> 1;
        float* part = cpart + (size_t)(grp * 2 + slot) * MT * kTileN;
        float cs[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // rows r and r + 8 of this warp, then the 8 row pairs (lanes
            // with the same c) by a fixed butterfly; padded rows hold zeros
            float v = s[nt][e] * p.scale + s[nt][2 + e] * p.scale;
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            cs[nt][e] = v;
          }
        }
        if (mt != 0 && use > 0 && cap_live &&
            !mbar_wait(&capfree[grp * 2 + slot], (use - 1) & 1)) {
          flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
          cap_live = false;
        }
        if (r == 0) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            *reinterpret_cast<float2*>(&part[mt * kTileN + nt * 8 + 2 * c]) =
                make_float2(cs[nt][0], cs[nt][1]);
        }
        __syncwarp();
        if (mt != 0) {
          if (lane == 0) mbar_arrive(&capfull[grp * 2 + slot]);
        } else {
          if (MT > 1 && cap_live && !mbar_wait(&capfull[grp * 2 + slot], use & 1)) {
            flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
            cap_live = false;
          }
          if (cap_live) {
#pragma unroll
            for (int jj = 0; jj < kTileN / 32; ++jj) {
              const int j = jj * 32 + lane;
              const int pos = tile_pos + j;
              if (pos < L) {
                float A = part[j];
                for (int m2 = 1; m2 < MT; ++m2) A = A + part[m2 * kTileN + j];
                p.capture[((size_t)b * p.num_kv_heads + h) * p.max_prefix + pos] = A;
              }
            }
          }
          __syncwarp();
          if (MT > 1 && lane == 0) mbar_arrive(&capfree[grp * 2 + slot]);
        }
      }

      // online softmax (base 2); only the last tiles need the causal mask
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (tile_pos + kTileN <= L + 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            s[nt][e] *= p.scale_log2;
            s[nt][2 + e] *= p.scale_log2;
            mx0 = fmaxf(mx0, s[nt][e]);
            mx1 = fmaxf(mx1, s[nt][2 + e]);
          }
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = tile_pos + nt * 8 + 2 * c + e;
            s[nt][e] = (pos <= lim0) ? s[nt][e] * p.scale_log2 : -INFINITY;
            s[nt][2 + e] = (pos <= lim1) ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, s[nt][e]);
            mx1 = fmaxf(mx1, s[nt][2 + e]);
          }
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
      if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
        for (int dn = 0; dn < DN; ++dn) {
          acc[dn][0] *= corr0;
          acc[dn][1] *= corr0;
          acc[dn][2] *= corr1;
          acc[dn][3] *= corr1;
        }
      }
      uint32_t pa[NT / 2][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p00 = ex2(s[nt][0] - ref0), p01 = ex2(s[nt][1] - ref0);
        const float p10 = ex2(s[nt][2] - ref1), p11 = ex2(s[nt][3] - ref1);
        l0 += p00 + p01;
        l1 += p10 + p11;
        pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p00, p01);
        pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p10, p11);
      }

      // O += P V
      const bool ragged = tile_pos + kTileN > n_b;
#pragma unroll
      for (int kk = 0; kk < NT / 2; ++kk) {
        const int posA = tile_pos + kk * 16 + 2 * c;
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vt + sw128_offset(kk * 16 + vrow, 2 * dp + vchk, kTileN), v0, v1, v2, v3);
          if (ragged) {
            v0 = mask_pair(v0, posA, n_b);
            v2 = mask_pair(v2, posA, n_b);
            v1 = mask_pair(v1, posA + 8, n_b);
            v3 = mask_pair(v3, posA + 8, n_b);
          }
          mma_16816(acc[2 * dp], pa[kk], v0, v1);
          mma_16816(acc[2 * dp + 1], pa[kk], v2, v3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  __syncthreads();  // ring idle: every issued load was consumed

  // ---------------------------------------------- merge the NG tile groups
  float* sO = reinterpret_cast<float*>(ring);          // [n_cons][16][HD]
  float* sML = sO + (size_t)n_cons * 16 * HD;          // [n_cons][16][2]
  float* sW = sML + (size_t)n_cons * 16 * 2;           // [M][NG]
  float* sRow = sW + (size_t)Mpad * NG;                // [M][2]
  if (warp < n_cons) {
    float* o = sO + (size_t)warp * 16 * HD;
    const int r = lane >> 2, c = lane & 3;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      const int col = dn * 8 + 2 * c;
      *reinterpret_cast<float2*>(&o[r * HD + col]) = make_float2(acc[dn][0], acc[dn][1]);
      *reinterpret_cast<float2*>(&o[(r + 8) * HD + col]) = make_float2(acc[dn][2], acc[dn][3]);
    }
    if (c == 0) {
      sML[(warp * 16 + r) * 2] = mrun0;
      sML[(warp * 16 + r) * 2 + 1] = l0;
      sML[(warp * 16 + r + 8) * 2] = mrun1;
      sML[(warp * 16 + r + 8) * 2 + 1] = l1;
    }
  }
  __syncthreads();
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    const int mt = m >> 4, rr = m & 15;
    float mx = -INFINITY;
    for (int gq = 0; gq < NG; ++gq) mx = fmaxf(mx, sML[((gq * MT + mt) * 16 + rr) * 2]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
    for (int gq = 0; gq < NG; ++gq) {
      const float w = ex2(sML[((gq * MT + mt) * 16 + rr) * 2] - ref);
      sW[m * NG + gq] = w;
      lt += w * sML[((gq * MT + mt) * 16 + rr) * 2 + 1];
    }
    sRow[m * 2] = mx;
    sRow[m * 2 + 1] = lt;
    if (p.splits == 1) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      for (int gq = 0; gq < NG; ++gq) sW[m * NG + gq] *= inv;
    }
  }
  __syncthreads();

  const size_t bh = (size_t)b * p.num_kv_heads + h;
  if (p.splits == 1) {
    for (int e = threadIdx.x; e < M * (HD / 2); e += blockDim.x) {
      const int m = e / (HD / 2), d = (e - m * (HD / 2)) * 2;
      const int mt = m >> 4, rr = m & 15;
      float o0 = 0.f, o1 = 0.f;
      for (int gq = 0; gq < NG; ++gq) {
        const float w = sW[m * NG + gq];
        const float2 v =
            *reinterpret_cast<const float2*>(&sO[((size_t)(gq * MT + mt) * 16 + rr) * HD + d]);
        o0 += w * v.x;
        o1 += w * v.y;
      }
      int i, qi;
      row_of(m, g, R, i, qi);
      *reinterpret_cast<__nv_bfloat162*>(
          &p.out[((size_t)(b * R + i) * p.num_q_heads + h * g + qi) * HD + d]) =
          __floats2bfloat162_rn(o0, o1);
    }
    return;
  }

  // split-K: publish the partial; verify_merge_kernel combines the splits
  float* po = p.part_o + ((bh * p.splits + split) * M) * HD;
  float* pml = p.part_ml + (bh * p.splits + split) * M * 2;
  for (int e = threadIdx.x; e < M * (HD / 2); e += blockDim.x) {
    const int m = e / (HD / 2), d = (e - m * (HD / 2)) * 2;
    const int mt = m >> 4, rr = m & 15;
    float o0 = 0.f, o1 = 0.f;
    for (int gq = 0; gq < NG; ++gq) {
      const float w = sW[m * NG + gq];
      const float2 v =
          *reinterpret_cast<const float2*>(&sO[((size_t)(gq * MT + mt) * 16 + rr) * HD + d]);
      o0 += w * v.x;
      o1 += w * v.y;
    }
    *reinterpret_cast<float2*>(&po[(size_t)m * HD + d]) = make_float2(o0, o1);
  }
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    pml[m * 2] = sRow[m * 2];
    pml[m * 2 + 1] = sRow[m * 2 + 1];
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
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int L = p.prefix_lens[b];
  if (L < 1 || L > p.max_prefix ||
      (L + p.n_rows + kPageSize - 1) / kPageSize > p.max_pages_per_seq)
    return;  // the verify kernel skipped this sequence (and flagged it)
  const int M = p.m_rows, S = p.splits;
  const size_t bh = (size_t)b * p.num_kv_heads + h;
  int i, qi;
  row_of(m, p.group, p.n_rows, i, qi);
  merge_splits<HD>(p.part_o + (bh * S * M + m) * HD, (size_t)M * HD, p.part_ml + (bh * S * M + m) * 2,
                   (size_t)M * 2, S,
                   p.out + ((size_t)(b * p.n_rows + i) * p.num_q_heads + h * p.group + qi) * HD, smem_f);
}

struct VerifyPlan {
  int hd, m_rows, m_tiles, groups, splits, tiles_per_split, stages;
  size_t smem_bytes;
  size_t off_ml, ws_bytes;
};

bool make_verify_plan(int batch, int n_rows, int num_q_heads, int num_kv_heads, int head_dim,
                      int max_prefix, int num_splits, VerifyPlan* pl) {
  if (batch <= 0 || n_rows <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_prefix <= 0)
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->hd = head_dim;
  pl->m_rows = g * n_rows;
  pl->m_tiles = ceil_div(pl->m_rows, 16);
  // tile groups working on alternating tiles; consumers + producer <= 8 warps
  pl->groups = pl->m_tiles <= 2 ? 3 : (pl->m_tiles <= 3 ? 2 : 1);
  const int tiles = ceil_div(max_prefix + n_rows, kTileN);
  int tps;
  if (num_splits > 0) {
    tps = ceil_div(tiles, std::min(num_splits, tiles));
  } else {
    const int pairs = batch * num_kv_heads;
    const int sms = device_sm_count();
    int splits = std::max(1, sms / pairs);
    tps = ceil_div(tiles, splits);
    if (batch > 1) tps = std::min(tps, 32);  // ragged lengths: small chunks balance SMs
    tps = std::max(tps, std::min(tiles, 4));
  }
  if (ceil_div(tiles, tps) > kMaxSplits) tps = ceil_div(tiles, kMaxSplits);
  pl->tiles_per_split = tps;
  pl->splits = ceil_div(tiles, tps);
  const int stage_bytes = 2 * kTileN * head_dim * 2;
  const int n_cons = pl->m_tiles * pl->groups;
  const int mpad = pl->m_tiles * 16;
  auto smem_for = [&](int stages) {
    return 1024 + (size_t)stages * stage_bytes + (size_t)mpad * head_dim * 2 +
           (size_t)pl->groups * 16 * 72 * 4 + (size_t)pl->groups * 2 * pl->m_tiles * kTileN * 4 +
           2 * stages * 8 + 4 * pl->groups * 8 + 16;
  };
  // ring depth: a multiple of the group count (see the consumer loop), 192 KB
  // at head_dim 128, shrunk if the whole layout would not fit
  int stages = (head_dim == 128 ? 6 : 12);
  while (stages > pl->groups && smem_for(stages) > 227 * 1024) stages -= pl->groups;
  // the ring is reused after the main loop for the merge of the tile groups
  const size_t merge_bytes =
      (size_t)n_cons * 16 * (head_dim + 2) * 4 + (size_t)mpad * (pl->groups + 2) * 4;
  if ((size_t)stages * stage_bytes < merge_bytes) return false;
  pl->stages = stages;
  pl->smem_bytes = smem_for(stages);
  const size_t o_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * head_dim * 4;
  const size_t ml_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * 2 * 4;
  pl->off_ml = align_up(o_bytes, 256);
  pl->ws_bytes = pl->splits > 1 ? pl->off_ml + align_up(ml_bytes, 256) : 0;
  return true;
}

template <int HD>
cudaError_t launch_verify(const VerifyPlan& pl, const CUtensorMap& tk, const CUtensorMap& tv,
                          const VerifyParams& p, dim3 grid, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t vcfg = {};
  vcfg.gridDim = grid;
  vcfg.blockDim = dim3((pl.m_tiles * pl.groups + 1) * 32, 1, 1);
  vcfg.dynamicSmemBytes = pl.smem_bytes;
  vcfg.stream = stream;
  vcfg.attrs = pdl;
  vcfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&vcfg, verify_kernel<HD>, tk, tv, p);
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
      capture_mode != VG_CAPTURE_ROWS && capture_mode != VG_CAPTURE_ALL_SUM)
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

  VerifyParams p;
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
  p.splits = pl.splits;
  p.tiles_per_split = pl.tiles_per_split;
  p.stages = pl.stages;
  p.groups = pl.groups;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * kLog2e;
  dim3 grid(pl.splits, kv->num_kv_heads, batch);
  const cudaError_t e = kv->head_dim == 128 ? launch_verify<128>(pl, tk, tv, p, grid, stream)
                                             : launch_verify<64>(pl, tk, tv, p, grid, stream);
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
  uint8_t* scratch = static_cast<uint8_t*>(noalloc_scratch_on_current_device());
  if (!scratch) return VG_ERR_LAUNCH;
  // The array keeps the previous call's contents; nothing in it has to start
  // at zero: every partial is written before the merge reads it.
  return vg_verify_attention(kv, q, prefix_lens, batch, n_rows, num_q_heads, max_prefix,
                             softmax_scale, out, capture_mode, capture, num_splits, scratch,
                             kNoAllocScratchBytes, error_flag, stream);
}
