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
//  * Consumer warp (mt, pg) owns rows [16 mt, 16 mt + 16) and a 64/PG
//    position slice of every tile; it keeps its own online-softmax state.
//  * Capture epilogue: the first-tile warps stage their 16 x (64/PG) logits
//    in shared memory and write either the raw two rows or their per-KV-head
//    sum in a fixed order, with coalesced stores.
//  * Splits over the KV length are merged by the last CTA of each
//    (sequence, KV head) to finish (atomic ticket, no waiting).
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
  int32_t* tickets;   // [B][Hkv]
  int32_t* error_flag;
  int batch, n_rows, num_q_heads, num_kv_heads, group, m_rows, m_tiles;
  int max_prefix, max_pages_per_seq, num_pages;
  int capture_mode, splits, tiles_per_split, stages;
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

template <int HD>
struct VerifyLayout {
  static constexpr int kTileBytes = kTileN * HD * 2;     // one of K / V
  static constexpr int kStageBytes = 2 * kTileBytes;
};

template <int HD, int PG>
__global__ void __launch_bounds__(416, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const VerifyParams p) {
  constexpr int NPW = kTileN / PG;  // positions per warp per tile
  constexpr int NT = NPW / 8;       // S n-tiles per warp
  constexpr int KS = HD / 16;       // k-steps of Q K^T
  constexpr int DN = HD / 8;        // O n-tiles
  constexpr int CH = HD / 8;        // 16-byte chunks per row
  constexpr int kTileBytes = VerifyLayout<HD>::kTileBytes;
  constexpr int kStageBytes = VerifyLayout<HD>::kStageBytes;
  constexpr int kCapCols = 32;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, R = p.n_rows, M = p.m_rows;
  const int n_cons = p.m_tiles * PG;
  const int Mpad = p.m_tiles * 16;
  const int stages = p.stages;

  uint8_t* ring = smem;
  uint8_t* qs = ring + stages * kStageBytes;
  float* cbuf = reinterpret_cast<float*>(qs + Mpad * HD * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(cbuf + PG * 16 * kCapCols);
  uint64_t* empty = full + stages;
  int* s_flag = reinterpret_cast<int*>(empty + stages);

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
      mbar_init(&empty[s], n_cons);
    }
    fence_barrier_init();
  }
  // Q rows of this KV head -> shared (same swizzled layout as K), padding zero.
  for (int idx = threadIdx.x; idx < Mpad * CH; idx += blockDim.x) {
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
  __syncthreads();

  float mrun0 = -INFINITY, mrun1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;

  if (warp == n_cons) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const uint64_t pol = l2_policy_evict_first();
      for (int lt = 0; lt < ntiles; ++lt) {
        const int st = lt % stages;
        if (lt >= stages && !mbar_wait(&empty[st], ((lt / stages) - 1) & 1)) {
          flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
          break;
        }
        uint8_t* kt = ring + st * kStageBytes;
        uint8_t* vt = kt + kTileBytes;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
#pragma unroll
        for (int pi = 0; pi < kTileN / kPageSize; ++pi) {
          const int lp = (t0 + lt) * (kTileN / kPageSize) + pi;
          int phys = p.num_pages;  // out of range: TMA fills zeros
          if (lp < npages_b) {
            const int e = p.page_table[(size_t)b * p.max_pages_per_seq + lp];
            if (e >= 0 && e < p.num_pages)
              phys = e;
            else
              flag_error(p.error_flag, VG_DEVERR_PAGE);
          }
#pragma unroll
          for (int dh = 0; dh < HD / 64; ++dh) {
            const int off = dh * kTileN * 128 + pi * kPageSize * 128;
            tma_load_4d(kt + off, &tmk, &full[st], dh * 64, 0, h, phys, pol);
            tma_load_4d(vt + off, &tmv, &full[st], dh * 64, 0, h, phys, pol);
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------- consumers
    const int mt = warp / PG, pg = warp - (warp / PG) * PG;
    const int r = lane >> 2, c = lane & 3;
    const int m0 = mt * 16 + r, m1 = m0 + 8;
    int lim0 = n_b - 1, lim1 = n_b - 1;  // last attended position of each row
    {
      int i, qi;
      if (m0 < M) { row_of(m0, g, R, i, qi); lim0 = L + i; }
      if (m1 < M) { row_of(m1, g, R, i, qi); lim1 = L + i; }
    }
    // Q fragments: held in registers by the 4-slice variant; the 2-slice
    // variant (many row tiles, more warps) re-reads them per tile instead.
    constexpr bool kQReg = (PG == 4);
    const uint32_t qs_u = smem_u32(qs);
    uint32_t qa[kQReg ? KS : 1][4];
    const int qrow = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
    if (kQReg) {
#pragma unroll
      for (int ks = 0; ks < (kQReg ? KS : 1); ++ks)
        ldsm_x4(qs_u + sw128_offset(qrow, 2 * ks + (lane >> 4), Mpad), qa[ks][0], qa[ks][1],
                qa[ks][2], qa[ks][3]);
    }
    const bool cap_warp = (mt == 0) && (p.capture_mode != VG_CAPTURE_NONE);
    float* cb = cbuf + pg * 16 * kCapCols;
    const uint32_t ring_u = smem_u32(ring);

    for (int lt = 0; lt < ntiles; ++lt) {
      const int st = lt % stages;
      if (!mbar_wait(&full[st], (lt / stages) & 1)) {
        flag_error(p.error_flag, VG_DEVERR_TIMEOUT);
        break;
      }
      const uint32_t kt = ring_u + st * kStageBytes, vt = kt + kTileBytes;
      const int tile_pos = (t0 + lt) * kTileN;
      const int pbase = tile_pos + pg * NPW;

      // S = Q K^T for 16 rows x NPW positions
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        if (kQReg) {
          a[0] = qa[kQReg ? ks : 0][0];
          a[1] = qa[kQReg ? ks : 0][1];
          a[2] = qa[kQReg ? ks : 0][2];
          a[3] = qa[kQReg ? ks : 0][3];
        } else {
          ldsm_x4(qs_u + sw128_offset(qrow, 2 * ks + (lane >> 4), Mpad), a[0], a[1], a[2], a[3]);
        }
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int prow = pg * NPW + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt + sw128_offset(prow, 2 * ks + ((lane >> 3) & 1), kTileN), b0, b1, b2, b3);
          mma_16816(s[2 * np], a, b0, b1);
          mma_16816(s[2 * np + 1], a, b2, b3);
        }
      }

      // Collect-2-Query capture (prefix positions only)
      if (cap_warp && pbase < L) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = nt * 8 + 2 * c;
          cb[r * kCapCols + col] = s[nt][0] * p.scale;
          cb[r * kCapCols + col + 1] = s[nt][1] * p.scale;
          cb[(r + 8) * kCapCols + col] = s[nt][2] * p.scale;
          cb[(r + 8) * kCapCols + col + 1] = s[nt][3] * p.scale;
        }
        __syncwarp();
        if (lane < NPW) {
          const int pos = pbase + lane;
          if (pos < L) {
            const int s1 = (R > 1) ? g : 0;
            if (p.capture_mode == VG_CAPTURE_GROUP_SUM) {
              float G = cb[lane] + cb[s1 * kCapCols + lane];
              for (int qi = 1; qi < g; ++qi)
                G = G + (cb[qi * kCapCols + lane] + cb[(s1 + qi) * kCapCols + lane]);
              p.capture[((size_t)b * p.num_kv_heads + h) * p.max_prefix + pos] = G;
            } else {
              for (int qi = 0; qi < g; ++qi) {
                const size_t base = ((size_t)b * p.num_q_heads + h * g + qi) * 2;
                p.capture[base * p.max_prefix + pos] = cb[qi * kCapCols + lane];
                p.capture[(base + 1) * p.max_prefix + pos] = cb[(s1 + qi) * kCapCols + lane];
              }
            }
          }
        }
        __syncwarp();
      }

      // online softmax (base 2)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = pbase + nt * 8 + 2 * c + e;
          s[nt][e] = (pos <= lim0) ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][2 + e] = (pos <= lim1) ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
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
        const int p0 = pg * NPW + kk * 16;
        const int mi = lane >> 3;
        const int prow = p0 + (lane & 7) + ((mi & 1) << 3);
        const int posA = tile_pos + p0 + 2 * c;
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vt + sw128_offset(prow, 2 * dp + (mi >> 1), kTileN), v0, v1, v2, v3);
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

  // ---------------------------------------------- merge the PG slices
  float* sO = reinterpret_cast<float*>(ring);          // [n_cons][16][HD]
  float* sML = sO + (size_t)n_cons * 16 * HD;          // [n_cons][16][2]
  float* sW = sML + (size_t)n_cons * 16 * 2;           // [M][PG]
  float* sRow = sW + (size_t)Mpad * PG;                // [M][2]
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
    for (int pg = 0; pg < PG; ++pg) mx = fmaxf(mx, sML[((mt * PG + pg) * 16 + rr) * 2]);
    const float ref = safe_ref(mx);
    float lt = 0.f;
    for (int pg = 0; pg < PG; ++pg) {
      const float w = ex2(sML[((mt * PG + pg) * 16 + rr) * 2] - ref);
      sW[m * PG + pg] = w;
      lt += w * sML[((mt * PG + pg) * 16 + rr) * 2 + 1];
    }
    sRow[m * 2] = mx;
    sRow[m * 2 + 1] = lt;
    if (p.splits == 1) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      for (int pg = 0; pg < PG; ++pg) sW[m * PG + pg] *= inv;
    }
  }
  __syncthreads();

  const size_t bh = (size_t)b * p.num_kv_heads + h;
  if (p.splits == 1) {
    for (int e = threadIdx.x; e < M * (HD / 2); e += blockDim.x) {
      const int m = e / (HD / 2), d = (e - m * (HD / 2)) * 2;
      const int mt = m >> 4, rr = m & 15;
      float o0 = 0.f, o1 = 0.f;
      for (int pg = 0; pg < PG; ++pg) {
        const float w = sW[m * PG + pg];
        const float2 v = *reinterpret_cast<const float2*>(&sO[((size_t)(mt * PG + pg) * 16 + rr) * HD + d]);
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

  // split-K: publish the partial, the last CTA of (b, h) merges
  float* po = p.part_o + ((bh * p.splits + split) * M) * HD;
  float* pml = p.part_ml + (bh * p.splits + split) * M * 2;
  for (int e = threadIdx.x; e < M * (HD / 2); e += blockDim.x) {
    const int m = e / (HD / 2), d = (e - m * (HD / 2)) * 2;
    const int mt = m >> 4, rr = m & 15;
    float o0 = 0.f, o1 = 0.f;
    for (int pg = 0; pg < PG; ++pg) {
      const float w = sW[m * PG + pg];
      const float2 v = *reinterpret_cast<const float2*>(&sO[((size_t)(mt * PG + pg) * 16 + rr) * HD + d]);
      o0 += w * v.x;
      o1 += w * v.y;
    }
    *reinterpret_cast<float2*>(&po[(size_t)m * HD + d]) = make_float2(o0, o1);
  }
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    pml[m * 2] = sRow[m * 2];
    pml[m * 2 + 1] = sRow[m * 2 + 1];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_flag = (atomicAdd(&p.tickets[bh], 1) == p.splits - 1);
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();

  float* sWs = reinterpret_cast<float*>(ring);  // [splits][M]
  const float* mlb = p.part_ml + bh * p.splits * M * 2;
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    float mx = -INFINITY;
    for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, __ldcg(&mlb[((size_t)s * M + m) * 2]));
    const float ref = safe_ref(mx);
    float lt = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float w = ex2(__ldcg(&mlb[((size_t)s * M + m) * 2]) - ref);
      sWs[s * M + m] = w;
      lt += w * __ldcg(&mlb[((size_t)s * M + m) * 2 + 1]);
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    for (int s = 0; s < p.splits; ++s) sWs[s * M + m] *= inv;
  }
  __syncthreads();
  const float* pob = p.part_o + bh * p.splits * M * HD;
  for (int e = threadIdx.x; e < M * (HD / 4); e += blockDim.x) {
    const int m = e / (HD / 4), d = (e - m * (HD / 4)) * 4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.splits; ++s) {
      const float w = sWs[s * M + m];
      const float4 v = __ldcg(reinterpret_cast<const float4*>(&pob[((size_t)s * M + m) * HD + d]));
      o.x += w * v.x;
      o.y += w * v.y;
      o.z += w * v.z;
      o.w += w * v.w;
    }
    int i, qi;
    row_of(m, g, R, i, qi);
    __nv_bfloat16* dst = &p.out[((size_t)(b * R + i) * p.num_q_heads + h * g + qi) * HD + d];
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(o.x, o.y);
    *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(o.z, o.w);
  }
  if (threadIdx.x == 0) p.tickets[bh] = 0;
}

struct VerifyPlan {
  int hd, m_rows, m_tiles, pg, splits, tiles_per_split, stages;
  size_t smem_bytes;
  size_t off_ml, off_tickets, ws_bytes;
};

bool make_verify_plan(int batch, int n_rows, int num_q_heads, int num_kv_heads, int head_dim,
                      int max_prefix, int num_splits, VerifyPlan* pl) {
  if (batch <= 0 || n_rows <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_prefix <= 0)
    return false;
  const int g = num_q_heads / num_kv_heads;
  pl->hd = head_dim;
  pl->m_rows = g * n_rows;
  pl->m_tiles = ceil_div(pl->m_rows, 16);
  pl->pg = pl->m_tiles <= 3 ? 4 : 2;
  const int tiles = ceil_div(max_prefix + n_rows, kTileN);
  int tps;
  if (num_splits > 0) {
    tps = ceil_div(tiles, std::min(num_splits, tiles));
  } else {
    const int pairs = batch * num_kv_heads;
    const int sms = device_sm_count();
    const int splits = std::max(1, sms / pairs);
    tps = ceil_div(tiles, splits);
    if (batch > 1) tps = std::min(tps, 32);  // ragged lengths: small chunks balance SMs
    tps = std::max(tps, std::min(tiles, 4));
  }
  if (ceil_div(tiles, tps) > kMaxSplits) tps = ceil_div(tiles, kMaxSplits);
  pl->tiles_per_split = tps;
  pl->splits = ceil_div(tiles, tps);
  const int stage_bytes = 2 * kTileN * head_dim * 2;
  const int n_cons = pl->m_tiles * pl->pg;
  const int mpad = pl->m_tiles * 16;
  // the ring is reused after the main loop for the slice merge and the split merge
  const size_t merge_bytes =
      std::max((size_t)n_cons * 16 * (head_dim + 2) * 4 + (size_t)mpad * (pl->pg + 2) * 4,
               (size_t)pl->splits * pl->m_rows * 4);
  pl->stages = std::max(4, (int)ceil_div((int)merge_bytes, stage_bytes));
  pl->smem_bytes = 1024 + (size_t)pl->stages * stage_bytes + (size_t)mpad * head_dim * 2 +
                   (size_t)pl->pg * 16 * 32 * 4 + 2 * pl->stages * 8 + 16;
  const size_t o_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * head_dim * 4;
  const size_t ml_bytes = (size_t)batch * num_kv_heads * pl->splits * pl->m_rows * 2 * 4;
  pl->off_ml = align_up(o_bytes, 256);
  pl->off_tickets = pl->off_ml + align_up(ml_bytes, 256);
  pl->ws_bytes = pl->splits > 1 ? pl->off_tickets + align_up((size_t)batch * num_kv_heads * 4, 256)
                                 : 0;
  return true;
}

template <int HD, int PG>
cudaError_t launch_verify(const VerifyPlan& pl, const CUtensorMap& tk, const CUtensorMap& tv,
                          const VerifyParams& p, dim3 grid, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  static size_t attr_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && (!attr_set[dev] || attr_bytes[dev] < pl.smem_bytes)) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel<HD, PG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)std::max<size_t>(pl.smem_bytes, 200 * 1024));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
    attr_bytes[dev] = std::max<size_t>(pl.smem_bytes, 200 * 1024);
  }
  const int threads = (pl.m_tiles * PG + 1) * 32;
  verify_kernel<HD, PG><<<grid, threads, pl.smem_bytes, stream>>>(tk, tv, p);
  return cudaGetLastError();
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
      capture_mode != VG_CAPTURE_ROWS)
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
  p.tickets = pl.ws_bytes ? reinterpret_cast<int32_t*>(ws + pl.off_tickets) : nullptr;
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
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * kLog2e;
  dim3 grid(pl.splits, kv->num_kv_heads, batch);
  cudaError_t e;
  if (kv->head_dim == 128)
    e = pl.pg == 4 ? launch_verify<128, 4>(pl, tk, tv, p, grid, stream)
                   : launch_verify<128, 2>(pl, tk, tv, p, grid, stream);
  else
    e = pl.pg == 4 ? launch_verify<64, 4>(pl, tk, tv, p, grid, stream)
                   : launch_verify<64, 2>(pl, tk, tv, p, grid, stream);
  return e == cudaSuccess ? VG_OK : VG_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of vg_verify_attention (declared in vg.h).
//
// Its split partials and merge tickets live in one file-scope device array of
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
  if (pl.ws_bytes > 0) {
    // The array keeps the previous call's contents: the merge tickets must
    // start at zero, the partials are always written before they are read.
    if (cudaMemsetAsync(scratch + pl.off_tickets, 0, (size_t)batch * kv->num_kv_heads * 4,
                        stream) != cudaSuccess)
      return VG_ERR_LAUNCH;
  }
  return vg_verify_attention(kv, q, prefix_lens, batch, n_rows, num_q_heads, max_prefix,
                             softmax_scale, out, capture_mode, capture, num_splits, scratch,
                             kNoAllocScratchBytes, error_flag, stream);
}
