// Device code shared by the split-KV decode kernels (decode.cu,
// decode_fp16.cu): online softmax, per-CTA merge of the warps' partial
// softmax states, and the last-CTA merge of the split partials.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace vqkv {
namespace {

constexpr float kSoftmaxSlack = 8.0f;   // rescale only when a score exceeds m by 2^8

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
// Initial running max: finite, so exp2(m_old - m_new) and exp2(score - m)
// never see inf - inf; masked scores are -inf and give p = 0.
constexpr float kMInit = -1e30f;

// Combine area (floats), used after the tile loop: each warp's O rows (one
// per softmax column, pitch kPitch: 128 channels after a per-column skew of
// up to 31 floats that spreads the stash stores over the banks), then the
// warps' m, l, their scale factors and the CTA's max per column.
template <int WARPS>
struct CombineSmem {
  static constexpr int kPitch = kHeadDim + 32;   // a multiple of 32: the pitch itself is bank-neutral
  static constexpr int kO = WARPS * 8 * kPitch;
  static constexpr int kM = kO, kL = kM + WARPS * 8, kF = kL + WARPS * 8, kMax = kF + WARPS * 8;
  static constexpr int kBytes = (kMax + 8) * 4;
};

// Clamp the sequence length to [0, max_seq_len]; report out-of-range once.
__device__ __forceinline__ int load_len(const DecodeParams& p, int b) {
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_seq_len) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.err, VQKV_DEVERR_SEQ_LEN);
    L = L < 0 ? 0 : p.max_seq_len;
  }
  return L;
}

// Online-softmax update for one tile.  sc = scores for tokens {gid, gid+8}
// x heads {2tig, 2tig+1} (log2 domain).  Returns P packed for the P.V MMA.
template <int NACC>
__device__ __forceinline__ void softmax_tile(float (&sc)[4], float& m0, float& m1, float& l0,
                                             float& l1, float (&acc)[NACC][4], uint32_t& bP0,
                                             uint32_t& bP1) {
  const bool need = (sc[0] > m0 + kSoftmaxSlack) | (sc[2] > m0 + kSoftmaxSlack) |
                    (sc[1] > m1 + kSoftmaxSlack) | (sc[3] > m1 + kSoftmaxSlack);
  if (__any_sync(0xffffffffu, need)) {
    float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    const float a0 = fast_exp2(m0 - n0);
    const float a1 = fast_exp2(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      acc[i][0] *= a0;
      acc[i][1] *= a1;
      acc[i][2] *= a0;
      acc[i][3] *= a1;
    }
  }
  const float p0 = fast_exp2(sc[0] - m0), p1 = fast_exp2(sc[1] - m1);
  const float p2 = fast_exp2(sc[2] - m0), p3 = fast_exp2(sc[3] - m1);
  l0 += p0 + p2;
  l1 += p1 + p3;
  bP0 = movmatrix_t(pack_half2(p0, p1));   // P[tokens 2tig, 2tig+1][head gid]
  bP1 = movmatrix_t(pack_half2(p2, p3));   // P[tokens 2tig+8, 2tig+9][head gid]
}

// Online-softmax update for T tiles at once (one running max for all of
// them), then P packed for the P.V MMA of each tile.
template <int T, int NACC>
__device__ __forceinline__ void softmax_tiles(float (&sc)[T][4], float& m0, float& m1, float& l0, float& l1,
                                              float (&acc)[NACC][4], uint32_t (&bP)[T][2]) {
  bool need = false;
#pragma unroll
  for (int i = 0; i < T; ++i)
    need |= (sc[i][0] > m0 + kSoftmaxSlack) | (sc[i][2] > m0 + kSoftmaxSlack) |
            (sc[i][1] > m1 + kSoftmaxSlack) | (sc[i][3] > m1 + kSoftmaxSlack);
  if (__any_sync(0xffffffffu, need)) {
    float x0 = fmaxf(sc[0][0], sc[0][2]), x1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
    for (int i = 1; i < T; ++i) {
      x0 = fmaxf(x0, fmaxf(sc[i][0], sc[i][2]));
      x1 = fmaxf(x1, fmaxf(sc[i][1], sc[i][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
    m0 = n0;
    m1 = n1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int i = 0; i < NACC; ++i) {
      acc[i][0] *= a0;
      acc[i][1] *= a1;
      acc[i][2] *= a0;
      acc[i][3] *= a1;
    }
  }
#pragma unroll
  for (int i = 0; i < T; ++i) {
    const float p0 = fast_exp2(sc[i][0] - m0), p1 = fast_exp2(sc[i][1] - m1);
    const float p2 = fast_exp2(sc[i][2] - m0), p3 = fast_exp2(sc[i][3] - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    bP[i][0] = movmatrix_t(pack_half2(p0, p1));
    bP[i][1] = movmatrix_t(pack_half2(p2, p3));
  }
}

// Offset of O's row for softmax column c (query c / g, head c % g) of KV
// head kvh of sequence b; O is [B][M][Hq][128].
__device__ __forceinline__ size_t out_row(const DecodeParams& p, int b, int kvh, int c) {
  const int m = c / p.g, h = c - m * p.g;
  return (((size_t)b * p.M + m) * p.Hq + kvh * p.g + h) * kHeadDim;
}

// Per-lane visible-token limits of the lane's two softmax columns col0 +
// 2tig and col0 + 2tig + 1 (col0: the CTA's first column): query m of M
// sees tokens t < L - M + m + 1 (columns past ncols are padding and see all
// L).  lim_min is the smallest limit of any column.
struct ColumnLimits {
  int lim0, lim1, lim_min;
};
__device__ __forceinline__ ColumnLimits column_limits(const DecodeParams& p, int L, int tig, int col0) {
  const int c0 = col0 + 2 * tig, c1 = c0 + 1;
  return {c0 < p.ncols ? L - p.M + c0 / p.g + 1 : L, c1 < p.ncols ? L - p.M + c1 / p.g + 1 : L, L - p.M + 1};
}

// Masks the scores of tokens t0 (sc[0], sc[1]) and t0 + 8 (sc[2], sc[3]) in
// columns 2tig, 2tig+1 that their query does not see.
__device__ __forceinline__ void mask_scores(float (&sc)[4], int t0, const ColumnLimits& cl) {
  if (t0 >= cl.lim0) sc[0] = neg_inf();
  if (t0 >= cl.lim1) sc[1] = neg_inf();
  if (t0 + 8 >= cl.lim0) sc[2] = neg_inf();
  if (t0 + 8 >= cl.lim1) sc[3] = neg_inf();
}

// Merge the per-warp states of the CTA into one partial (m, l, O) per head.
// With one split that is O itself.  Otherwise write the partial to the
// workspace; then, when the plan defers the merge (CTAs that cover several
// sequences must not stall between them), the combine kernel merges the
// splits after the decode kernel.  Else take the (b, kvh) ticket; the CTA
// that arrives last merges all split partials into O (fp16).  Ordering: the CTA's partial stores
// happen before thread 0's acq_rel ticket increment (CTA barrier, then a
// cumulative gpu-scope release); the last CTA's acquire and the barrier
// after it order its partial loads after every other CTA's stores.
// Query layout a decode kernel is compiled for: one query per sequence,
// several with all columns in one CTA, or several in column groups.
enum QueryLayout : int { kOneQuery = 0, kQueries = 1, kQueryGroups = 2 };

// The CTA's columns: col0 .. col0 + nloc - 1 of the KV head's ncols
// (column group blockIdx.z % cgroups).
__device__ __forceinline__ int cta_col0(const DecodeParams& p) { return 8 * (int)(blockIdx.z % p.cgroups); }
__device__ __forceinline__ int cta_bgroup(const DecodeParams& p) { return (int)(blockIdx.z / p.cgroups); }

// The CTAs that contribute to one (sequence, KV head, column group): this
// CTA is number `part` of `n_parts`; the partials of all of them are rows
// ncols * kPartialStride floats apart starting `first` floats into
// p.partials (at the CTA's first column).
struct MergeSpan {
  int part, n_parts;
  size_t first;
};

// Split plan: CTA `split` of p.n_splits, partials [B][Hkv][n_splits][ncols].
__device__ __forceinline__ MergeSpan split_span(const DecodeParams& p, int b, int kvh, int split, int col0) {
  return {split, p.n_splits, ((size_t)(b * p.Hkv + kvh) * p.n_splits * p.ncols + col0) * kPartialStride};
}

// COLGROUPS: the launch may split the columns into groups (multi-query
// decode); otherwise the CTA holds all ncols columns.  DimOf: the stash
// layout (row skew).
template <int WARPS, bool COLGROUPS, typename DimOf>
__device__ __forceinline__ void finish_sequence(const DecodeParams& p, int b, int kvh, const MergeSpan& ms,
                                                float* s_comb, int* s_last) {
  using C = CombineSmem<WARPS>;
  const float* wO = s_comb;
  const float* wm = s_comb + C::kM;
  const float* wl = s_comb + C::kL;
  float* wf = s_comb + C::kF;
  float* wM = s_comb + C::kMax;
  const int col0 = COLGROUPS ? cta_col0(p) : 0;
  const int G = COLGROUPS ? min(8, p.ncols - col0) : p.ncols;   // this CTA's columns
  const size_t split_stride = (size_t)p.ncols * kPartialStride;
  float* part = p.partials + ms.first + (size_t)ms.part * split_stride;
  const int n_parts = ms.n_parts;
  const unsigned ticket = COLGROUPS ? (unsigned)((b * p.Hkv + kvh) * p.cgroups + blockIdx.z % p.cgroups)
                                    : (unsigned)(b * p.Hkv + kvh);
  // each warp's scale against the CTA's max of the column, once per (warp,
  // column) rather than once per output
  for (int i = threadIdx.x; i < WARPS * 8; i += WARPS * 32) {
    const int h = i & 7;
    float M = kMInit;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, wm[w * 8 + h]);
    wf[i] = fast_exp2(wm[i] - M);
    if (i < 8) wM[h] = M;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * kHeadDim; e += WARPS * 32) {
    const int h = e >> 7, d = e & 127;
    const float* col = wO + h * C::kPitch + DimOf::skew(h) + d;
    float o = 0.f;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) o += col[w * 8 * C::kPitch] * wf[w * 8 + h];
    if (n_parts == 1 || d == 0) {
      float l = 0.f;
#pragma unroll 4
      for (int w = 0; w < WARPS; ++w) l += wl[w * 8 + h] * wf[w * 8 + h];
      if (n_parts == 1) {
        p.out[out_row(p, b, kvh, col0 + h) + d] = __float2half_rn(l > 0.f ? o / l : 0.f);
        continue;
      }
      part[h * kPartialStride + 128] = wM[h];
      part[h * kPartialStride + 129] = l;
    }
    part[h * kPartialStride + d] = o;
  }
  if (n_parts == 1 || p.defer_merge) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.tickets + ticket)
                 : "memory");
    *s_last = (prev == (unsigned)(n_parts - 1));
  }
  __syncthreads();
  if (*s_last) {
    // Thread t merges 8 channels of one column (item t % items) over every
    // R-th split (t / items), straight from the partials: a batch of splits
    // has all its loads in flight at once and one rescale; the R threads of
    // an item then meet in shared memory.
    constexpr int THREADS = WARPS * 32, BATCH = 6;
    const float* base = p.partials + ms.first;
    const int items = G * (kHeadDim / 8), R = THREADS / items;
    const int item = threadIdx.x % items, r = threadIdx.x / items;
    const int h = item / (kHeadDim / 8), d8 = (item % (kHeadDim / 8)) * 8;
    float M = kMInit, Ls = 0.f, O[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) O[i] = 0.f;
    if (r < R) {
      const float* col = base + h * kPartialStride;
      for (int s0 = r; s0 < n_parts; s0 += BATCH * R) {
        float2 ml[BATCH];
        float4 oa[BATCH], ob[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
          const int sp = s0 + j * R;
          if (sp < n_parts) {
            const float* ph = col + (size_t)sp * split_stride;
            ml[j] = __ldcg(reinterpret_cast<const float2*>(ph + 128));
            oa[j] = __ldcg(reinterpret_cast<const float4*>(ph + d8));
            ob[j] = __ldcg(reinterpret_cast<const float4*>(ph + d8 + 4));
          } else {
            ml[j] = make_float2(kMInit, 0.f);
            oa[j] = ob[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        float n = M;
#pragma unroll
        for (int j = 0; j < BATCH; ++j) n = fmaxf(n, ml[j].x);
        const float fa = fast_exp2(M - n);
        Ls *= fa;
#pragma unroll
        for (int i = 0; i < 8; ++i) O[i] *= fa;
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
          const float f = fast_exp2(ml[j].x - n);
          Ls += ml[j].y * f;
          O[0] += oa[j].x * f, O[1] += oa[j].y * f, O[2] += oa[j].z * f, O[3] += oa[j].w * f;
          O[4] += ob[j].x * f, O[5] += ob[j].y * f, O[6] += ob[j].z * f, O[7] += ob[j].w * f;
        }
        M = n;
      }
    }
    if (R > 1) {   // [R][items] states of 12 floats (m, l, O[8], pad)
      float* xs = s_comb + (size_t)threadIdx.x * 12;
      if (r < R) {
        *reinterpret_cast<float4*>(xs) = make_float4(M, Ls, 0.f, 0.f);
        *reinterpret_cast<float4*>(xs + 4) = make_float4(O[0], O[1], O[2], O[3]);
        *reinterpret_cast<float4*>(xs + 8) = make_float4(O[4], O[5], O[6], O[7]);
      }
      __syncthreads();
      if (r == 0) {
        for (int q = 1; q < R; ++q) {
          const float* ys = s_comb + (size_t)(q * items + item) * 12;
          const float4 y0 = *reinterpret_cast<const float4*>(ys);
          const float4 y1 = *reinterpret_cast<const float4*>(ys + 4);
          const float4 y2 = *reinterpret_cast<const float4*>(ys + 8);
          const float n = fmaxf(M, y0.x);
          const float fa = fast_exp2(M - n), fb = fast_exp2(y0.x - n);
          Ls = Ls * fa + y0.y * fb;
          O[0] = O[0] * fa + y1.x * fb, O[1] = O[1] * fa + y1.y * fb;
          O[2] = O[2] * fa + y1.z * fb, O[3] = O[3] * fa + y1.w * fb;
          O[4] = O[4] * fa + y2.x * fb, O[5] = O[5] * fa + y2.y * fb;
          O[6] = O[6] * fa + y2.z * fb, O[7] = O[7] * fa + y2.w * fb;
          M = n;
        }
      }
    }
    if (r == 0) {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      uint4 packed;
      packed.x = pack_half2(O[0] * inv, O[1] * inv);
      packed.y = pack_half2(O[2] * inv, O[3] * inv);
      packed.z = pack_half2(O[4] * inv, O[5] * inv);
      packed.w = pack_half2(O[6] * inv, O[7] * inv);
      __half* dst = p.out + out_row(p, b, kvh, col0 + h) + d8;
      if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {   // out needs only 2-byte alignment
        *reinterpret_cast<uint4*>(dst) = packed;
      } else {
        const uint32_t w[4] = {packed.x, packed.y, packed.z, packed.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[2 * i] = __ushort_as_half((unsigned short)(w[i] & 0xffffu));
          dst[2 * i + 1] = __ushort_as_half((unsigned short)(w[i] >> 16));
        }
      }
    }
    if (threadIdx.x == 0) p.tickets[ticket] = 0u;   // ready for the next call
  }
}

// Merge the split partials of softmax column blockIdx.x % ncols of KV head
// blockIdx.x / ncols of sequence b = blockIdx.y into O (fp16); thread d owns
// channel d.  The combine kernel
// of plans that defer the merge.
__device__ __forceinline__ void combine_splits(const DecodeParams& p) {
  constexpr int U = 8;   // splits whose loads are in flight together
  const int b = blockIdx.y, d = threadIdx.x;
  const int kvh = blockIdx.x / p.ncols, h = blockIdx.x - kvh * p.ncols;   // h: softmax column
  const size_t stride = (size_t)p.ncols * kPartialStride;
  const float* base = p.partials + (size_t)(b * p.Hkv + kvh) * p.n_splits * stride + h * kPartialStride;
  float M = kMInit, O = 0.f, Ls = 0.f;
  for (int s0 = 0; s0 < p.n_splits; s0 += U) {
    float ms[U], ls[U], os[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool in = s0 + u < p.n_splits;
      const float* ph = base + (in ? s0 + u : 0) * stride;
      ms[u] = in ? __ldcg(ph + 128) : kMInit;
      ls[u] = in ? __ldcg(ph + 129) : 0.f;
      os[u] = in ? __ldcg(ph + d) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float n = fmaxf(M, ms[u]);
      const float fa = fast_exp2(M - n), fb = fast_exp2(ms[u] - n);
      O = O * fa + os[u] * fb;
      Ls = Ls * fa + ls[u] * fb;
      M = n;
    }
  }
  p.out[out_row(p, b, kvh, h) + d] = __float2half_rn(Ls > 0.f ? O / Ls : 0.f);
}

// Store one warp's (m, l, O) into the combine area.  acc holds O^T fragments:
// acc[mt] = rows {gid, gid+8} (channels dim_of(mt, gid), dim_of(mt, gid+8))
// x heads {2tig, 2tig+1}.  Row h of the warp starts DimOf::skew(h) floats
// into its pitch; with that skew the stores of a warp fall on distinct banks.
template <int WARPS, int NMT, typename DimOf>
__device__ __forceinline__ void stash_warp(float* s_comb, int warp, int lane, const float (&acc)[NMT][4],
                                           float m0, float m1, float l0, float l1, DimOf dim_of) {
  using C = CombineSmem<WARPS>;
  const int gid = lane >> 2, tig = lane & 3;
  float* wm = s_comb + C::kM;
  float* wl = s_comb + C::kL;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const int h0 = 2 * tig;
  float* r0 = s_comb + (warp * 8 + h0) * C::kPitch + DimOf::skew(h0);
  float* r1 = s_comb + (warp * 8 + h0 + 1) * C::kPitch + DimOf::skew(h0 + 1);
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt) {
    const int d0 = dim_of(mt, gid), d1 = dim_of(mt, gid + 8);
    if (DimOf::kPairs) {   // d1 == d0 + 1, d0 even
      *reinterpret_cast<float2*>(r0 + d0) = make_float2(acc[mt][0], acc[mt][2]);
      *reinterpret_cast<float2*>(r1 + d0) = make_float2(acc[mt][1], acc[mt][3]);
    } else {
      r0[d0] = acc[mt][0];
      r1[d0] = acc[mt][1];
      r0[d1] = acc[mt][2];
      r1[d1] = acc[mt][3];
    }
  }
  if (gid == 0) {
    wm[warp * 8 + h0] = m0;
    wm[warp * 8 + h0 + 1] = m1;
    wl[warp * 8 + h0] = l0;
    wl[warp * 8 + h0 + 1] = l1;
  }
}

// Channel held by row r (0..15) of P.V M-tile mt, per kernel's row order,
// and the skew of stashed row h.
//   kPairs: rows gid and gid+8 hold two adjacent channels (stored as float2);
//   the skews make a half-warp's float2 stores (or a warp's scalar stores)
//   cover the 32 banks once.
struct Vq2Dim {   // channel pair offset 4*gid
  static constexpr bool kPairs = true;
  __device__ int operator()(int mt, int r) const { return 4 * (8 * (mt >> 1) + (r & 7)) + 2 * (mt & 1) + (r >> 3); }
  __device__ static int skew(int h) { const int t = (h >> 1) & 3; return 2 * (t & 1) + 16 * (t >> 1); }
};
struct Vq4Dim {   // the two channels of subvector 8mt + r%8 (rows gid, gid+8); channel pair offset 2*gid
  static constexpr bool kPairs = true;
  __device__ int operator()(int mt, int r) const { return 2 * (8 * mt + (r & 7)) + (r >> 3); }
  __device__ static int skew(int h) { return 8 * ((h >> 1) & 3); }
};
struct Vq15Dim {   // channel pair offset 8*gid
  static constexpr bool kPairs = true;
  __device__ int operator()(int mt, int r) const { return 8 * (8 * (mt >> 2) + (r & 7)) + 2 * (mt & 3) + (r >> 3); }
  __device__ static int skew(int h) { return 2 * ((h >> 1) & 3); }
};
struct NaturalDim {   // channel offset gid, rows gid+8 eight channels on
  static constexpr bool kPairs = false;
  __device__ int operator()(int mt, int r) const { return 16 * mt + r; }
  __device__ static int skew(int h) { return 8 * ((h >> 1) & 3); }
};

}  // namespace
}  // namespace vqkv
