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

template <int WARPS>
struct CombineSmem {
  static constexpr int kO = WARPS * 8 * 128;     // floats
  static constexpr int kBytes = (kO + 2 * WARPS * 8) * 4;
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

// COLGROUPS: the launch may split the columns into groups (multi-query
// decode); otherwise the CTA holds all ncols columns.
template <int WARPS, bool COLGROUPS>
__device__ __forceinline__ void finish_sequence(const DecodeParams& p, int b, int kvh, int split,
                                                float* s_comb, int* s_last) {
  constexpr int NO = (8 * kHeadDim + WARPS * 32 - 1) / (WARPS * 32);   // outputs per thread in the merge
  const float* wO = s_comb;
  const float* wm = s_comb + CombineSmem<WARPS>::kO;
  const float* wl = wm + WARPS * 8;
  const int col0 = COLGROUPS ? cta_col0(p) : 0;
  const int G = COLGROUPS ? min(8, p.ncols - col0) : p.ncols;   // this CTA's columns
  float* part = p.partials + (((size_t)(b * p.Hkv + kvh) * p.n_splits + split) * p.ncols + col0) * kPartialStride;
  const unsigned ticket = COLGROUPS ? (unsigned)((b * p.Hkv + kvh) * p.cgroups + blockIdx.z % p.cgroups)
                                    : (unsigned)(b * p.Hkv + kvh);
  for (int e = threadIdx.x; e < G * kHeadDim; e += WARPS * 32) {
    const int h = e >> 7, d = e & 127;
    float M = kMInit;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, wm[w * 8 + h]);
    float o = 0.f, l = 0.f;
#pragma unroll 4
    for (int w = 0; w < WARPS; ++w) {
      const float f = fast_exp2(wm[w * 8 + h] - M);
      o += wO[(w * 8 + h) * kHeadDim + d] * f;
      l += wl[w * 8 + h] * f;
    }
    if (p.n_splits == 1) {
      p.out[out_row(p, b, kvh, col0 + h) + d] = __float2half_rn(l > 0.f ? o / l : 0.f);
      continue;
    }
    part[h * kPartialStride + d] = o;
    if (d == 0) {
      part[h * kPartialStride + 128] = M;
      part[h * kPartialStride + 129] = l;
    }
  }
  if (p.n_splits == 1 || p.defer_merge) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.tickets + ticket)
                 : "memory");
    *s_last = (prev == (unsigned)(p.n_splits - 1));
  }
  __syncthreads();
  if (*s_last) {
    // All split partials of (b, kvh) are staged in shared memory by the whole
    // CTA (coalesced, every load in flight at once), then each thread merges
    // one output (head, channel) with a running max.  Chunks of splits when
    // they do not all fit.
    const float* base = p.partials + ((size_t)(b * p.Hkv + kvh) * p.n_splits * p.ncols + col0) * kPartialStride;
    const int per_split = G * kPartialStride;                    // this CTA's columns of one split
    const size_t split_stride = (size_t)p.ncols * kPartialStride;
    const int chunk = max(1, min(p.n_splits, CombineSmem<WARPS>::kBytes / 4 / per_split));
    float M[NO], O[NO], Ls[NO];
    for (int k = 0; k < NO; ++k) M[k] = kMInit, O[k] = 0.f, Ls[k] = 0.f;
    for (int s0 = 0; s0 < p.n_splits; s0 += chunk) {
      const int ns = min(chunk, p.n_splits - s0);
      if (COLGROUPS) {
        for (int i = threadIdx.x; i < ns * per_split; i += WARPS * 32) {
          const int sp = i / per_split, r = i - sp * per_split;
          s_comb[i] = __ldcg(base + (size_t)(s0 + sp) * split_stride + r);
        }
      } else {   // all columns: the chunk is contiguous
        for (int i = threadIdx.x; i < ns * per_split; i += WARPS * 32) s_comb[i] = __ldcg(base + s0 * per_split + i);
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < NO; ++k) {
        const int e = threadIdx.x + k * WARPS * 32;
        if (e < G * kHeadDim) {
          const int h = e >> 7, d = e & 127;
          for (int s = 0; s < ns; ++s) {
            const float* ph = s_comb + s * per_split + h * kPartialStride;
            const float ms = ph[128];
            const float n = fmaxf(M[k], ms);
            const float fa = fast_exp2(M[k] - n), fb = fast_exp2(ms - n);
            O[k] = O[k] * fa + ph[d] * fb;
            Ls[k] = Ls[k] * fa + ph[129] * fb;
            M[k] = n;
          }
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < NO; ++k) {
      const int e = threadIdx.x + k * WARPS * 32;
      if (e < G * kHeadDim) {
        const int h = e >> 7, d = e & 127;
        p.out[out_row(p, b, kvh, col0 + h) + d] = __float2half_rn(Ls[k] > 0.f ? O[k] / Ls[k] : 0.f);
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
// acc[mt] = rows {gid, gid+8} (channels dim0(mt), dim0(mt)+1) x heads {2tig, 2tig+1}.
template <int WARPS, int NMT, typename DimOf>
__device__ __forceinline__ void stash_warp(float* s_comb, int warp, int lane, const float (&acc)[NMT][4],
                                           float m0, float m1, float l0, float l1, DimOf dim_of) {
  const int gid = lane >> 2, tig = lane & 3;
  float* wO = s_comb;
  float* wm = s_comb + CombineSmem<WARPS>::kO;
  float* wl = wm + WARPS * 8;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const int h0 = warp * 8 + 2 * tig;
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt) {
    const int d0 = dim_of(mt, gid), d1 = dim_of(mt, gid + 8);
    wO[h0 * kHeadDim + d0] = acc[mt][0];
    wO[(h0 + 1) * kHeadDim + d0] = acc[mt][1];
    wO[h0 * kHeadDim + d1] = acc[mt][2];
    wO[(h0 + 1) * kHeadDim + d1] = acc[mt][3];
  }
  if (gid == 0) {
    wm[h0] = m0;
    wm[h0 + 1] = m1;
    wl[h0] = l0;
    wl[h0 + 1] = l1;
  }
}

// Channel held by row r (0..15) of P.V M-tile mt, per kernel's row order.
struct Vq2Dim {
  __device__ int operator()(int mt, int r) const { return 4 * (8 * (mt >> 1) + (r & 7)) + 2 * (mt & 1) + (r >> 3); }
};
struct Vq15Dim {
  __device__ int operator()(int mt, int r) const { return 8 * (8 * (mt >> 2) + (r & 7)) + 2 * (mt & 3) + (r >> 3); }
};
struct NaturalDim {
  __device__ int operator()(int mt, int r) const { return 16 * mt + r; }
};

}  // namespace
}  // namespace vqkv
