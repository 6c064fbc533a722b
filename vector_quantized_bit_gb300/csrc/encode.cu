// VQ encode for sm_103a: smoothing, Hadamard rotation, nearest centroid, pack
// (VecInfer paper summary page, "Summary": channel-wise smoothing followed by
// a Hadamard rotation of the keys, K-Means codebook; arXiv summary page,
// "方法详解", stages 1-2).
//
// 1.25-, 2-, 3- and 4-bit: one warp per row (or one CTA per row when rows
// are few); lane l holds channels 4l..4l+3.  1.5-bit: tensor-core screening with an exact
// re-rank (below).  For keys the transform
// x' = (x / s) . H / sqrt(128) is carried in double-float arithmetic (pairs
// of fp32 with error-free sums and products) and rounded to fp32 once, so the
// vector handed to the nearest-centroid search is the correctly rounded fp32
// value of the exact transform.  Distances are fp32 direct differences; the
// argmin keeps the lowest index on equal distances.
#include <type_traits>

#include "common.cuh"
#include "encode_common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace vqkv {
namespace {

constexpr int ENC_WARPS = 8;
constexpr int ENC_THREADS = ENC_WARPS * 32;

// First byte of the tile holding token t of stream (b, kvh) (tiles of
// `tile_tokens` tokens, `tile_bytes` bytes), contiguous or through the block
// table; nullptr (and the error bit) for a block id outside the pool.
__device__ __forceinline__ uint8_t* tile_base(const EncodeParams& p, int b, int kvh, int t, int tile_tokens,
                                              int tile_bytes) {
  bool bad = false;
  const long long off = p.block_table ? tile_offset<true>(p, b, kvh, t / tile_tokens, tile_bytes, &bad)
                                      : tile_offset<false>(p, b, kvh, t / tile_tokens, tile_bytes, &bad);
  if (bad) {
    if (p.err) atomicOr(p.err, VQKV_DEVERR_BLOCK);
    return nullptr;
  }
  return p.codes + off;
}

// Smoothing factors of KV head kvh for keys, nullptr for values.
__device__ __forceinline__ const float* key_s(const EncodeParams& p, int kvh) {
  return p.role == VQKV_ROLE_K ? p.s + (size_t)kvh * kHeadDim : nullptr;
}

// ------------------------------------------------------------------ VQ2 / VQ4
// 256-entry codebooks, one byte per code.  DSUB = 4 (2 bit): lane l holds
// subvector l (channels 4l..4l+3); DSUB = 2 (4 bit): lane l holds
// subvectors 2l and 2l+1 (channels 4l, 4l+1 and 4l+2, 4l+3).
// SPLIT = 1: one warp per row, 256 candidates per lane (many 4-bit rows;
// many 2-bit rows go to the tensor-memory kernel below).
// SPLIT = 8: the CTA's 8 warps share one row, 32 candidates each (few rows,
// e.g. a decode-step append: latency instead of throughput).
template <int SPLIT, int DSUB>
__global__ void __launch_bounds__(ENC_THREADS) encode_vq2_kernel(const EncodeParams p) {
  using Centroid = typename std::conditional<DSUB == 4, float4, float2>::type;
  constexpr int kTileBytes = 16 * (kHeadDim / DSUB);
  __shared__ Centroid s_cb[256];
  __shared__ Best s_part[SPLIT > 1 ? ENC_WARPS * 32 : 1];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_dependents_launch();
  for (int c = threadIdx.x; c < 256; c += ENC_THREADS) {
    if constexpr (DSUB == 4) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.cb) + (size_t)kvh * 256 + c);
      const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
      const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
      s_cb[c] = make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
    } else {
      const __half2 a = __ldg(reinterpret_cast<const __half2*>(p.cb) + (size_t)kvh * 256 + c);
      s_cb[c] = make_float2(__low2float(a), __high2float(a));
    }
  }
  __syncthreads();
  const int rows = p.B * p.n_rows;
  const int r0 = (SPLIT == 1) ? blockIdx.x * ENC_WARPS + warp : blockIdx.x;
  const int rstep = (SPLIT == 1) ? gridDim.x * ENC_WARPS : gridDim.x;
  const int c_lo = (SPLIT == 1) ? 0 : warp * (256 / SPLIT);
  const int c_hi = c_lo + 256 / SPLIT;
  for (int r = r0; r < rows; r += rstep) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (lane == 0 && (SPLIT == 1 || warp == 0) && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    float x[4];
    transform_row(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim, key_s(p, kvh), lane, x);
    if constexpr (DSUB == 4) {   // lane = subvector j (channels 4j..4j+3)
      const Best part = vq2_search(x, c_lo, c_hi, [&](int c) { return s_cb[c]; });
      Best bst = merge_warps<SPLIT>(part, warp, lane, s_part);
      if (SPLIT == 1 || warp == 0) {
        count_near_ties(p.near_tie, is_near_tie(bst.d, bst.s), lane, 0xffffffffu);
        uint8_t* tb = tile_base(p, b, kvh, t, 16, kTileBytes);
        if (tb) tb[vq2_code_offset(p.role, t & 15, lane)] = (uint8_t)bst.i;
      }
    } else {   // lane = subvectors 2l, 2l+1
      Best pa, pb;
      vq4_search(x, c_lo, c_hi, [&](int c) { return s_cb[c]; }, pa, pb);
      Best ba = merge_warps<SPLIT>(pa, warp, lane, s_part);
      Best bb = merge_warps<SPLIT>(pb, warp, lane, s_part);
      if (SPLIT == 1 || warp == 0) {
        count_near_ties(p.near_tie, is_near_tie(ba.d, ba.s), lane, 0xffffffffu);
        count_near_ties(p.near_tie, is_near_tie(bb.d, bb.s), lane, 0xffffffffu);
        uint8_t* tb = tile_base(p, b, kvh, t, 16, kTileBytes);
        if (tb) {
          tb[vq4_code_offset(p.role, t & 15, 2 * lane)] = (uint8_t)ba.i;
          tb[vq4_code_offset(p.role, t & 15, 2 * lane + 1)] = (uint8_t)bb.i;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ VQ3
// 4096-entry codebooks of 4-channel subvectors, 12-bit codes in 3-byte
// pairs (j, j+16).  Lane l holds subvector l (channels 4l..4l+3) and scans
// the whole codebook (SPLIT = 1, 8 warps, one row per warp) or a slice of
// 4096 / SPLIT candidates (SPLIT = 16 warps sharing one row per CTA), with
// the fp32 codebook (or each warp's slice of it) in shared memory (64 KB,
// read by broadcast).  Lanes 0..15 then write pair l from their own code
// and lane l + 16's.  The library launches SPLIT = 16 for few rows (a
// decode step's append); many rows go to the tensor-memory kernel below.
constexpr size_t kEnc3Smem = 4096 * sizeof(float4);
constexpr int ENC3_SPLIT = 16;

// Search of one subvector over candidates [c_lo, c_hi) (a multiple of 4):
// fp32 direct differences, four chains over the candidates of each residue
// mod 4 (independent latency chains), merged by distance, then index.
template <typename Load>
__device__ __forceinline__ Best vq3_search(const float (&x)[4], int c_lo, int c_hi, Load load) {
  Best ch[4] = {best_init(), best_init(), best_init(), best_init()};
#pragma unroll 2
  for (int c = c_lo; c < c_hi; c += 4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 cv = load(c + k);
      float u = __fsub_rn(x[0], cv.x), d = __fmul_rn(u, u);
      u = __fsub_rn(x[1], cv.y); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[2], cv.z); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[3], cv.w); d = __fmaf_rn(u, u, d);
      best_push(ch[k], d, c + k);
    }
  }
  return best_merge(best_merge(ch[0], ch[1]), best_merge(ch[2], ch[3]));
}

template <int SPLIT>
__global__ void __launch_bounds__(SPLIT == 1 ? ENC_THREADS : SPLIT * 32) encode_vq3_kernel(const EncodeParams p) {
  constexpr int kThreads = SPLIT == 1 ? ENC_THREADS : SPLIT * 32;
  constexpr int kWarps = kThreads / 32;
  extern __shared__ __align__(16) unsigned char enc_smem[];
  float4* s_cb = reinterpret_cast<float4*>(enc_smem);
  __shared__ Best s_part[SPLIT > 1 ? SPLIT * 32 : 1];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c_lo = (SPLIT == 1) ? 0 : warp * (4096 / SPLIT);
  const int c_hi = c_lo + 4096 / SPLIT;
  grid_dependency_wait();
  grid_dependents_launch();
  {
    // the whole codebook (SPLIT = 1, by the CTA) or this warp's slice
    // (SPLIT > 1, by the warp): every load in flight before the first store
    constexpr int kPer = SPLIT == 1 ? 4096 / kThreads : 4096 / SPLIT / 32;
    const int first = SPLIT == 1 ? threadIdx.x : c_lo + lane;
    const int stride = SPLIT == 1 ? kThreads : 32;
    const uint2* g = reinterpret_cast<const uint2*>(p.cb) + (size_t)kvh * 4096 + first;
    uint2 raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) raw[i] = __ldg(g + i * stride);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const __half2 a = *reinterpret_cast<const __half2*>(&raw[i].x);
      const __half2 b = *reinterpret_cast<const __half2*>(&raw[i].y);
      s_cb[first + i * stride] = make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
    }
  }
  if (SPLIT == 1)
    __syncthreads();
  else
    __syncwarp();
  const int rows = p.B * p.n_rows;
  const int r0 = (SPLIT == 1) ? blockIdx.x * kWarps + warp : blockIdx.x;
  const int rstep = (SPLIT == 1) ? gridDim.x * kWarps : gridDim.x;
  for (int r = r0; r < rows; r += rstep) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (lane == 0 && (SPLIT == 1 || warp == 0) && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    float x[4];
    transform_row(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim, key_s(p, kvh), lane, x);
    const Best part = vq3_search(x, c_lo, c_hi, [&](int c) { return s_cb[c]; });
    const Best bst = merge_warps<SPLIT>(part, warp, lane, s_part);
    if (SPLIT == 1 || warp == 0) {
      count_near_ties(p.near_tie, is_near_tie(bst.d, bst.s), lane, 0xffffffffu);
      const int hi = __shfl_down_sync(0xffffffffu, bst.i, 16);
      uint8_t* tb = tile_base(p, b, kvh, t, 16, 768);
      if (tb && lane < 16) {
        tb[vq3_byte_offset(p.role, t & 15, lane, 0)] = (uint8_t)(bst.i & 0xff);
        tb[vq3_byte_offset(p.role, t & 15, lane, 1)] = (uint8_t)(((bst.i >> 8) & 0xf) | ((hi & 0xf) << 4));
        tb[vq3_byte_offset(p.role, t & 15, lane, 2)] = (uint8_t)(hi >> 4);
      }
    }
  }
}

// ------------------------------------------------------------------ VQ125
// 1024-entry codebooks of 8-channel subvectors, 10-bit codes.  Lane l
// searches subvector l % 16 (channels 8j..8j+7, taken from lanes 2j and
// 2j+1) over half l / 16 of its warp's candidates (the whole codebook for
// SPLIT = 1, 1024 / SPLIT per warp otherwise); the halves merge across
// lanes l and l + 16.  Lanes 0..3 then pack the row's four 40-bit groups
// (K: subvectors g, g+4, g+8, g+12; V: 2g, 2g+1, 2g+8, 2g+9) and write 5
// bytes each.  The library launches SPLIT = 8 for few rows (a decode step's
// append); many rows go to the tensor-memory kernel below.

// Search of one 8-channel subvector over candidates [c_lo, c_hi) (a multiple
// of 4): fp32 direct differences in channel order, four chains over the
// candidates of each residue mod 4, merged by distance, then index.
// s_cb: centroid c as two float4 at 2c (channels 0..3) and 2c+1 (4..7).
__device__ __forceinline__ Best vq125_search(const float (&x)[8], int c_lo, int c_hi, const float4* s_cb) {
  Best ch[4] = {best_init(), best_init(), best_init(), best_init()};
#pragma unroll 2
  for (int c = c_lo; c < c_hi; c += 4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 a = s_cb[2 * (c + k)], b = s_cb[2 * (c + k) + 1];
      float u = __fsub_rn(x[0], a.x), d = __fmul_rn(u, u);
      u = __fsub_rn(x[1], a.y); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[2], a.z); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[3], a.w); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[4], b.x); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[5], b.y); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[6], b.z); d = __fmaf_rn(u, u, d);
      u = __fsub_rn(x[7], b.w); d = __fmaf_rn(u, u, d);
      best_push(ch[k], d, c + k);
    }
  }
  return best_merge(best_merge(ch[0], ch[1]), best_merge(ch[2], ch[3]));
}

template <int SPLIT>
__global__ void __launch_bounds__(ENC_THREADS) encode_vq125_kernel(const EncodeParams p) {
  __shared__ float4 s_cb[2 * 1024];
  __shared__ Best s_part[SPLIT > 1 ? ENC_WARPS * 32 : 1];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kSpan = 1024 / SPLIT;   // candidates of one warp
  const int c_lo = (SPLIT == 1 ? 0 : warp * kSpan) + (lane >> 4) * (kSpan / 2);
  const int c_hi = c_lo + kSpan / 2;
  grid_dependency_wait();
  grid_dependents_launch();
  {
    // every codebook load in flight before the first store
    constexpr int kPer = 1024 / ENC_THREADS;
    const uint4* g = reinterpret_cast<const uint4*>(p.cb) + (size_t)kvh * 1024 + threadIdx.x;
    uint4 raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) raw[i] = __ldg(g + i * ENC_THREADS);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = threadIdx.x + i * ENC_THREADS;
      const __half2* h = reinterpret_cast<const __half2*>(&raw[i]);
      s_cb[2 * c] = make_float4(__low2float(h[0]), __high2float(h[0]), __low2float(h[1]), __high2float(h[1]));
      s_cb[2 * c + 1] = make_float4(__low2float(h[2]), __high2float(h[2]), __low2float(h[3]), __high2float(h[3]));
    }
  }
  __syncthreads();
  const bool key = p.role == VQKV_ROLE_K;
  const int rows = p.B * p.n_rows;
  const int r0 = (SPLIT == 1) ? blockIdx.x * ENC_WARPS + warp : blockIdx.x;
  const int rstep = (SPLIT == 1) ? gridDim.x * ENC_WARPS : gridDim.x;
  for (int r = r0; r < rows; r += rstep) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (lane == 0 && (SPLIT == 1 || warp == 0) && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    float x[4];
    transform_row(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim, key_s(p, kvh), lane, x);
    const int j = lane & 15;
    float xs[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      xs[k] = __shfl_sync(0xffffffffu, x[k], 2 * j);
      xs[4 + k] = __shfl_sync(0xffffffffu, x[k], 2 * j + 1);
    }
    Best part = vq125_search(xs, c_lo, c_hi, s_cb);
    part = best_merge(part, best_shfl_xor(part, 16));
    const Best bst = merge_warps<SPLIT>(part, warp, lane, s_part);
    if (SPLIT == 1 || warp == 0) {
      count_near_ties(p.near_tie, is_near_tie(bst.d, bst.s), lane, 0xffffu);
      const int g = lane & 3;
      const uint32_t c0 = __shfl_sync(0xffffffffu, bst.i, key ? g : 2 * g);
      const uint32_t c1 = __shfl_sync(0xffffffffu, bst.i, key ? g + 4 : 2 * g + 1);
      const uint32_t c2 = __shfl_sync(0xffffffffu, bst.i, key ? g + 8 : 2 * g + 8);
      const uint32_t c3 = __shfl_sync(0xffffffffu, bst.i, key ? g + 12 : 2 * g + 9);
      const unsigned long long grp =
          (unsigned long long)(c0 | (c1 << 10) | (c2 << 20)) | ((unsigned long long)c3 << 30);
      uint8_t* tb = tile_base(p, b, kvh, t, 16, 320);
      if (tb && lane < 4) {
        const int rr = t & 15;
        const int run = key ? 4 * (rr & 7) + g : 4 * g + ((rr & 7) >> 1);
        const int n0 = key ? 5 * (rr >> 3) : 5 * (2 * (rr >> 3) + (rr & 1));
#pragma unroll
        for (int q = 0; q < 5; ++q) tb[vq125_run_byte(p.role, run, n0 + q)] = (uint8_t)(grp >> (8 * q));
      }
    }
  }
}

// ------------------------------------------------------------------ VQ15, tensor-core screening
// Many rows of 1.5-bit encode: the distance search against 4096 centroids is
// a dense contraction, run as one augmented mma.m16n8k16 per 8 centroids:
//   A[j] = [x_hi (8 ch), 1, 1, 0...] and [x_lo (8 ch), 0...]  (16 subvectors
//          of a row; x' = x_hi + x_lo in fp16 to ~2^-22)
//   B[c] = [-2 c (8 ch), |c|^2_hi, |c|^2_lo, 0...]
//   D[j][c] = |c|^2 - 2 x'_j.c  (two MMAs; the squared distance less the
//          per-subvector constant |x'_j|^2, which does not change a ranking)
// Each lane keeps the best and second-best screened distance of its
// centroid columns.  A centroid whose screened distance is within 2*eps of
// the best can be the exact nearest, where eps bounds the screening error
// (screen_eps); those candidates are
// re-ranked with exact fp32 direct differences (channel order 0..7, one
// rounding per operation), so every decision equals the exhaustive fp32
// search's.  If a lane's second-best is also
// within the margin (a third candidate may hide behind it) the subvector is
// searched exhaustively.
constexpr int TC_WARPS = 16;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int TC_TABLE_BYTES = 4096 * 4 * 8;                 // [centroid][tig]{b0b1, b2b3}

// fp16 hi and lo parts of two fp32 values: a ~= hi.x + lo.x to about 2^-22
// relative (lo may be subnormal: then to about 6e-8 absolute).
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const __half2 l = __floats2half2_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Bound on |screened - exact| for one candidate of a subvector with norm
// xnorm, centroid norms <= cmax: the hi/lo splits of x and |c|^2 leave
// ~2^-22 relative (plus fp16 subnormal steps), and the tensor-core fp32
// accumulation and the exact search's own fp32 roundings stay well inside
// 1.5e-5 (|x| + cmax)^2.
__device__ __forceinline__ float screen_eps(float xnorm, float cmax) {
  const float sc = xnorm + cmax;
  return 9.5367431640625e-7f * xnorm * cmax + 4.76837158203125e-7f * cmax * cmax + 1e-6f * (cmax + 1.f) +
         1.5e-5f * sc * sc;
}

__device__ __forceinline__ void top2_push(float v, int n, float& b1, float& b2, int& i1) {
  const bool lt = v < b1;
  b2 = fminf(b2, fmaxf(b1, v));
  b1 = fminf(b1, v);
  i1 = lt ? n : i1;
}

// Exact fp32 distance of subvector x (8 channels) to centroid c: direct
// differences in channel order, one rounding per operation.
__device__ __forceinline__ float exact_d8(const float* x, const uint2* tbl, int c) {
  float y[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {   // -2c pairs of tig t
    const __half2 h = *reinterpret_cast<const __half2*>(&tbl[c * 4 + t].x);
    y[2 * t] = -0.5f * __low2float(h);
    y[2 * t + 1] = -0.5f * __high2float(h);
  }
  float e = __fsub_rn(x[0], y[0]);
  float d = __fmul_rn(e, e);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    e = __fsub_rn(x[i], y[i]);
    d = __fmaf_rn(e, e, d);
  }
  return d;
}

// The same distance to centroid c read from the fp16 codebook in global
// memory (cb8: its 8 channels).  x_i - c_i is the same correctly rounded
// difference as above, so the two agree bit for bit.
__device__ __forceinline__ float exact_d8_cb(const float* x, const __half* cb8) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(cb8));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float y[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
    y[2 * t] = f.x;
    y[2 * t + 1] = f.y;
  }
  float e = __fsub_rn(x[0], y[0]);
  float d = __fmul_rn(e, e);
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    e = __fsub_rn(x[i], y[i]);
    d = __fmaf_rn(e, e, d);
  }
  return d;
}

// The same for 4 channels (2-bit codebooks).
__device__ __forceinline__ float exact_d4_cb(const float* x, const __half* cb4) {
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(cb4));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  float e = __fsub_rn(x[0], a.x);
  float d = __fmul_rn(e, e);
  e = __fsub_rn(x[1], a.y);
  d = __fmaf_rn(e, e, d);
  e = __fsub_rn(x[2], b.x);
  d = __fmaf_rn(e, e, d);
  e = __fsub_rn(x[3], b.y);
  return __fmaf_rn(e, e, d);
}

// Largest centroid norm the fp16 screening tables hold exactly: -2c stays
// exact and |c|^2 <= 16384 keeps its fp16 hi + lo split finite.  A KV head
// with a larger centroid is searched exhaustively, from the codebook in
// global memory (slow, but only such codebooks pay for it).
constexpr float kScreenCmax = 128.f;

// B table [centroid][tig]{-2c pair, (|c|^2, 1) or 0} of KV head kvh in
// shared memory, and the largest centroid norm (returned; s_cmax is one
// float of scratch).  Called by every thread of the CTA.
__device__ __forceinline__ float build_tc_table(const EncodeParams& p, int kvh, uint2* s_tbl, float* s_cmax) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = 4096 / TC_THREADS;
  uint4 raws[kPer];   // every load in flight before the first use
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    raws[k] = __ldg(reinterpret_cast<const uint4*>(p.cb) + (size_t)kvh * 4096 + threadIdx.x + k * TC_THREADS);
  float cmax = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int c = threadIdx.x + k * TC_THREADS;
    const uint32_t w[4] = {raws[k].x, raws[k].y, raws[k].z, raws[k].w};
    float nn = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[t]);
      const float a = __low2float(h), b = __high2float(h);
      nn = __fmaf_rn(a, a, nn);
      nn = __fmaf_rn(b, b, nn);
      const __half2 m2 = __floats2half2_rn(-2.f * a, -2.f * b);   // exact
      s_tbl[c * 4 + t].x = *reinterpret_cast<const uint32_t*>(&m2);
    }
    const __half nh = __float2half_rn(nn);   // |c|^2 as fp16 hi + lo
    const __half2 tail = __halves2half2(nh, __float2half_rn(nn - __half2float(nh)));
    s_tbl[c * 4 + 0].y = *reinterpret_cast<const uint32_t*>(&tail);
    s_tbl[c * 4 + 1].y = s_tbl[c * 4 + 2].y = s_tbl[c * 4 + 3].y = 0u;
    cmax = fmaxf(cmax, sqrtf(nn));
  }
  for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  if (threadIdx.x == 0) *s_cmax = 0.f;
  __syncthreads();
  if (lane == 0) atomicMax(reinterpret_cast<int*>(s_cmax), __float_as_int(cmax));   // non-negative floats
  __syncthreads();
  return *s_cmax;
}

// Many rows of 1.5-bit or 2-bit encode on the fifth-generation tensor cores.
// A tile is 128 (row, subvector) pairs, the M of one tcgen05 MMA: 8 rows of
// 16 subvectors (1.5 bit) or 4 rows of 32 (2 bit); the 4096 (256) centroids
// are 32 (2) chunks of N = 128.  One MMA per chunk writes to tensor memory
//   D[m][c] = [x_hi, 1, 1] . [-2c, |c|^2_hi, |c|^2_lo] = |c|^2 - 2 x_hi . c,
// the screened distance less the subvector's own |x'_j|^2, with x_hi the fp16
// rounding of the transformed subvector (A) and the [-2c, |c|^2_hi, |c|^2_lo]
// table of all the KV head's centroids (B) in shared memory behind matrix
// descriptors.  Its error is bounded by screen_eps_hi.  (A second MMA with
// the fp16 remainder of x' would tighten the bound but doubles the shared
// memory and tensor memory traffic, which bound this kernel.)
//
// Roles (12 warps, one CTA per SM, persistent over the KV head's tiles; 12
// warps leave each SM sub-partition 3 warps, so up to 168 registers a thread,
// enough for a whole 128-column chunk in flight per epilogue thread):
//   warps 8, 9   producers: transform rows pw, pw + 2, ... of each tile
//                (smoothing + Hadamard in double-float for keys), write
//                A, x' and |x'_j|^2 into one of 4 stages;
//   warps 10, 11 one thread each issues the MMAs of one epilogue warpgroup,
//                chunk by chunk into that warpgroup's two 128-column
//                tensor-memory buffers (warp 10 also allocates the 512
//                columns); separate issuers keep one warpgroup's wait for a
//                free buffer from holding up the other's MMAs;
//   warps 0-3, 4-7  two epilogue warpgroups taking alternate tiles: thread m
//                owns tensor-memory lane m, i.e. subvector m % S of row m / S
//                (S = 16 or 32 subvectors a row).
// The epilogue does not rank candidates one by one: per group of 32
// consecutive centroids it takes the group minimum, which the tensor-memory
// load computes itself (tcgen05.ld.red ... .min, one load per group), and
// keeps the four smallest group minima B1 <= B2 <= B3 <= B4, each carrying
// its group id.  A centroid can be the exact nearest only if its screened
// distance is within 2 eps of B1, so with B4 above that margin every
// candidate lies in G1, G2 or G3 (the latter two only when B2, B3 are within
// the margin): those groups are re-ranked with exact fp32 direct differences
// (as exact_d8), the lowest index winning ties; G1 by each lane, the rarer
// G2 / G3 by the whole warp, one lane's group at a time.  With B4 inside the
// margin, or a row whose transformed values do not fit fp16, the warp
// searches that subvector exhaustively.  Every decision therefore equals
// the exhaustive fp32 search's.
//
// Every wait is bounded: a wait that runs out sets VQKV_DEVERR_TIMEOUT (when
// the caller passed an error word) and an abort flag that ends every role's
// loop; the MMA thread then waits (bounded) for its MMAs before the tensor
// memory is freed.
namespace um {
constexpr int M = 128;                        // MMA rows: (row, subvector) pairs of a tile
constexpr int N = 128;                        // centroids per MMA
constexpr int NBUF = 2;                       // tensor-memory buffers per epilogue warpgroup
constexpr int GROUP = 32;                     // centroids per group minimum
constexpr int STAGES = 4;
constexpr int PROD_WARPS = 2;
constexpr int MMA_WARP = 8 + PROD_WARPS;      // 10 (warpgroup 0's issuer; 11: warpgroup 1's)
constexpr int THREADS = (MMA_WARP + 2) * 32;  // 384
constexpr int A_BYTES = M * 32;               // one A tile: 128 x 16 fp16
constexpr int NBAR = 2 * STAGES + 4 * NBUF + 2;   // A full / empty, tensor-memory full / empty, MMAs done x 2
constexpr uint32_t TMEM_COLS = 512;           // 2 warpgroups x NBUF buffers x N
static_assert(2 * NBUF * N <= (int)TMEM_COLS && N % GROUP == 0, "tensor-memory plan");
constexpr uint32_t MAX_POLLS = 1u << 22;
// row flags
constexpr int F_OK = 0, F_EXHAUSTIVE = 1, F_SKIP = 2;
}  // namespace um

// Per code mode: 8-channel subvectors (1.5 bit: 4096 centroids; 1.25 bit:
// 1024), 16 a row, 8 rows a tile; or 4-channel ones (2 bit: 256 centroids;
// 3 bit: 4096), 32 a row, 4 rows a tile.
template <int MODE>
struct UmGeo {
  static constexpr int DSUB = (MODE == VQKV_MODE_VQ15 || MODE == VQKV_MODE_VQ125) ? 8 : 4;
  static constexpr int E = MODE == VQKV_MODE_VQ2 ? 256 : MODE == VQKV_MODE_VQ125 ? 1024 : 4096;
  static constexpr int SUBV = kHeadDim / DSUB;           // subvectors per row
  static constexpr int ROWS = um::M / SUBV;               // rows per tile
  static constexpr int CHUNKS = E / um::N;               // MMAs per tile
  static constexpr int TABLE_BYTES = E * 32;             // B: E centroids x 16 fp16
  static constexpr int ST_A = 0, ST_X = um::A_BYTES;
  static constexpr int ST_NORM = ST_X + ROWS * kHeadDim * 4, ST_FLAG = ST_NORM + um::M * 4;
  static constexpr int ST_POS = ST_FLAG + um::M * 4;
  static constexpr int STAGE_BYTES = ST_POS + 16 * 4;   // + cache position of each row
  static constexpr int OFF_STAGES = TABLE_BYTES;
  static constexpr int OFF_BAR = OFF_STAGES + um::STAGES * STAGE_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + um::NBAR * 8;   // tensor-memory base, abort flag, max centroid norm
  // 4-channel modes: the codebook again as plain fp16 [E][4], 8 bytes a
  // centroid, so that 16 lanes reading 16 consecutive centroids hit 16
  // distinct bank pairs in the exact re-rank (the B table's 32-byte rows give
  // only 8)
  static constexpr int OFF_CB4 = OFF_MISC + 16;
  static constexpr size_t SMEM = OFF_CB4 + (DSUB == 4 ? E * 8 : 0);
  static_assert(SMEM <= 227 * 1024 && STAGE_BYTES % 16 == 0 && OFF_BAR % 8 == 0, "UMMA encode shared memory");
  static_assert(CHUNKS % um::NBUF == 0 && E / um::GROUP <= 128 && ROWS <= 16, "tile plan (7-bit group ids)");
};

// Bound on |screened - exact| for one candidate of the single-MMA screen:
// the fp16 rounding of x' leaves |x' - x_hi| <= 2^-11 |x'| per channel
// (normal range; subnormal steps are covered by the absolute term), so
// |2 (x' - x_hi) . c| <= 2^-10 |x'| |c|; the |c|^2 split, the tensor-core
// fp32 accumulation and the exact search's own roundings are covered as in
// screen_eps.
__device__ __forceinline__ float screen_eps_hi(float xnorm, float cmax) {
  const float sc = xnorm + cmax;
  return 9.765625e-4f * xnorm * cmax + 4.76837158203125e-7f * cmax * cmax + 1e-6f * (cmax + 1.f) +
         1.5e-5f * sc * sc;
}

// Bounded wait on an mbarrier phase by every lane of a warp (or one thread:
// pass a one-lane mask): false, with the abort flag set, when it runs out
// or another role aborted.
__device__ __forceinline__ bool um_wait(uint32_t mbar, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                        unsigned mask) {
  bool ok = false;
  for (uint32_t i = 0; i < um::MAX_POLLS; ++i) {
    if (mbar_try_wait(mbar, parity)) {
      ok = true;
      break;
    }
    if ((i & 31) == 31 && *abort_flag) break;
  }
  ok = __all_sync(mask, ok);
  if (!ok && !*abort_flag) {
    *abort_flag = 1;
    if (err) atomicOr(err, VQKV_DEVERR_TIMEOUT);
  }
  return ok;
}

// Exact fp32 distance of subvector x (D = 8 or 4 channels) to centroid c
// read from the B table (-2c as fp16, halved exactly): direct differences in
// channel order, one rounding per operation, the same arithmetic as
// exact_d8 and vq2_search.
// x_i - c_i is formed as fma(0.5, h_i, x_i) with h_i = -2 c_i: 0.5 h_i = -c_i
// exactly, so it is the same correctly rounded difference.
template <int D>
__device__ __forceinline__ float exact_d_umma(const float (&x)[D], const unsigned char* table, int c) {
  uint32_t w[D / 2];
  if constexpr (D == 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(table + umma_kmajor_offset((uint32_t)c, 0));
    w[0] = raw.x, w[1] = raw.y, w[2] = raw.z, w[3] = raw.w;
  } else {
    const uint2 raw = *reinterpret_cast<const uint2*>(table + umma_kmajor_offset((uint32_t)c, 0));
    w[0] = raw.x, w[1] = raw.y;
  }
  float h[D];
#pragma unroll
  for (int t = 0; t < D / 2; ++t) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
    h[2 * t] = f.x;
    h[2 * t + 1] = f.y;
  }
  float e = __fmaf_rn(0.5f, h[0], x[0]);
  float d = __fmul_rn(e, e);
#pragma unroll
  for (int i = 1; i < D; ++i) {
    e = __fmaf_rn(0.5f, h[i], x[i]);
    d = __fmaf_rn(e, e, d);
  }
  return d;
}

// Exact search state: best distance and index, second-best distance.
// Candidates may come in any index order: lower distance, then lower index.
__device__ __forceinline__ void exact_push(float d, int c, float& dex, int& cex, float& dsec) {
  if (d < dex || (d == dex && c < cex)) {
    dsec = dex;
    dex = d;
    cex = c;
  } else {
    dsec = fminf(dsec, d);
  }
}

// Merges another disjoint candidate set's (best, index, second) into a state.
__device__ __forceinline__ void exact_merge(float od, int oc, float os, float& dex, int& cex, float& dsec) {
  if (od < dex || (od == dex && oc < cex)) {
    dsec = fminf(dex, os);
    dex = od;
    cex = oc;
  } else {
    dsec = fminf(dsec, od);
  }
}

// The warp's combined (best, index, second) over the lanes' states, in every lane.
__device__ __forceinline__ void exact_warp_reduce(float& d, int& c, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float od = __shfl_xor_sync(0xffffffffu, d, o), os = __shfl_xor_sync(0xffffffffu, s, o);
    const int oc = __shfl_xor_sync(0xffffffffu, c, o);
    exact_merge(od, oc, os, d, c, s);
  }
}

template <int MODE>
__global__ void __launch_bounds__(um::THREADS, 1) encode_umma_kernel(const EncodeParams p) {
  using namespace um;
  using Geo = UmGeo<MODE>;
  constexpr int DSUB = Geo::DSUB, E = Geo::E, SUBV = Geo::SUBV, ROWS = Geo::ROWS, CHUNKS = Geo::CHUNKS;
  constexpr int ST_A = Geo::ST_A, ST_X = Geo::ST_X, ST_NORM = Geo::ST_NORM, ST_FLAG = Geo::ST_FLAG;
  constexpr int ST_POS = Geo::ST_POS, STAGE_BYTES = Geo::STAGE_BYTES, OFF_STAGES = Geo::OFF_STAGES;
  constexpr int OFF_BAR = Geo::OFF_BAR, OFF_MISC = Geo::OFF_MISC;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + OFF_BAR;
  auto a_full = [&](int s) { return bar + 8u * s; };
  auto a_empty = [&](int s) { return bar + 8u * (STAGES + s); };
  auto t_full = [&](int wg, int b) { return bar + 8u * (2 * STAGES + NBUF * wg + b); };
  auto t_empty = [&](int wg, int b) { return bar + 8u * (2 * STAGES + 2 * NBUF + NBUF * wg + b); };
  auto done_bar = [&](int wg) { return bar + 8u * (2 * STAGES + 4 * NBUF + wg); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  float* s_cmax = reinterpret_cast<float*>(smem + OFF_MISC + 8);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(a_full(s), PROD_WARPS);
      mbar_init(a_empty(s), 4);
    }
    for (int wg = 0; wg < 2; ++wg)
      for (int b = 0; b < NBUF; ++b) {
        mbar_init(t_full(wg, b), 1);
        mbar_init(t_empty(wg, b), 4);
      }
    mbar_init(done_bar(0), 1);
    mbar_init(done_bar(1), 1);
    *s_abort = 0;
    *s_cmax = 0.f;
    mbar_init_fence();
  }
  if (warp == MMA_WARP) tmem_alloc(smem_u32(s_tmem), TMEM_COLS);
  grid_dependency_wait();
  grid_dependents_launch();
  __syncthreads();

  // B table: row c = [-2c (8 fp16), |c|^2 hi, |c|^2 lo, 0 x 6] (1.5 bit) or
  // [-2c (4 fp16), |c|^2 hi, |c|^2 lo, 0 x 10] (2 bit)
  {
    float cmax = 0.f;
    for (int c = threadIdx.x; c < E; c += THREADS) {
      uint32_t w[DSUB / 2];
      if constexpr (DSUB == 8) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.cb) + (size_t)kvh * E + c);
        w[0] = raw.x, w[1] = raw.y, w[2] = raw.z, w[3] = raw.w;
      } else {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.cb) + (size_t)kvh * E + c);
        w[0] = raw.x, w[1] = raw.y;
      }
      uint32_t m2[DSUB / 2];
      float nn = 0.f;
#pragma unroll
      for (int t = 0; t < DSUB / 2; ++t) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[t]);
        const float a = __low2float(h), b = __high2float(h);
        nn = __fmaf_rn(a, a, nn);
        nn = __fmaf_rn(b, b, nn);
        const __half2 mm = __floats2half2_rn(-2.f * a, -2.f * b);   // exact
        m2[t] = *reinterpret_cast<const uint32_t*>(&mm);
      }
      const __half nh = __float2half_rn(nn);
      const __half2 tail = __halves2half2(nh, __float2half_rn(nn - __half2float(nh)));
      const uint32_t tw = *reinterpret_cast<const uint32_t*>(&tail);
      unsigned char* row = smem + umma_kmajor_offset((uint32_t)c, 0);
      if constexpr (DSUB == 8) {
        *reinterpret_cast<uint4*>(row) = make_uint4(m2[0], m2[1], m2[2], m2[3]);
        *reinterpret_cast<uint4*>(row + 128) = make_uint4(tw, 0u, 0u, 0u);
      } else {
        *reinterpret_cast<uint4*>(row) = make_uint4(m2[0], m2[1], tw, 0u);
        *reinterpret_cast<uint4*>(row + 128) = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint2*>(smem + Geo::OFF_CB4)[c] = make_uint2(w[0], w[1]);
      }
      cmax = fmaxf(cmax, sqrtf(nn));
    }
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    if (lane == 0) atomicMax(reinterpret_cast<int*>(s_cmax), __float_as_int(cmax));   // non-negative floats
    fence_proxy_async_smem();
  }
  tcgen05_before_sync();
  __syncthreads();
  tcgen05_after_sync();
  const uint32_t tmem = *s_tmem;
  const float Cmax = *s_cmax;

  const int rows = p.B * p.n_rows;
  const int tiles = (rows + ROWS - 1) / ROWS;
  const int n_my = (int)blockIdx.x < tiles ? (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  if (warp >= 8 && warp < MMA_WARP) {
    // ---------------- producers: rows pw, pw + 3, pw + 6 (< 8) of every tile.
    // The raw rows of tile k + 1 are loaded while tile k is transformed.
    const int pw = warp - 8;
    // 1.5 bit: lanes 2j, 2j + 1 hold subvector j; 2 bit: lane j holds subvector j
    const int j = DSUB == 8 ? lane >> 1 : lane, half = DSUB == 8 ? lane & 1 : 0;
    constexpr int PR = (ROWS + PROD_WARPS - 1) / PROD_WARPS;   // rows per producer warp (4 / 2)
    const bool key = p.role == VQKV_ROLE_K;
    const float4 s4 = key ? *reinterpret_cast<const float4*>(p.s + (size_t)kvh * kHeadDim + 4 * lane)
                          : make_float4(1.f, 1.f, 1.f, 1.f);
    const float4 rs4 = make_float4(__frcp_rn(s4.x), __frcp_rn(s4.y), __frcp_rn(s4.z), __frcp_rn(s4.w));
    uint2 raw[PR];
    int pos_t[PR];   // cache position of the row, or -1 (no row / out of range)
    auto fetch = [&](int k) {
      const int gt = (int)blockIdx.x + k * (int)gridDim.x;
#pragma unroll
      for (int i = 0; i < PR; ++i) {
        const int r = pw + PROD_WARPS * i, row = gt * ROWS + r;
        pos_t[i] = -1;
        raw[i] = make_uint2(0u, 0u);
        if (r < ROWS && row < rows) {
          const int b = row / p.n_rows, n = row - b * p.n_rows;
          const int t = p.pos[b] + n;
          if (t < 0 || t >= p.cap_len) {
            if (lane == 0 && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
          } else {
            pos_t[i] = t;
            raw[i] = *reinterpret_cast<const uint2*>(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim +
                                                     4 * lane);
          }
        }
      }
    };
    if (n_my > 0) fetch(0);
    for (int k = 0; k < n_my; ++k) {
      uint2 cur[PR];
      int cur_t[PR];
#pragma unroll
      for (int i = 0; i < PR; ++i) cur[i] = raw[i], cur_t[i] = pos_t[i];
      if (k + 1 < n_my) fetch(k + 1);
      const int s = k % STAGES;
      if (!um_wait(a_empty(s), ((k / STAGES) & 1) ^ 1, s_abort, p.err, 0xffffffffu)) break;
      unsigned char* st = smem + OFF_STAGES + s * STAGE_BYTES;
#pragma unroll
      for (int i = 0; i < PR; ++i) {
        const int r = pw + PROD_WARPS * i;
        if (r >= ROWS) break;
        const int m = SUBV * r + j;
        int flag = F_SKIP;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (cur_t[i] >= 0) {
          if (key)
            transform_key_lean(cur[i], s4, rs4, lane, x);
          else
            transform_loaded(cur[i], false, s4, lane, x);
          // beyond fp16 screening (or not finite), or a codebook beyond the table: exhaustive
          flag = Cmax <= kScreenCmax ? F_OK : F_EXHAUSTIVE;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!(fabsf(x[e]) < 32768.f)) flag = F_EXHAUSTIVE;
        }
        if constexpr (DSUB == 8) {
          const uint32_t off = umma_kmajor_offset((uint32_t)m, 4u * half);
          *reinterpret_cast<uint2*>(st + ST_A + off) = make_uint2(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]));
          *reinterpret_cast<uint2*>(st + ST_A + off + 128) =
              make_uint2(half == 0 ? pack_half2(1.f, 1.f) : 0u, 0u);   // picks |c|^2 hi + lo
        } else {
          const uint32_t off = umma_kmajor_offset((uint32_t)m, 0u);
          *reinterpret_cast<uint4*>(st + ST_A + off) =
              make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(1.f, 1.f), 0u);
          *reinterpret_cast<uint4*>(st + ST_A + off + 128) = make_uint4(0u, 0u, 0u, 0u);
        }
        *reinterpret_cast<float4*>(st + ST_X + (r * kHeadDim + 4 * lane) * 4) = make_float4(x[0], x[1], x[2], x[3]);
        float nx = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
        if constexpr (DSUB == 8) {
          nx += __shfl_xor_sync(0xffffffffu, nx, 1);   // |x'_j|^2
          flag = max(flag, __shfl_xor_sync(0xffffffffu, flag, 1));
        }
        if (half == 0) {
          reinterpret_cast<float*>(st + ST_NORM)[m] = nx;
          reinterpret_cast<int*>(st + ST_FLAG)[m] = flag;
        }
        if (lane == 0) reinterpret_cast<int*>(st + ST_POS)[r] = cur_t[i];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full(s));
    }
  } else if (warp >= MMA_WARP) {
    // ---------------- one thread per epilogue warpgroup issues its MMAs
    const int wg = warp - MMA_WARP;
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16_f32(M, N);
      bool ok = true;
      int it = 0;
      for (int k = wg; ok && k < n_my; k += 2, ++it) {
        const int s = k % STAGES;
        ok = um_wait(a_full(s), (k / STAGES) & 1, s_abort, p.err, 1u);
        const uint64_t dA = umma_desc_kmajor(sbase + OFF_STAGES + s * STAGE_BYTES + ST_A);
        tcgen05_after_sync();
        for (int q = 0; ok && q < CHUNKS; ++q) {
          const int bsel = q % NBUF;
          const uint32_t use = (uint32_t)(it * (CHUNKS / NBUF) + q / NBUF);
          ok = um_wait(t_empty(wg, bsel), (use & 1) ^ 1, s_abort, p.err, 1u);
          if (!ok) break;
          tcgen05_after_sync();
          umma_f16(tmem + (uint32_t)((NBUF * wg + bsel) * N), dA, umma_desc_kmajor(sbase + (uint32_t)q * (N * 32)),
                   idesc, 0u);
          umma_commit(t_full(wg, bsel));
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      umma_commit(done_bar(wg));
      um_wait(done_bar(wg), 0, s_abort, p.err, 1u);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warpgroup wg: tiles wg, wg + 2, ...
    const int wg = warp >> 2, ml = 32 * (warp & 3) + lane;   // tensor-memory lane = MMA row
    const int r = ml / SUBV, j = ml % SUBV;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const unsigned char* table = smem;
    // exact fp32 distance of subvector xx to centroid c (as exact_d_umma)
    auto exact = [&](const float (&xx)[DSUB], int c) -> float {
      if constexpr (DSUB == 8) {
        return exact_d_umma<8>(xx, table, c);
      } else {
        const uint2 raw = *reinterpret_cast<const uint2*>(smem + Geo::OFF_CB4 + 8 * c);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        float e = __fsub_rn(xx[0], a.x);
        float d = __fmul_rn(e, e);
        e = __fsub_rn(xx[1], a.y);
        d = __fmaf_rn(e, e, d);
        e = __fsub_rn(xx[2], b.x);
        d = __fmaf_rn(e, e, d);
        e = __fsub_rn(xx[3], b.y);
        return __fmaf_rn(e, e, d);
      }
    };
    int it = 0;
    for (int k = wg; k < n_my; k += 2, ++it) {
      const float inf = __int_as_float(0x7f800000);
      float B1 = inf, B2 = inf, B3 = inf, B4 = inf;
      // the group minimum (from the tensor-memory load's own reduction) with
      // the group id in its 7 low mantissa bits, then the four smallest so
      // far: the packing moves a value by less than 2^-16 of itself, which
      // the margin below covers
      auto group = [&](float g, uint32_t gid) {
        const float gp = __uint_as_float((__float_as_uint(g) & ~0x7Fu) | gid);
        B4 = fminf(B4, fmaxf(B3, gp));
        B3 = fminf(B3, fmaxf(B2, gp));
        B2 = fminf(B2, fmaxf(B1, gp));
        B1 = fminf(B1, gp);
      };
      bool ok = true;
#pragma unroll 1
      for (int q = 0; q < CHUNKS; ++q) {
        const int bsel = q % NBUF;
        const uint32_t use = (uint32_t)(it * (CHUNKS / NBUF) + q / NBUF);
        ok = um_wait(t_full(wg, bsel), use & 1, s_abort, p.err, 0xffffffffu);
        if (!ok) break;
        tcgen05_after_sync();
        const uint32_t col = t_lane + (uint32_t)((NBUF * wg + bsel) * N);
        // the whole chunk in flight at once (one wait); the buffer is handed
        // back before the values are reduced
        float v0[32], v1[32], v2[32], v3[32];
        float g0 = inf, g1 = inf, g2 = inf, g3 = inf;
        tmem_ld32_min(col, v0, g0);
        tmem_ld32_min(col + 32, v1, g1);
        tmem_ld32_min(col + 64, v2, g2);
        tmem_ld32_min(col + 96, v3, g3);
        tmem_wait_ld();
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(t_empty(wg, bsel));
        group(g0, 4u * q);
        group(g1, 4u * q + 1u);
        group(g2, 4u * q + 2u);
        group(g3, 4u * q + 3u);
      }
      if (!ok) break;
      const int s = k % STAGES;
      if (!um_wait(a_full(s), (k / STAGES) & 1, s_abort, p.err, 0xffffffffu)) break;   // (complete already)
      const unsigned char* st = smem + OFF_STAGES + s * STAGE_BYTES;
      const int flag = reinterpret_cast<const int*>(st + ST_FLAG)[ml];
      float xv[DSUB];
      {
        const float4 a = *reinterpret_cast<const float4*>(st + ST_X + (r * kHeadDim + DSUB * j) * 4);
        xv[0] = a.x, xv[1] = a.y, xv[2] = a.z, xv[3] = a.w;
        if constexpr (DSUB == 8) {
          const float4 b = *reinterpret_cast<const float4*>(st + ST_X + (r * kHeadDim + 8 * j + 4) * 4);
          xv[4] = b.x, xv[5] = b.y, xv[6] = b.z, xv[7] = b.w;
        }
      }
      const float eps = screen_eps_hi(sqrtf(reinterpret_cast<const float*>(st + ST_NORM)[ml]), Cmax);
      // a group can hold a candidate within 2 eps of the best when its packed
      // minimum is within 2 eps plus both packing errors (< 2^-16 of each
      // value) of the packed best
      auto near = [&](float X) { return X <= B1 + 2.f * eps + 3.0517578125e-5f * (fabsf(B1) + fabsf(X)); };
      const bool exh = flag == F_EXHAUSTIVE || (flag == F_OK && near(B4));
      const bool need2 = flag == F_OK && !exh && near(B2), need3 = flag == F_OK && !exh && near(B3);
      const int G1 = (int)(__float_as_uint(B1) & 0x7Fu);
      float dex = __int_as_float(0x7f800000), dsec = dex;
      int cex = 0x7fffffff;
      // group G1 by each lane; lane l visits its group's centroids from the
      // (l % 8)-th on (1.5 bit: a centroid's 16 bytes sit in bank group c % 8,
      // so the 32 lanes spread over all 8 bank groups at every step) or the
      // (l % 16)-th on (2 bit: 8 bytes at bank pair c % 16)
      {
        const int rot = lane & (DSUB == 8 ? 7 : 15);
#pragma unroll 8
        for (int i = 0; i < GROUP; ++i) {
          const int c = GROUP * G1 + ((i + rot) & (GROUP - 1));
          exact_push(exact(xv, c), c, dex, cex, dsec);
        }
      }
      // groups G2 / G3 (few lanes) by the whole warp, one (lane, group) at a
      // time, one centroid per lane; exhaustive searches likewise
      const unsigned m2 = __ballot_sync(0xffffffffu, need2), m3 = __ballot_sync(0xffffffffu, need3);
      unsigned mx = __ballot_sync(0xffffffffu, exh);
      for (int pass = 0; pass < 2; ++pass) {
        unsigned mset = pass == 0 ? m2 : m3;
        const float Bp = pass == 0 ? B2 : B3;
        while (mset) {
          const int src = __ffs(mset) - 1;
          mset &= mset - 1;
          const int g = __shfl_sync(0xffffffffu, (int)(__float_as_uint(Bp) & 0x7Fu), src);
          float xs[DSUB];
#pragma unroll
          for (int i = 0; i < DSUB; ++i) xs[i] = __shfl_sync(0xffffffffu, xv[i], src);
          float d = exact(xs, GROUP * g + lane), sd = __int_as_float(0x7f800000);
          int c = GROUP * g + lane;
          exact_warp_reduce(d, c, sd);
          if (lane == src) exact_merge(d, c, sd, dex, cex, dsec);
        }
      }
      while (mx) {
        const int src = __ffs(mx) - 1;
        mx &= mx - 1;
        float xs[DSUB];
#pragma unroll
        for (int i = 0; i < DSUB; ++i) xs[i] = __shfl_sync(0xffffffffu, xv[i], src);
        float d = __int_as_float(0x7f800000), sd = d;
        int c = 0x7fffffff;
        if (!(Cmax <= kScreenCmax)) {   // centroids beyond the table: from global memory
          const __half* cb_head = p.cb + (size_t)kvh * E * DSUB;
          for (int cc = lane; cc < E; cc += 32) {
            const float dd = DSUB == 8 ? exact_d8_cb(xs, cb_head + (size_t)cc * 8) : exact_d4_cb(xs, cb_head + (size_t)cc * 4);
            exact_push(dd, cc, d, c, sd);
          }
        } else {
          for (int cc = lane; cc < E; cc += 32) exact_push(exact(xs, cc), cc, d, c, sd);
        }
        exact_warp_reduce(d, c, sd);
        if (lane == src) dex = d, cex = c, dsec = sd;   // every candidate: replaces the group search
      }
      count_near_ties(p.near_tie, flag != F_SKIP && is_near_tie(dex, dsec), lane, 0xffffffffu);
      const int row = ((int)blockIdx.x + k * (int)gridDim.x) * ROWS + r;
      const int b = row / p.n_rows;
      const int t = flag != F_SKIP ? reinterpret_cast<const int*>(st + ST_POS)[r] : 0;
      if constexpr (MODE == VQKV_MODE_VQ15) {
        // lane (row r, subvector j < 8) stores the pair (j, j + 8) of its row
        const int hi = __shfl_down_sync(0xffffffffu, cex, 8);
        if (j < 8 && flag != F_SKIP) {
          uint8_t* tb = tile_base(p, b, kvh, t, 64, 1536);
          if (tb) store_pair(tb + vq15_pair_offset(p.role, t & 63, j), cex, hi);
        }
      } else if constexpr (MODE == VQKV_MODE_VQ2) {   // one byte per subvector
        if (flag != F_SKIP) {
          uint8_t* tb = tile_base(p, b, kvh, t, 16, 512);
          if (tb) tb[vq2_code_offset(p.role, t & 15, j)] = (uint8_t)cex;
        }
      } else if constexpr (MODE == VQKV_MODE_VQ3) {   // lane j < 16 stores the 12-bit pair (j, j + 16)
        const int hi = __shfl_down_sync(0xffffffffu, cex, 16);
        if (j < 16 && flag != F_SKIP) {
          uint8_t* tb = tile_base(p, b, kvh, t, 16, 768);
          if (tb) {
            tb[vq3_byte_offset(p.role, t & 15, j, 0)] = (uint8_t)(cex & 0xff);
            tb[vq3_byte_offset(p.role, t & 15, j, 1)] = (uint8_t)(((cex >> 8) & 0xf) | ((hi & 0xf) << 4));
            tb[vq3_byte_offset(p.role, t & 15, j, 2)] = (uint8_t)(hi >> 4);
          }
        }
      } else {   // 1.25 bit: lanes j < 4 of each row's half-warp pack a 40-bit group
        const bool key = p.role == VQKV_ROLE_K;
        const int base = lane & 16, g = lane & 3;
        const uint32_t c0 = __shfl_sync(0xffffffffu, cex, base + (key ? g : 2 * g));
        const uint32_t c1 = __shfl_sync(0xffffffffu, cex, base + (key ? g + 4 : 2 * g + 1));
        const uint32_t c2 = __shfl_sync(0xffffffffu, cex, base + (key ? g + 8 : 2 * g + 8));
        const uint32_t c3 = __shfl_sync(0xffffffffu, cex, base + (key ? g + 12 : 2 * g + 9));
        if (j < 4 && flag != F_SKIP) {
          const unsigned long long grp =
              (unsigned long long)(c0 | (c1 << 10) | (c2 << 20)) | ((unsigned long long)c3 << 30);
          uint8_t* tb = tile_base(p, b, kvh, t, 16, 320);
          if (tb) {
            const int rr = t & 15;
            const int run = key ? 4 * (rr & 7) + g : 4 * g + ((rr & 7) >> 1);
            const int n0 = key ? 5 * (rr >> 3) : 5 * (2 * (rr >> 3) + (rr & 1));
#pragma unroll
            for (int q = 0; q < 5; ++q) tb[vq125_run_byte(p.role, run, n0 + q)] = (uint8_t)(grp >> (8 * q));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(a_empty(s));
    }
  }
  tcgen05_before_sync();
  __syncthreads();
  tcgen05_after_sync();
  if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}


// Few rows of 1.5-bit encode (a decode step's append): one row per CTA, its
// 4096 candidates split over the 16 warps (256 each, 32 screening MMAs per
// warp).  The margin test uses the best screened distance over all warps; a
// subvector any of whose 64 lane slices may hide a third candidate within
// the margin is searched exhaustively by the whole CTA.  Decisions equal the
// exhaustive fp32 search's, as in the kernel above.
constexpr size_t kTcSplitSmem = TC_TABLE_BYTES + (128 + 16 + 4 + TC_WARPS * 16 + 16) * 4 +
                                (TC_WARPS * 16 + TC_WARPS) * sizeof(Best);

__global__ void __launch_bounds__(TC_THREADS, 1) encode_vq15_tc_split_kernel(const EncodeParams p) {
  extern __shared__ __align__(16) unsigned char tsm[];
  uint2* s_tbl = reinterpret_cast<uint2*>(tsm);
  float* s_x = reinterpret_cast<float*>(tsm + TC_TABLE_BYTES);   // [128] x'
  float* s_xn = s_x + 128;                                        // [16] |x'_j|^2
  float* s_cmax = s_xn + 16;
  float* s_red = s_cmax + 4;                                      // [warp][16] screened minima
  int* s_hidden = reinterpret_cast<int*>(s_red + TC_WARPS * 16);  // [16]
  Best* s_fin = reinterpret_cast<Best*>(s_hidden + 16);           // [warp][16]
  Best* s_ex = s_fin + TC_WARPS * 16;                             // [warp] exhaustive partials
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  grid_dependency_wait();
  grid_dependents_launch();
  const int rows = p.B * p.n_rows;
  // warp 0 starts the loads of its first row before the table build
  auto row_ptr = [&](int r) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    return p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim + 4 * lane;
  };
  const float* ks = key_s(p, kvh);
  uint2 xraw = make_uint2(0u, 0u);
  float4 xs = make_float4(1.f, 1.f, 1.f, 1.f);
  if (warp == 0 && (int)blockIdx.x < rows) {
    xraw = *reinterpret_cast<const uint2*>(row_ptr(blockIdx.x));
    if (ks != nullptr) xs = *reinterpret_cast<const float4*>(ks + 4 * lane);
  }
  const float Cmax = build_tc_table(p, kvh, s_tbl, s_cmax);
  const bool big = !(Cmax <= kScreenCmax);   // every subvector exhaustive, from global memory
  const __half* cb_head = p.cb + (size_t)kvh * 4096 * 8;
  const uint32_t tbl_lane = smem_u32(s_tbl) + (gid * 4 + tig) * 8;
  const float inf = __int_as_float(0x7f800000);

  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (threadIdx.x == 0 && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    if (warp == 0) {
      float x[4];
      if (r != (int)blockIdx.x) xraw = *reinterpret_cast<const uint2*>(row_ptr(r));
      transform_loaded(xraw, ks != nullptr, xs, lane, x);
      float nx = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
      nx += __shfl_xor_sync(0xffffffffu, nx, 1);   // |x'_j|^2, j = lane / 2
      *reinterpret_cast<float4*>(s_x + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
      if ((lane & 1) == 0) s_xn[lane >> 1] = nx;
      if (lane < 16) s_hidden[lane] = big ? 1 : 0;
    }
    __syncthreads();
    const float2 xa = *reinterpret_cast<const float2*>(s_x + 8 * gid + 2 * tig);
    const float2 xb = *reinterpret_cast<const float2*>(s_x + 8 * (gid + 8) + 2 * tig);
    uint32_t a0, a0l, a1, a1l;
    split_half2(xa.x, xa.y, a0, a0l);
    split_half2(xb.x, xb.y, a1, a1l);
    const uint32_t a2 = tig == 0 ? pack_half2(1.f, 1.f) : 0u;   // picks |c|^2 hi + lo
    const uint32_t a3 = a2;
    float b1[2] = {inf, inf}, b2[2] = {inf, inf};
    int i1[2] = {0, 0};
    const int c_lo = warp * (4096 / TC_WARPS);
#pragma unroll 4
    for (int n0 = c_lo; n0 < c_lo + 4096 / TC_WARPS; n0 += 8) {
      const uint2 bf = lds64(tbl_lane + n0 * 32);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(d, a0, a1, a2, a3, bf.x, bf.y);
      mma_16816(d, a0l, a1l, 0u, 0u, bf.x, bf.y);
      const int c0 = n0 + 2 * tig;
      top2_push(d[0], c0, b1[0], b2[0], i1[0]);
      top2_push(d[1], c0 + 1, b1[0], b2[0], i1[0]);
      top2_push(d[2], c0, b1[1], b2[1], i1[1]);
      top2_push(d[3], c0 + 1, b1[1], b2[1], i1[1]);
    }
    // best screened distance of each subvector over the whole CTA
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float m = b1[h];
      m = fminf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fminf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (tig == 0) s_red[warp * 16 + gid + 8 * h] = m;
    }
    __syncthreads();
    Best cand[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = gid + 8 * h;
      float best = inf;
#pragma unroll 4
      for (int w = 0; w < TC_WARPS; ++w) best = fminf(best, s_red[w * 16 + j]);
      const float xnorm = sqrtf(s_xn[j]);
      const float eps = screen_eps(xnorm, Cmax);
      const float thr = best + 2.f * eps;
      if (b2[h] <= thr) atomicOr(&s_hidden[j], 1);   // a third candidate may hide in this slice
      cand[h] = {inf, inf, 0x7fffffff};
      if (b1[h] <= thr) cand[h] = {exact_d8(s_x + 8 * j, s_tbl, i1[h]), inf, i1[h]};
      // merge the group's 4 lanes: lower distance, then lower index
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) cand[h] = best_merge(cand[h], best_shfl_xor(cand[h], o));
      if (tig == 0) s_fin[warp * 16 + j] = cand[h];
    }
    __syncthreads();
    // subvectors with a possibly hidden candidate: exhaustive exact search,
    // candidate c = threadIdx.x + k * 512 (increasing per thread)
    for (int j = 0; j < 16; ++j) {
      if (!s_hidden[j]) continue;   // uniform: read after the barrier
      Best e = best_init();
      for (int c = threadIdx.x; c < 4096; c += TC_THREADS)
        best_push(e, big ? exact_d8_cb(s_x + 8 * j, cb_head + (size_t)c * 8) : exact_d8(s_x + 8 * j, s_tbl, c), c);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) e = best_merge(e, best_shfl_xor(e, o));
      if (lane == 0) s_ex[warp] = e;
      __syncthreads();
      if (threadIdx.x == 0) {
        Best m = s_ex[0];
        for (int w = 1; w < TC_WARPS; ++w) m = best_merge(m, s_ex[w]);
        s_fin[j] = m;   // warp 0's slot; the other warps' slots are dropped below
      }
      __syncthreads();
    }
    if (warp == 0) {
      const int j = lane & 15;
      Best m = s_fin[j];
      if (!s_hidden[j])
        for (int w = 1; w < TC_WARPS; ++w) m = best_merge(m, s_fin[w * 16 + j]);
      count_near_ties(p.near_tie, is_near_tie(m.d, m.s), lane, 0x0000ffffu);
      const int hi = __shfl_down_sync(0xffffffffu, m.i, 8);
      if (lane < 8) {
        uint8_t* tb = tile_base(p, b, kvh, t, 64, 1536);
        if (tb) store_pair(tb + vq15_pair_offset(p.role, t & 63, lane), m.i, hi);
      }
    }
    __syncthreads();   // s_x, s_hidden and s_fin are reused by the next row
  }
}

}  // namespace

int encode_warps_per_cta() { return ENC_WARPS; }

cudaError_t encode_prepare(int mode) {
  const cudaFuncAttribute smem_attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if (mode == VQKV_MODE_VQ3) {
    cudaError_t e = cudaFuncSetAttribute(encode_vq3_kernel<ENC3_SPLIT>, smem_attr, (int)kEnc3Smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(encode_umma_kernel<VQKV_MODE_VQ3>, smem_attr, (int)UmGeo<VQKV_MODE_VQ3>::SMEM);
    return e;
  }
  if (mode == VQKV_MODE_VQ125)
    return cudaFuncSetAttribute(encode_umma_kernel<VQKV_MODE_VQ125>, smem_attr, (int)UmGeo<VQKV_MODE_VQ125>::SMEM);
  if (mode == VQKV_MODE_VQ2)
    return cudaFuncSetAttribute(encode_umma_kernel<VQKV_MODE_VQ2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)UmGeo<VQKV_MODE_VQ2>::SMEM);
  if (mode != VQKV_MODE_VQ15) return cudaSuccess;
  {
    const cudaError_t e0 = cudaFuncSetAttribute(encode_umma_kernel<VQKV_MODE_VQ15>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)UmGeo<VQKV_MODE_VQ15>::SMEM);
    if (e0 != cudaSuccess) return e0;
    const cudaError_t e1 = cudaFuncSetAttribute(encode_vq15_tc_split_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSplitSmem);
    if (e1 != cudaSuccess) return e1;
  }
  return cudaSuccess;
}

cudaError_t encode_occupancy(int mode, int* blocks_per_sm) {
  if (mode == VQKV_MODE_VQ2)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_umma_kernel<VQKV_MODE_VQ2>,
                                                         um::THREADS, UmGeo<VQKV_MODE_VQ2>::SMEM);
  if (mode == VQKV_MODE_VQ4)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_vq2_kernel<1, 2>, ENC_THREADS, 0);
  if (mode == VQKV_MODE_VQ3)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_umma_kernel<VQKV_MODE_VQ3>,
                                                         um::THREADS, UmGeo<VQKV_MODE_VQ3>::SMEM);
  if (mode == VQKV_MODE_VQ125)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_umma_kernel<VQKV_MODE_VQ125>,
                                                         um::THREADS, UmGeo<VQKV_MODE_VQ125>::SMEM);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_umma_kernel<VQKV_MODE_VQ15>,
                                                       um::THREADS, UmGeo<VQKV_MODE_VQ15>::SMEM);
}

// split_rows: one row per CTA, candidates split over the CTA's warps.
cudaError_t launch_encode(int mode, const EncodeParams& p, int blocks_x, bool split_rows, cudaStream_t stream) {
  const dim3 grid(blocks_x, p.Hkv);
  if (mode == VQKV_MODE_VQ2) {
    if (split_rows) return launch_pdl(encode_vq2_kernel<ENC_WARPS, 4>, grid, dim3(ENC_THREADS), 0, stream, p);
    return launch_pdl(encode_umma_kernel<VQKV_MODE_VQ2>, grid, dim3(um::THREADS), UmGeo<VQKV_MODE_VQ2>::SMEM,
                      stream, p);
  }
  if (mode == VQKV_MODE_VQ4) {
    if (split_rows) return launch_pdl(encode_vq2_kernel<ENC_WARPS, 2>, grid, dim3(ENC_THREADS), 0, stream, p);
    return launch_pdl(encode_vq2_kernel<1, 2>, grid, dim3(ENC_THREADS), 0, stream, p);
  }
  if (mode == VQKV_MODE_VQ125) {
    if (split_rows) return launch_pdl(encode_vq125_kernel<ENC_WARPS>, grid, dim3(ENC_THREADS), 0, stream, p);
    return launch_pdl(encode_umma_kernel<VQKV_MODE_VQ125>, grid, dim3(um::THREADS), UmGeo<VQKV_MODE_VQ125>::SMEM,
                      stream, p);
  }
  if (mode == VQKV_MODE_VQ3) {
    if (split_rows)
      return launch_pdl(encode_vq3_kernel<ENC3_SPLIT>, grid, dim3(ENC3_SPLIT * 32), kEnc3Smem, stream, p);
    return launch_pdl(encode_umma_kernel<VQKV_MODE_VQ3>, grid, dim3(um::THREADS), UmGeo<VQKV_MODE_VQ3>::SMEM,
                      stream, p);
  }
  if (split_rows) return launch_pdl(encode_vq15_tc_split_kernel, grid, dim3(TC_THREADS), kTcSplitSmem, stream, p);
  return launch_pdl(encode_umma_kernel<VQKV_MODE_VQ15>, grid, dim3(um::THREADS), UmGeo<VQKV_MODE_VQ15>::SMEM,
                    stream, p);
}

}  // namespace vqkv
