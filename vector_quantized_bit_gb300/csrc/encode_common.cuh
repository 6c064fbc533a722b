// Device code of the encode step shared by the encode kernels (encode.cu)
// and the decode kernel's fused append (decode.cu): the key transform in
// double-float arithmetic, the nearest-centroid search state and the 2-bit
// search loop (VecInfer paper summary page, "Summary": smoothing, Hadamard
// rotation, nearest codebook centroid).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace vqkv {
namespace {

// ------------------------------------------------------- double-float
struct df {
  float h, l;
};

__device__ __forceinline__ df fast_two_sum(float a, float b) {   // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  const float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}

__device__ __forceinline__ df two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ df df_add(df a, df b) {
  df s = two_sum(a.h, b.h);
  const float e = __fadd_rn(s.l, __fadd_rn(a.l, b.l));
  return fast_two_sum(s.h, e);
}

__device__ __forceinline__ df df_neg(df a) { return {-a.h, -a.l}; }

__device__ __forceinline__ df df_mul(df a, float ch, float cl) {
  const float p = __fmul_rn(a.h, ch);
  float e = __fmaf_rn(a.h, ch, -p);
  e = __fmaf_rn(a.h, cl, e);
  e = __fmaf_rn(a.l, ch, e);
  return fast_two_sum(p, e);
}

// x / s as a double-float: quotient, plus the exact remainder divided by s.
__device__ __forceinline__ df df_div(float x, float s) {
  const float q = __fdiv_rn(x, s);
  const float r = __fmaf_rn(-q, s, x);
  return fast_two_sum(q, __fdiv_rn(r, s));
}

// Unnormalised FWHT (H[i][k] = (-1)^popcount(i & k)) of a 128-vector in
// double-float, 4 entries per lane.
__device__ __forceinline__ void fwht128_df(df (&v)[4], int lane) {
  {
    const df a = df_add(v[0], v[1]), b = df_add(v[0], df_neg(v[1]));
    const df c = df_add(v[2], v[3]), d = df_add(v[2], df_neg(v[3]));
    v[0] = df_add(a, c);
    v[2] = df_add(a, df_neg(c));
    v[1] = df_add(b, d);
    v[3] = df_add(b, df_neg(d));
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      df o;
      o.h = __shfl_xor_sync(0xffffffffu, v[i].h, m);
      o.l = __shfl_xor_sync(0xffffffffu, v[i].l, m);
      v[i] = upper ? df_add(o, df_neg(v[i])) : df_add(v[i], o);
    }
  }
}

// sqrt(2) as fp32 hi + lo; 1/sqrt(128) = sqrt(2) / 16.
__device__ __forceinline__ float sqrt2_hi() { return __int_as_float(0x3fb504f3); }
__device__ __forceinline__ float sqrt2_lo() { return __int_as_float(0x32cfe77a); }

// Transform of one row from the lane's four fp16 channels (raw) and, for a
// key, their smoothing factors s: fp32 result.  Values stay as they are.
__device__ __forceinline__ void transform_loaded(uint2 raw, bool key, float4 s, int lane, float (&x)[4]) {
  const __half2 x01 = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 x23 = *reinterpret_cast<const __half2*>(&raw.y);
  x[0] = __low2float(x01);
  x[1] = __high2float(x01);
  x[2] = __low2float(x23);
  x[3] = __high2float(x23);
  if (key) {
    df v[4] = {df_div(x[0], s.x), df_div(x[1], s.y), df_div(x[2], s.z), df_div(x[3], s.w)};
    fwht128_df(v, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const df r = df_mul(v[i], sqrt2_hi(), sqrt2_lo());
      x[i] = __fmul_rn(r.h, 0.0625f);   // exact scaling; r.h is RN(r.h + r.l)
    }
  }
}

// s + t as a hi + lo pair with lo = the rounding error of s + the low parts
// (TwoSum, no renormalisation); 8 operations.
__device__ __forceinline__ void lean_add(float ah, float al, float bh, float bl, float& sh, float& sl) {
  const float t = __fadd_rn(ah, bh);
  const float bb = __fsub_rn(t, ah);
  const float e = __fadd_rn(__fsub_rn(ah, __fsub_rn(t, bb)), __fsub_rn(bh, bb));
  sh = t;
  sl = __fadd_rn(__fadd_rn(al, bl), e);
}

// The key transform of transform_loaded in fewer operations, for the
// encode kernels: x / s as the product with the reciprocal rs = RN(1 / s)
// plus the FMA remainder times rs, and each butterfly's rounding error
// carried in an fp32 low part without renormalisation; the sum is rounded
// once at the end.  Every term keeps a relative error near 2^-44, so the
// result is the correctly rounded fp32 of the fp64 transform except where
// that lies within about 2^-20 of an fp32 ulp of a rounding boundary.
__device__ __forceinline__ void transform_key_lean(uint2 raw, float4 s, float4 rs, int lane, float (&x)[4]) {
  const __half2 x01 = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 x23 = *reinterpret_cast<const __half2*>(&raw.y);
  const float xv[4] = {__low2float(x01), __high2float(x01), __low2float(x23), __high2float(x23)};
  const float sv[4] = {s.x, s.y, s.z, s.w}, rv[4] = {rs.x, rs.y, rs.z, rs.w};
  float h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = __fmul_rn(xv[i], rv[i]);
    l[i] = __fmul_rn(__fmaf_rn(-h[i], sv[i], xv[i]), rv[i]);
  }
  {
    float ah, al, bh, bl, ch, cl, dh, dl;
    lean_add(h[0], l[0], h[1], l[1], ah, al);
    lean_add(h[0], l[0], -h[1], -l[1], bh, bl);
    lean_add(h[2], l[2], h[3], l[3], ch, cl);
    lean_add(h[2], l[2], -h[3], -l[3], dh, dl);
    lean_add(ah, al, ch, cl, h[0], l[0]);
    lean_add(ah, al, -ch, -cl, h[2], l[2]);
    lean_add(bh, bl, dh, dl, h[1], l[1]);
    lean_add(bh, bl, -dh, -dl, h[3], l[3]);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float oh = __shfl_xor_sync(0xffffffffu, h[i], m);
      const float ol = __shfl_xor_sync(0xffffffffu, l[i], m);
      // lower lane: v + o; upper lane: o - v
      lean_add(oh, ol, upper ? -h[i] : h[i], upper ? -l[i] : l[i], h[i], l[i]);
    }
  }
  // x' = (h + l) * sqrt(2) / 16, rounded once
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const df v = two_sum(h[i], l[i]);
    const float pr = __fmul_rn(v.h, sqrt2_hi());
    float e = __fmaf_rn(v.h, sqrt2_hi(), -pr);
    e = __fmaf_rn(v.h, sqrt2_lo(), e);
    e = __fmaf_rn(v.l, sqrt2_hi(), e);
    x[i] = __fmul_rn(__fadd_rn(pr, e), 0.0625f);
  }
}

// The same, reading the lane's 4 fp16 channels and smoothing factors (keys
// through transform_key_lean).
__device__ __forceinline__ void transform_row(const __half* xrow, const float* s_row, int lane, float (&x)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(xrow + 4 * lane);
  if (s_row == nullptr) {
    transform_loaded(raw, false, make_float4(1.f, 1.f, 1.f, 1.f), lane, x);
    return;
  }
  const float4 s = *reinterpret_cast<const float4*>(s_row + 4 * lane);
  transform_key_lean(raw, s, make_float4(__frcp_rn(s.x), __frcp_rn(s.y), __frcp_rn(s.z), __frcp_rn(s.w)), lane, x);
}

// Adds the lanes of `mask` whose `tie` is set to *counter (if not null).
__device__ __forceinline__ void count_near_ties(unsigned long long* counter, bool tie, int lane, unsigned mask) {
  if (counter == nullptr) return;
  const unsigned n = __popc(__ballot_sync(0xffffffffu, tie) & mask);
  if (lane == 0 && n) atomicAdd(counter, (unsigned long long)n);
}

__device__ __forceinline__ bool is_near_tie(float best, float second) {
  return __fsub_rn(second, best) < 1e-6f * fmaxf(best, 1e-30f);
}

// Running nearest-centroid state of one search chain: best distance, its
// index, second-best distance.  Chains scan disjoint candidate sets in
// increasing index order, so a strict "<" keeps the lowest index on ties.
struct Best {
  float d, s;
  int i;
};

__device__ __forceinline__ Best best_init() {
  const float inf = __int_as_float(0x7f800000);
  return {inf, inf, 0};
}

__device__ __forceinline__ void best_push(Best& b, float d, int c) {
  const bool lt = d < b.d;
  b.s = lt ? b.d : fminf(b.s, d);
  b.i = lt ? c : b.i;
  b.d = lt ? d : b.d;
}

// Merge two chains over disjoint candidates: lower distance, then lower index.
__device__ __forceinline__ Best best_merge(Best a, Best b) {
  if (b.d < a.d || (b.d == a.d && b.i < a.i)) return {b.d, fminf(a.d, b.s), b.i};
  return {a.d, fminf(a.s, b.d), a.i};
}

__device__ __forceinline__ Best best_shfl_xor(Best b, int m) {
  return {__shfl_xor_sync(0xffffffffu, b.d, m), __shfl_xor_sync(0xffffffffu, b.s, m),
          __shfl_xor_sync(0xffffffffu, b.i, m)};
}

// Cross-warp merge for SPLIT > 1: every warp searched a slice of the
// candidates for the same row; warp 0 ends up with the merged state.
template <int SPLIT>
__device__ __forceinline__ Best merge_warps(Best b, int warp, int lane, Best* s_part) {
  if (SPLIT == 1) return b;
  __syncthreads();   // the previous row's readers are done with s_part
  s_part[warp * 32 + lane] = b;
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int w = 1; w < SPLIT; ++w) b = best_merge(b, s_part[w * 32 + lane]);
  }
  return b;
}

// 2-bit search of one subvector (lane's 4 channels x) over candidates
// [c_lo, c_hi) (an even count): fp32 direct differences, two chains over
// even / odd candidates, merged.  load(c) returns centroid c as a float4.
template <typename Load>
__device__ __forceinline__ Best vq2_search(const float (&x)[4], int c_lo, int c_hi, Load load) {
  Best e = best_init(), o = best_init();
#pragma unroll 4
  for (int c = c_lo; c < c_hi; c += 2) {
    const float4 ca = load(c), cb = load(c + 1);
    float u = __fsub_rn(x[0], ca.x), d0 = __fmul_rn(u, u);
    u = __fsub_rn(x[1], ca.y); d0 = __fmaf_rn(u, u, d0);
    u = __fsub_rn(x[2], ca.z); d0 = __fmaf_rn(u, u, d0);
    u = __fsub_rn(x[3], ca.w); d0 = __fmaf_rn(u, u, d0);
    float v = __fsub_rn(x[0], cb.x), d1 = __fmul_rn(v, v);
    v = __fsub_rn(x[1], cb.y); d1 = __fmaf_rn(v, v, d1);
    v = __fsub_rn(x[2], cb.z); d1 = __fmaf_rn(v, v, d1);
    v = __fsub_rn(x[3], cb.w); d1 = __fmaf_rn(v, v, d1);
    best_push(e, d0, c);
    best_push(o, d1, c + 1);
  }
  return best_merge(e, o);
}

// Byte offset of 2-bit code (token t, subvector j) in a K or V stream
// (the layout of include/vqkv.h).
__device__ __forceinline__ long long vq2_code_offset(int role, int t, int j) {
  const int tile = t >> 4, rr = t & 15;
  return (role == VQKV_ROLE_K)
             ? 512LL * tile + 16 * (4 * (rr & 7) + (j & 3)) + 8 * (rr >> 3) + (j >> 2)
             : 512LL * tile + 16 * (4 * (j & 7) + ((rr & 7) >> 1)) + 4 * (j >> 3) + 2 * (rr >> 3) + (rr & 1);
}

// 4-bit search of the lane's two subvectors (channels (x0, x1) and (x2, x3))
// over candidates [c_lo, c_hi) (an even count): fp32 direct differences,
// even / odd chains per subvector, merged.  load(c) returns centroid c as a
// float2.
template <typename Load>
__device__ __forceinline__ void vq4_search(const float (&x)[4], int c_lo, int c_hi, Load load, Best& a, Best& b) {
  Best ae = best_init(), ao = best_init(), be = best_init(), bo = best_init();
#pragma unroll 4
  for (int c = c_lo; c < c_hi; c += 2) {
    const float2 ca = load(c), cb = load(c + 1);
    float u = __fsub_rn(x[0], ca.x), d = __fmul_rn(u, u);
    u = __fsub_rn(x[1], ca.y), d = __fmaf_rn(u, u, d);
    best_push(ae, d, c);
    u = __fsub_rn(x[0], cb.x), d = __fmul_rn(u, u);
    u = __fsub_rn(x[1], cb.y), d = __fmaf_rn(u, u, d);
    best_push(ao, d, c + 1);
    u = __fsub_rn(x[2], ca.x), d = __fmul_rn(u, u);
    u = __fsub_rn(x[3], ca.y), d = __fmaf_rn(u, u, d);
    best_push(be, d, c);
    u = __fsub_rn(x[2], cb.x), d = __fmul_rn(u, u);
    u = __fsub_rn(x[3], cb.y), d = __fmaf_rn(u, u, d);
    best_push(bo, d, c + 1);
  }
  a = best_merge(ae, ao);
  b = best_merge(be, bo);
}

// Byte offset of the 4-bit code (one byte) of subvector j (0..63) of token
// t in a K or V stream (the layout of include/vqkv.h).
__device__ __forceinline__ long long vq4_code_offset(int role, int t, int j) {
  const int tile = t >> 4, rr = t & 15;
  return (role == VQKV_ROLE_K)
             ? 1024LL * tile + 512 * (rr >> 3) + 16 * (4 * (rr & 7) + (j & 3)) + 2 * (j >> 3) + ((j >> 2) & 1)
             : 1024LL * tile + 512 * (j >> 5) + 16 * (4 * (j & 7) + ((rr & 7) >> 1)) + 4 * ((j >> 3) & 3) +
                   2 * (rr >> 3) + (rr & 1);
}

// Byte offset of the first byte of 1.5-bit pair `pair` (subvectors pair and
// pair + 8) of token t in a K or V stream (the layout of include/vqkv.h).
__device__ __forceinline__ long long vq15_pair_offset(int role, int t, int pair) {
  const int tile = t >> 6, u = (t & 63) >> 4, rr = t & 15;
  return (role == VQKV_ROLE_K)
             ? 1536LL * tile + 48 * (4 * (rr & 7) + (pair & 3)) + 12 * u + 6 * (rr >> 3) + 3 * (pair >> 2)
             : 1536LL * tile + 48 * (4 * pair + ((rr & 7) >> 1)) + 12 * u + 3 * ((rr & 1) + 2 * (rr >> 3));
}

// Byte offset of byte k (0..2) of 3-bit pair `pair` (subvectors pair and
// pair + 16) of token t in a K or V stream (the layout of include/vqkv.h:
// each lane's 24-byte run split into a 16-byte and an 8-byte plane).
__device__ __forceinline__ long long vq3_byte_offset(int role, int t, int pair, int k) {
  const int tile = t >> 4, rr = t & 15;
  const int lane = (role == VQKV_ROLE_K) ? 4 * (rr & 7) + (pair & 3) : 4 * (pair & 7) + ((rr & 7) >> 1);
  const int n = (role == VQKV_ROLE_K) ? 12 * (rr >> 3) + 3 * (pair >> 2) + k
                                      : 6 * (2 * (rr >> 3) + (rr & 1)) + 3 * (pair >> 3) + k;
  return 768LL * tile + (n < 16 ? 16 * lane + n : 512 + 8 * lane + n - 16);
}

// Byte offset within a 1.25-bit tile of byte n of K run L (10 bytes: 8 in
// plane 0, 2 in plane 1) or V run R (20 bytes: 16 + 4) (the layout of
// include/vqkv.h).
__device__ __forceinline__ int vq125_run_byte(int role, int run, int n) {
  return (role == VQKV_ROLE_K) ? (n < 8 ? 8 * run + n : 256 + 2 * run + n - 8)
                               : (n < 16 ? 16 * run + n : 256 + 4 * run + n - 16);
}

// Writes codes lo (subvector pair) and hi (pair + 8) as 3 bytes.
__device__ __forceinline__ void store_pair(uint8_t* dst, int lo, int hi) {
  dst[0] = (uint8_t)(lo & 0xff);
  dst[1] = (uint8_t)(((lo >> 8) & 0xf) | ((hi & 0xf) << 4));
  dst[2] = (uint8_t)(hi >> 4);
}

}  // namespace
}  // namespace vqkv
