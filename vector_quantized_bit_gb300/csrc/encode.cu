// VQ encode for sm_103a: smoothing, Hadamard rotation, nearest centroid, pack
// (VecInfer paper summary page, "Summary": channel-wise smoothing followed by
// a Hadamard rotation of the keys, K-Means codebook; arXiv summary page,
// "方法详解", stages 1-2).
//
// One warp per row; lane l holds channels 4l..4l+3.  For keys the transform
// x' = (x / s) . H / sqrt(128) is carried in double-float arithmetic (pairs
// of fp32 with error-free sums and products) and rounded to fp32 once, so the
// vector handed to the nearest-centroid search is the correctly rounded fp32
// value of the exact transform.  Distances are fp32 direct differences; the
// argmin keeps the lowest index on equal distances.
#include "common.cuh"
#include "encode_common.cuh"
#include "internal.h"

namespace vqkv {
namespace {

constexpr int ENC_WARPS = 8;
constexpr int ENC_THREADS = ENC_WARPS * 32;

// Smoothing factors of KV head kvh for keys, nullptr for values.
__device__ __forceinline__ const float* key_s(const EncodeParams& p, int kvh) {
  return p.role == VQKV_ROLE_K ? p.s + (size_t)kvh * kHeadDim : nullptr;
}

// ------------------------------------------------------------------ VQ2
// SPLIT = 1: one warp per row, lane = subvector, 256 candidates per lane.
// SPLIT = 8: the CTA's 8 warps share one row, 32 candidates each (few rows,
// e.g. a decode-step append: latency instead of throughput).
template <int SPLIT>
__global__ void __launch_bounds__(ENC_THREADS) encode_vq2_kernel(const EncodeParams p) {
  __shared__ float4 s_cb[256];
  __shared__ Best s_part[SPLIT > 1 ? ENC_WARPS * 32 : 1];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_dependents_launch();
  for (int c = threadIdx.x; c < 256; c += ENC_THREADS) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.cb) + (size_t)kvh * 256 + c);
    const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
    s_cb[c] = make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
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
    // lane = subvector j (channels 4j..4j+3)
    const Best part = vq2_search(x, c_lo, c_hi, [&](int c) { return s_cb[c]; });
    Best bst = merge_warps<SPLIT>(part, warp, lane, s_part);
    if (SPLIT == 1 || warp == 0) {
      count_near_ties(p.near_tie, is_near_tie(bst.d, bst.s), lane, 0xffffffffu);
      p.codes[((long long)b * p.Hkv + kvh) * p.stream_bytes + vq2_code_offset(p.role, t, lane)] = (uint8_t)bst.i;
    }
  }
}

// ------------------------------------------------------------------ VQ15
// Codebook as fp32 in shared memory (128 KB).  The two lanes of a subvector
// (channels 8J..8J+7 live on lanes 2J, 2J+1) both hold all 8 channels and
// search half of the candidates each (of the CTA's slice when SPLIT > 1).
template <int SPLIT>
__global__ void __launch_bounds__(ENC_THREADS) encode_vq15_kernel(const EncodeParams p) {
  extern __shared__ __align__(16) float4 s_cb15[];   // [4096][2]
  __shared__ Best s_part[SPLIT > 1 ? ENC_WARPS * 32 : 1];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_dependents_launch();
  for (int c = threadIdx.x; c < 4096; c += ENC_THREADS) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.cb) + (size_t)kvh * 4096 + c);
    const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
    const __half2 cc = *reinterpret_cast<const __half2*>(&raw.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&raw.w);
    s_cb15[2 * c] = make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
    s_cb15[2 * c + 1] = make_float4(__low2float(cc), __high2float(cc), __low2float(d), __high2float(d));
  }
  __syncthreads();
  const int rows = p.B * p.n_rows;
  const int half = lane & 1;
  const int r0 = (SPLIT == 1) ? blockIdx.x * ENC_WARPS + warp : blockIdx.x;
  const int rstep = (SPLIT == 1) ? gridDim.x * ENC_WARPS : gridDim.x;
  constexpr int kSlice = 4096 / SPLIT;   // candidates of this warp
  const int c_lo = ((SPLIT == 1) ? 0 : warp * kSlice) + half * (kSlice / 2);
  const int c_hi = c_lo + kSlice / 2;
  for (int r = r0; r < rows; r += rstep) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (lane == 0 && (SPLIT == 1 || warp == 0) && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    float x[4];
    transform_row(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim, key_s(p, kvh), lane, x);
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], 1);
      y[i] = half ? o : x[i];
      y[4 + i] = half ? x[i] : o;
    }
    Best e = best_init(), od = best_init();
#pragma unroll 2
    for (int c = c_lo; c < c_hi; c += 2) {
      float dd[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float4 lo = s_cb15[2 * (c + k)], hi = s_cb15[2 * (c + k) + 1];
        float u = __fsub_rn(y[0], lo.x);
        float d = __fmul_rn(u, u);
        u = __fsub_rn(y[1], lo.y); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[2], lo.z); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[3], lo.w); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[4], hi.x); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[5], hi.y); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[6], hi.z); d = __fmaf_rn(u, u, d);
        u = __fsub_rn(y[7], hi.w); d = __fmaf_rn(u, u, d);
        dd[k] = d;
      }
      best_push(e, dd[0], c);
      best_push(od, dd[1], c + 1);
    }
    // the two halves of the pair hold disjoint candidate sets: merge them
    Best mine = best_merge(e, od);
    Best bst = best_merge(mine, best_shfl_xor(mine, 1));
    bst = merge_warps<SPLIT>(bst, warp, lane, s_part);
    if (SPLIT == 1 || warp == 0) {
      count_near_ties(p.near_tie, is_near_tie(bst.d, bst.s), lane, 0x55555555u);
      // lanes 2p (p < 8) hold subvector p; subvector p+8 sits on lane 2p+16
      const int hi_code = __shfl_down_sync(0xffffffffu, bst.i, 16);
      if (lane < 16 && half == 0) {
        const int pair = lane >> 1;
        const int tile = t >> 6, u = (t & 63) >> 4, rr = t & 15;
        const long long off = (p.role == VQKV_ROLE_K)
                                  ? 1536LL * tile + 48 * (4 * (rr & 7) + (pair & 3)) + 12 * u + 6 * (rr >> 3) + 3 * (pair >> 2)
                                  : 1536LL * tile + 48 * (4 * pair + ((rr & 7) >> 1)) + 12 * u + 3 * ((rr & 1) + 2 * (rr >> 3));
        uint8_t* dst = p.codes + ((long long)b * p.Hkv + kvh) * p.stream_bytes + off;
        dst[0] = (uint8_t)(bst.i & 0xff);
        dst[1] = (uint8_t)(((bst.i >> 8) & 0xf) | ((hi_code & 0xf) << 4));
        dst[2] = (uint8_t)(hi_code >> 4);
      }
    }
  }
}

constexpr size_t kV15EncSmem = 4096 * 2 * sizeof(float4);

// ------------------------------------------------------------------ VQ15, tensor-core screening
// Many rows of 1.5-bit encode: the distance search against 4096 centroids is
// a dense contraction, run as one augmented mma.m16n8k16 per 8 centroids:
//   A[j] = [x~_j (8 ch), 1, |x~_j|^2, 0...]   (16 subvectors of a row; x~ = fp16(x'))
//   B[c] = [-2 c (8 ch), |c|^2, 1, 0...]
//   D[j][c] = |x~_j|^2 + |c|^2 - 2 x~_j.c      (screened squared distance, fp32)
// Each lane keeps the best and second-best screened distance of its
// centroid columns.  A centroid whose screened distance is within 2*eps of
// the best can be the exact nearest, where eps bounds the screening error
// (fp16 rounding of x' and |c|^2, fp32 accumulation); those candidates are
// re-ranked with the exact fp32 direct differences of the CUDA-core search,
// so every decision equals that search's.  If a lane's second-best is also
// within the margin (a third candidate may hide behind it) the subvector is
// searched exhaustively.
constexpr int TC_WARPS = 16;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int TC_TABLE_BYTES = 4096 * 4 * 8;                 // [centroid][tig]{b0b1, b2b3}
constexpr size_t kTcSmem = TC_TABLE_BYTES + TC_WARPS * (128 + 16) * 4 + 16;

__device__ __forceinline__ void top2_push(float v, int n, float& b1, float& b2, int& i1) {
  const bool lt = v < b1;
  b2 = fminf(b2, fmaxf(b1, v));
  b1 = fminf(b1, v);
  i1 = lt ? n : i1;
}

// Exact fp32 distance of subvector x (8 channels) to centroid c, same
// operation order as the CUDA-core search.
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

__global__ void __launch_bounds__(TC_THREADS, 1) encode_vq15_tc_kernel(const EncodeParams p) {
  extern __shared__ __align__(16) unsigned char tsm[];
  uint2* s_tbl = reinterpret_cast<uint2*>(tsm);
  float* s_x = reinterpret_cast<float*>(tsm + TC_TABLE_BYTES);           // [warp][128] x'
  float* s_xn = s_x + TC_WARPS * 128;                                      // [warp][16] |x'_j|^2
  float* s_cmax = s_xn + TC_WARPS * 16;
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  grid_dependency_wait();
  grid_dependents_launch();

  // B table and the largest centroid norm of this KV head
  float cmax = 0.f;
  for (int c = threadIdx.x; c < 4096; c += TC_THREADS) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.cb) + (size_t)kvh * 4096 + c);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
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
    const __half2 tail = __floats2half2_rn(nn, 1.f);
    s_tbl[c * 4 + 0].y = *reinterpret_cast<const uint32_t*>(&tail);
    s_tbl[c * 4 + 1].y = s_tbl[c * 4 + 2].y = s_tbl[c * 4 + 3].y = 0u;
    cmax = fmaxf(cmax, sqrtf(nn));
  }
  for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  if (threadIdx.x == 0) *s_cmax = 0.f;
  __syncthreads();
  if (lane == 0) atomicMax(reinterpret_cast<int*>(s_cmax), __float_as_int(cmax));   // non-negative floats
  __syncthreads();
  const float Cmax = *s_cmax;
  float* wx = s_x + warp * 128;
  float* wxn = s_xn + warp * 16;
  const uint32_t tbl_lane = smem_u32(s_tbl) + (gid * 4 + tig) * 8;   // + 32 per centroid

  const int rows = p.B * p.n_rows;
  for (int r = blockIdx.x * TC_WARPS + warp; r < rows; r += gridDim.x * TC_WARPS) {
    const int b = r / p.n_rows, n = r - b * p.n_rows;
    const int t = p.pos[b] + n;
    if (t < 0 || t >= p.cap_len) {
      if (lane == 0 && p.err) atomicOr(p.err, VQKV_DEVERR_POSITION);
      continue;
    }
    float x[4];
    transform_row(p.x + (((size_t)b * p.Hkv + kvh) * p.n_rows + n) * kHeadDim, key_s(p, kvh), lane, x);
    float nx = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    nx += __shfl_xor_sync(0xffffffffu, nx, 1);   // |x'_j|^2, j = lane / 2
    __syncwarp();
    *reinterpret_cast<float4*>(wx + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    if ((lane & 1) == 0) wxn[lane >> 1] = nx;
    __syncwarp();
    // A fragments: subvectors gid (a0a1, a4a5) and gid+8 (a2a3, a6a7)
    const float2 xa = *reinterpret_cast<const float2*>(wx + 8 * gid + 2 * tig);
    const float2 xb = *reinterpret_cast<const float2*>(wx + 8 * (gid + 8) + 2 * tig);
    const uint32_t a0 = pack_half2(xa.x, xa.y), a1 = pack_half2(xb.x, xb.y);
    const uint32_t a2 = tig == 0 ? pack_half2(1.f, wxn[gid]) : 0u;
    const uint32_t a3 = tig == 0 ? pack_half2(1.f, wxn[gid + 8]) : 0u;

    float b1a = __int_as_float(0x7f800000), b2a = b1a, b1b = b1a, b2b = b1a;
    int i1a = 0, i1b = 0;
#pragma unroll 4
    for (int n0 = 0; n0 < 4096; n0 += 8) {
      const uint2 bf = lds64(tbl_lane + n0 * 32);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(d, a0, a1, a2, a3, bf.x, bf.y);
      const int c0 = n0 + 2 * tig;
      top2_push(d[0], c0, b1a, b2a, i1a);
      top2_push(d[1], c0 + 1, b1a, b2a, i1a);
      top2_push(d[2], c0, b1b, b2b, i1b);
      top2_push(d[3], c0 + 1, b1b, b2b, i1b);
    }
    // per subvector (gid: "a", gid+8: "b"): margin, candidates, exact re-rank
    int code[2];
    bool tie[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = gid + 8 * h;
      float b1 = h ? b1b : b1a, b2 = h ? b2b : b2a;
      const int i1 = h ? i1b : i1a;
      float best = b1;
      best = fminf(best, __shfl_xor_sync(0xffffffffu, best, 1));
      best = fminf(best, __shfl_xor_sync(0xffffffffu, best, 2));
      const float xnorm = sqrtf(wxn[j]);
      const float sc = xnorm + Cmax;
      const float eps = 9.765625e-4f * xnorm * Cmax + 4.8828125e-4f * Cmax * Cmax + 1.5e-5f * sc * sc;
      const float thr = best + 2.f * eps;
      const bool hidden = b2 <= thr;   // a third candidate of this lane may be within the margin
      const bool any_hidden = ((__ballot_sync(0xffffffffu, hidden) >> (4 * gid)) & 0xfu) != 0;
      const float* xj = wx + 8 * j;
      float dex = __int_as_float(0x7f800000), dsec = dex;
      int cex = 0x7fffffff;
      if (!any_hidden) {
        if (b1 <= thr) {
          dex = exact_d8(xj, s_tbl, i1);
          cex = i1;
        }
      } else {
        // exhaustive exact search, the 4 lanes of the group take 1024 centroids each
        for (int c = tig; c < 4096; c += 4) {
          const float dc = exact_d8(xj, s_tbl, c);
          if (dc < dex) {
            dsec = dex;
            dex = dc;
            cex = c;
          } else {
            dsec = fminf(dsec, dc);
          }
        }
      }
      // merge the group's 4 lanes: lower distance, then lower index
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float od = __shfl_xor_sync(0xffffffffu, dex, o);
        const float os = __shfl_xor_sync(0xffffffffu, dsec, o);
        const int oc = __shfl_xor_sync(0xffffffffu, cex, o);
        if (od < dex || (od == dex && oc < cex)) {
          dsec = fminf(dex, os);
          dex = od;
          cex = oc;
        } else {
          dsec = fminf(dsec, od);
        }
      }
      code[h] = cex;
      tie[h] = is_near_tie(dex, dsec);
    }
    count_near_ties(p.near_tie, tie[0], lane, 0x11111111u);
    count_near_ties(p.near_tie, tie[1], lane, 0x11111111u);
    // lane (gid, tig 0) holds the pair (gid, gid+8) of this token
    if (tig == 0) {
      const int pair = gid;
      const int tile = t >> 6, u = (t & 63) >> 4, rr = t & 15;
      const long long off = (p.role == VQKV_ROLE_K)
                                ? 1536LL * tile + 48 * (4 * (rr & 7) + (pair & 3)) + 12 * u + 6 * (rr >> 3) + 3 * (pair >> 2)
                                : 1536LL * tile + 48 * (4 * pair + ((rr & 7) >> 1)) + 12 * u + 3 * ((rr & 1) + 2 * (rr >> 3));
      uint8_t* dst = p.codes + ((long long)b * p.Hkv + kvh) * p.stream_bytes + off;
      dst[0] = (uint8_t)(code[0] & 0xff);
      dst[1] = (uint8_t)(((code[0] >> 8) & 0xf) | ((code[1] & 0xf) << 4));
      dst[2] = (uint8_t)(code[1] >> 4);
    }
  }
}

}  // namespace

int encode_warps_per_cta() { return ENC_WARPS; }

cudaError_t encode_prepare(int mode) {
  if (mode != VQKV_MODE_VQ15) return cudaSuccess;
  {
    const cudaError_t e0 = cudaFuncSetAttribute(encode_vq15_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)kTcSmem);
    if (e0 != cudaSuccess) return e0;
  }
  cudaError_t e = cudaFuncSetAttribute(encode_vq15_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kV15EncSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(encode_vq15_kernel<ENC_WARPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kV15EncSmem);
}

cudaError_t encode_occupancy(int mode, int* blocks_per_sm) {
  if (mode == VQKV_MODE_VQ2)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_vq2_kernel<1>, ENC_THREADS, 0);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_vq15_kernel<1>, ENC_THREADS,
                                                       kV15EncSmem);
}

// split_rows: one row per CTA, candidates split over the CTA's warps.
cudaError_t launch_encode(int mode, const EncodeParams& p, int blocks_x, bool split_rows, cudaStream_t stream) {
  const dim3 grid(blocks_x, p.Hkv);
  if (mode == VQKV_MODE_VQ2) {
    if (split_rows) return launch_pdl(encode_vq2_kernel<ENC_WARPS>, grid, dim3(ENC_THREADS), 0, stream, p);
    return launch_pdl(encode_vq2_kernel<1>, grid, dim3(ENC_THREADS), 0, stream, p);
  }
  if (split_rows) return launch_pdl(encode_vq15_kernel<ENC_WARPS>, grid, dim3(ENC_THREADS), kV15EncSmem, stream, p);
  return launch_pdl(encode_vq15_tc_kernel, grid, dim3(TC_THREADS), kTcSmem, stream, p);
}

}  // namespace vqkv
