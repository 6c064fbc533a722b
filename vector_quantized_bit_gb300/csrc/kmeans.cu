// Offline calibration on the GPU: key smoothing factors, the key transform
// variants of the transform ablation, and K-Means codebook training
// (k-means++ seeding, Lloyd assign / update).
//
// VecInfer ("VecInfer: Efficient LLM Inference with Low-Bit KV Cache via
// Outlier-Suppressed Vector Quantization", summary page, "Summary") smooths
// the keys channel-wise, rotates them with a Hadamard transform and trains
// its codebooks offline with K-Means; "Key points" gives the codebook shapes
// (2^8 x 4, 2^12 x 8) and the ablation over the two transforms and their
// order.  Readings (k-means++ with the draws passed in, distances decided in
// fp32 with ties to the lowest index, fp64 means, empty clusters kept, s_c =
// sqrt(max |K_c|)) follow the calibration oracle.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "vqkv.h"

namespace vqkv {
namespace {

constexpr float kInvSqrt128 = 0.0883883461356163f;   // fp32 nearest to 1/sqrt(128)

// -------------------------------------------------------------- smoothing

// Lane's 4 channels (4*lane .. 4*lane+3) of row r as fp32.
__device__ __forceinline__ float4 load4(const __half* rows, long long r, int lane) {
  const uint2 raw = *reinterpret_cast<const uint2*>(rows + r * kHeadDim + 4 * lane);
  const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}
__device__ __forceinline__ float4 load4(const float* rows, long long r, int lane) {
  return *reinterpret_cast<const float4*>(rows + r * kHeadDim + 4 * lane);
}

// Per-channel max |x| over the rows, folded into mx (fp32 bits: for
// non-negative floats the unsigned order is the numeric order).
template <typename T>
__global__ void __launch_bounds__(256) absmax_kernel(const T* rows, long long n, unsigned* mx) {
  __shared__ float s_m[8][kHeadDim];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long W = ((long long)gridDim.x * blockDim.x) >> 5;
  float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
  for (long long r = (((long long)blockIdx.x * blockDim.x) >> 5) + warp; r < n; r += W) {
    const float4 v = load4(rows, r, lane);
    m0 = fmaxf(m0, fabsf(v.x));
    m1 = fmaxf(m1, fabsf(v.y));
    m2 = fmaxf(m2, fabsf(v.z));
    m3 = fmaxf(m3, fabsf(v.w));
  }
  *reinterpret_cast<float4*>(&s_m[warp][4 * lane]) = make_float4(m0, m1, m2, m3);
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_m[w][threadIdx.x]);
    atomicMax(mx + threadIdx.x, __float_as_uint(m));
  }
}

// s_c = sqrt(max_c) (correctly rounded), 1 where the maximum is 0.
__global__ void smoothing_finish_kernel(float* s) {
  const int c = threadIdx.x;
  const float m = __uint_as_float(reinterpret_cast<unsigned*>(s)[c]);
  s[c] = m > 0.f ? __fsqrt_rn(m) : 1.f;
}

// ------------------------------------------------------------ transforms

// out = rotate(x / s_pre) / s_post, one warp per row, rotation Hn = H/sqrt(128)
// as an in-register fast Walsh-Hadamard transform.
template <typename T>
__global__ void __launch_bounds__(256) calib_transform_kernel(const T* x, long long n, const float* s_pre,
                                                               int rotate, const float* s_post, float* out) {
  const int lane = threadIdx.x & 31;
  const long long W = ((long long)gridDim.x * blockDim.x) >> 5;
  float4 sp = make_float4(1.f, 1.f, 1.f, 1.f), sq = sp;
  if (s_pre) sp = *reinterpret_cast<const float4*>(s_pre + 4 * lane);
  if (s_post) sq = *reinterpret_cast<const float4*>(s_post + 4 * lane);
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n; r += W) {
    const float4 a = load4(x, r, lane);
    float v[4] = {a.x, a.y, a.z, a.w};
    if (s_pre) {
      v[0] = __fdiv_rn(v[0], sp.x), v[1] = __fdiv_rn(v[1], sp.y);
      v[2] = __fdiv_rn(v[2], sp.z), v[3] = __fdiv_rn(v[3], sp.w);
    }
    if (rotate) {
      fwht128_f32(v, lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] *= kInvSqrt128;
    }
    if (s_post) {
      v[0] = __fdiv_rn(v[0], sq.x), v[1] = __fdiv_rn(v[1], sq.y);
      v[2] = __fdiv_rn(v[2], sq.z), v[3] = __fdiv_rn(v[3], sq.w);
    }
    *reinterpret_cast<float4*>(out + r * kHeadDim + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// ---------------------------------------------------------------- K-Means

// ||x - c||^2 from direct differences, fp32, a fixed order of operations.
template <int DIM>
__device__ __forceinline__ float dist2(const float (&x)[DIM], const float* c) {
  float u = __fsub_rn(x[0], c[0]);
  float d = __fmul_rn(u, u);
#pragma unroll
  for (int i = 1; i < DIM; ++i) {
    u = __fsub_rn(x[i], c[i]);
    d = __fmaf_rn(u, u, d);
  }
  return d;
}

template <int DIM>
__device__ __forceinline__ void load_point(const float* pts, long long p, float (&x)[DIM]) {
  if (DIM == 2) {
    const float2 a = *reinterpret_cast<const float2*>(pts + p * DIM);
    x[0] = a.x, x[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < DIM; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(pts + p * DIM + i);
      x[i] = a.x, x[i + 1] = a.y, x[i + 2] = a.z, x[i + 3] = a.w;
    }
  }
}

constexpr int kAssignThreads = 256;
constexpr int kAssignChunk = 1024;   // centroids staged in shared memory at a time

// Nearest centroid of every point (one thread per point): the centroids pass
// through shared memory in chunks, two search chains (even / odd centroids)
// for instruction-level parallelism, merged with the lowest-index rule.
template <int DIM>
__global__ void __launch_bounds__(kAssignThreads) kmeans_assign_kernel(const float* pts, int n, const float* cent,
                                                                       int k, int* out_idx, float* out_dist) {
  __shared__ __align__(16) float s_c[kAssignChunk * DIM];
  const int p = blockIdx.x * kAssignThreads + threadIdx.x;
  float x[DIM];
  if (p < n) {
    load_point<DIM>(pts, p, x);
  } else {
#pragma unroll
    for (int i = 0; i < DIM; ++i) x[i] = 0.f;
  }
  float be = INFINITY, bo = INFINITY;
  int ie = 0, io = 1;
  for (int c0 = 0; c0 < k; c0 += kAssignChunk) {
    const int nc = min(kAssignChunk, k - c0);
    __syncthreads();
    for (int i = threadIdx.x; i < nc * DIM; i += kAssignThreads) s_c[i] = cent[(size_t)c0 * DIM + i];
    __syncthreads();
    int c = 0;
#pragma unroll 2
    for (; c + 1 < nc; c += 2) {
      const float d0 = dist2<DIM>(x, s_c + c * DIM);
      const float d1 = dist2<DIM>(x, s_c + (c + 1) * DIM);
      if (d0 < be) be = d0, ie = c0 + c;
      if (d1 < bo) bo = d1, io = c0 + c + 1;
    }
    if (c < nc) {   // odd chunk length: the last centroid joins the chain of its parity
      const float d = dist2<DIM>(x, s_c + c * DIM);
      const int ci = c0 + c;
      if (ci & 1) {
        if (d < bo) bo = d, io = ci;
      } else if (d < be) {
        be = d, ie = ci;
      }
    }
  }
  if (p < n) {
    const bool odd = bo < be || (bo == be && io < ie);
    out_idx[p] = odd ? io : ie;
    if (out_dist) out_dist[p] = odd ? bo : be;
  }
}

// Lloyd update, deterministic and O(n + k * blocks): the points are put in
// cluster order by a stable counting sort (per-block histograms, one scan,
// a rank-preserving scatter), then each cluster's points are summed in
// index order.
constexpr int kSortBlock = 1024;   // points per histogram / scatter block (one warp each)

// H[c][blk] = points of block blk assigned to cluster c (assignments outside
// [0, k) are not counted).
__global__ void __launch_bounds__(32) sort_count_kernel(const int* __restrict__ idx, int n, int k, int nblk,
                                                        int* __restrict__ H) {
  extern __shared__ int s_cnt[];   // [k]
  const int blk = blockIdx.x, lane = threadIdx.x;
  for (int c = lane; c < k; c += 32) s_cnt[c] = 0;
  __syncwarp();
  const int p0 = blk * kSortBlock, p1 = min(n, p0 + kSortBlock);
  for (int p = p0 + lane; p < p1; p += 32) {
    const int c = __ldg(idx + p);
    if (c >= 0 && c < k) atomicAdd(s_cnt + c, 1);
  }
  __syncwarp();
  for (int c = lane; c < k; c += 32) H[(size_t)c * nblk + blk] = s_cnt[c];
}

// Per cluster (one warp each): H[c][blk] <- exclusive prefix of H[c][:]
// over the blocks, tot[c] <- the cluster's count.
__global__ void __launch_bounds__(256) sort_block_prefix_kernel(int* __restrict__ H, int k, int nblk,
                                                                int* __restrict__ tot) {
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (c >= k) return;
  int* row = H + (size_t)c * nblk;
  int carry = 0;
  for (int b0 = 0; b0 < nblk; b0 += 32) {
    const int h = b0 + lane < nblk ? row[b0 + lane] : 0;
    int v = h;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (b0 + lane < nblk) row[b0 + lane] = carry + v - h;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) tot[c] = carry;
}

// start[c] = exclusive prefix of tot over the clusters, start[k] = total.
__global__ void __launch_bounds__(1024) sort_cluster_scan_kernel(const int* __restrict__ tot, int k,
                                                                 int* __restrict__ start) {
  __shared__ int s_w[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = (k + 1023) / 1024;
  const int lo = min(k, t * per), hi = min(k, lo + per);
  int sum = 0;
  for (int c = lo; c < hi; ++c) sum += tot[c];
  int v = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) s_w[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = s_w[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    s_w[lane] = w;
  }
  __syncthreads();
  int run = v - sum + (warp > 0 ? s_w[warp - 1] : 0);
  for (int c = lo; c < hi; ++c) {
    start[c] = run;
    run += tot[c];
  }
  if (t == 1023) start[k] = s_w[31];
}

// perm[pos] = point index, in cluster order, stable: one warp walks its
// block's points 32 at a time; lanes of a round that share a cluster are
// ranked by lane, and a per-cluster counter carries the rank across rounds.
__global__ void __launch_bounds__(32) sort_scatter_kernel(const int* __restrict__ idx, int n, int k, int nblk,
                                                          const int* __restrict__ H, const int* __restrict__ start,
                                                          int* __restrict__ perm) {
  extern __shared__ int s_cnt[];   // [k] points of each cluster placed so far in this block
  const int blk = blockIdx.x, lane = threadIdx.x;
  for (int c = lane; c < k; c += 32) s_cnt[c] = 0;
  __syncwarp();
  const int p0 = blk * kSortBlock, p1 = min(n, p0 + kSortBlock);
  for (int r = p0; r < p1; r += 32) {
    const int p = r + lane;
    const int c = p < p1 ? __ldg(idx + p) : -1;
    const bool ok = c >= 0 && c < k;
    const unsigned same = __match_any_sync(0xffffffffu, ok ? c : -1);
    const unsigned lower = same & ((1u << lane) - 1u);
    if (ok) {
      const int base = s_cnt[c];
      perm[start[c] + H[(size_t)c * nblk + blk] + base + __popc(lower)] = p;
    }
    __syncwarp();
    if (ok && lower == 0) s_cnt[c] += __popc(same);
    __syncwarp();
  }
}

// c_out[c] = fp64 mean of cluster c's points (sorted positions
// [start[c], start[c+1]), index order), summed by one warp: lane l takes
// positions l, l + 32, ..., then a fixed shuffle tree; c_in[c] if empty.
template <int DIM>
__global__ void __launch_bounds__(256) cluster_mean_kernel(const float* __restrict__ pts, const int* __restrict__ perm,
                                                           const int* __restrict__ start, int k,
                                                           const float* __restrict__ c_in, float* __restrict__ c_out) {
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (c >= k) return;
  const int lo = start[c], hi = start[c + 1];
  double sum[DIM];
#pragma unroll
  for (int i = 0; i < DIM; ++i) sum[i] = 0.0;
  for (int q = lo + lane; q < hi; q += 32) {
    float x[DIM];
    load_point<DIM>(pts, __ldg(perm + q), x);
#pragma unroll
    for (int i = 0; i < DIM; ++i) sum[i] += (double)x[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int i = 0; i < DIM; ++i) sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], off);
  if (lane < DIM) {
    double v = sum[0];
#pragma unroll
    for (int i = 1; i < DIM; ++i) v = lane == i ? sum[i] : v;
    const int cnt = hi - lo;
    c_out[(size_t)c * DIM + lane] = cnt > 0 ? __double2float_rn(v / (double)cnt) : c_in[(size_t)c * DIM + lane];
  }
}

constexpr int kSeedThreads = 1024;
constexpr int kSeedBatch = 8;   // points whose loads are in flight together

// Inclusive scan of one value per thread over the CTA (fixed order: a
// shuffle scan per warp, then over the warp totals).
__device__ __forceinline__ double block_inclusive_scan(double v, double* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    double w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0.0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const double before = warp > 0 ? s_warp[warp - 1] : 0.0;
  __syncthreads();   // s_warp is rewritten by the next scan
  return v + before;
}

// k-means++ seeding in one CTA.  D^2 lives in `d2` (fp32, the same distance
// arithmetic as the assignment); each thread owns a contiguous range of
// points and sums its D^2 in fp64 in index order; the running sums of the
// ranges come from a fixed-order scan.  Centre i (i >= 1) is the first point
// whose inclusive running sum exceeds u[i] * sum D^2 (floor(u[i] * n) when
// every D^2 is 0, the last point when rounding leaves the threshold past the
// end); centre 0 is floor(u[0] * n).  Writes the picks and their
// coordinates.
template <int DIM>
__global__ void __launch_bounds__(kSeedThreads) kmeans_seed_kernel(const float* __restrict__ pts, int n, int k,
                                                                   const float* __restrict__ u, float* __restrict__ d2,
                                                                   int* __restrict__ seeds, float* __restrict__ cent) {
  __shared__ double s_warp[32];
  __shared__ double s_incl[kSeedThreads];
  __shared__ int s_pick;
  const int t = threadIdx.x;
  const int chunk = (n + kSeedThreads - 1) / kSeedThreads;
  const int p_lo = min(n, t * chunk), p_hi = min(n, p_lo + chunk);
  if (t == 0) s_pick = min(n - 1, (int)floor((double)u[0] * (double)n));
  __syncthreads();
  for (int i = 0; i < k; ++i) {
    const int pick = s_pick;
    if (t == 0) seeds[i] = pick;
    if (t < DIM) cent[(size_t)i * DIM + t] = pts[(size_t)pick * DIM + t];
    if (i == k - 1) break;
    float c[DIM];
    load_point<DIM>(pts, pick, c);
    double local = 0.0;
    for (int p0 = p_lo; p0 < p_hi; p0 += kSeedBatch) {
      float x[kSeedBatch][DIM], old[kSeedBatch];
#pragma unroll
      for (int j = 0; j < kSeedBatch; ++j) {
        const int p = min(p0 + j, p_hi - 1);
        load_point<DIM>(pts, p, x[j]);
        old[j] = i == 0 ? INFINITY : d2[p];
      }
#pragma unroll
      for (int j = 0; j < kSeedBatch; ++j) {
        if (p0 + j < p_hi) {
          const float nd = fminf(old[j], dist2<DIM>(x[j], c));
          d2[p0 + j] = nd;
          local += (double)nd;
        }
      }
    }
    // the total and this range's exclusive prefix, both as the scan produced
    // them (the last thread's and the previous thread's inclusive sums)
    const double incl = block_inclusive_scan(local, s_warp);
    s_incl[t] = incl;
    __syncthreads();
    const double total = s_incl[kSeedThreads - 1];
    const double prev = t > 0 ? s_incl[t - 1] : 0.0;
    const double ui = (double)u[i + 1];
    if (!(total > 0.0)) {
      if (t == 0) s_pick = min(n - 1, (int)floor(ui * (double)n));
    } else {
      const double thr = ui * total;
      if (t == 0) s_pick = n - 1;   // the threshold past the last running sum
      __syncthreads();
      // exactly one thread owns the first range whose running sum crosses
      // thr; its warp walks that range 32 points at a time (running sum =
      // the range's prefix + a warp scan) and takes the first point past thr
      const unsigned owner = __ballot_sync(0xffffffffu, prev <= thr && incl > thr && p_lo < p_hi);
      if (owner) {
        const int lane = t & 31, src = __ffs(owner) - 1;
        const int q_lo = __shfl_sync(0xffffffffu, p_lo, src), q_hi = __shfl_sync(0xffffffffu, p_hi, src);
        double carry = __shfl_sync(0xffffffffu, prev, src);
        int found = q_hi - 1;
        for (int q0 = q_lo; q0 < q_hi; q0 += 32) {
          double v = q0 + lane < q_hi ? (double)d2[q0 + lane] : 0.0;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const double o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
          }
          const double acc = carry + v;
          const unsigned past = __ballot_sync(0xffffffffu, q0 + lane < q_hi && acc > thr);
          if (past) {
            found = q0 + __ffs(past) - 1;
            break;
          }
          carry = __shfl_sync(0xffffffffu, acc, 31);
        }
        if (lane == 0) s_pick = found;
      }
    }
    __syncthreads();
  }
}

// The same seeding spread over a cluster of CTAs, each holding a slice of
// the points and their D^2 in shared memory (distributed shared memory for
// the slice totals and the pick).  Slices are contiguous in index order, so
// the running sum in index order is (slices before) + (CTA scan) + (warp
// walk of one thread's points), all in a fixed order.
constexpr int kSeedCtaThreads = 512;

template <int DIM>
__global__ void __launch_bounds__(kSeedCtaThreads) kmeans_seed_cluster_kernel(const float* __restrict__ pts, int n,
                                                                              int k, const float* __restrict__ u,
                                                                              int* __restrict__ seeds,
                                                                              float* __restrict__ cent, int slice) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) float s_dyn[];
  float* sp = s_dyn;                          // [slice][DIM]
  float* sd2 = s_dyn + (size_t)slice * DIM;   // [slice]
  __shared__ double s_warp[32];
  __shared__ double s_incl[kSeedCtaThreads];
  __shared__ double s_ctot[16];
  __shared__ int s_pick;
  const int t = threadIdx.x, lane = t & 31;
  const int rank = (int)cl.block_rank(), C = (int)cl.num_blocks();
  const int g_lo = min(n, rank * slice), m = min(n, g_lo + slice) - g_lo;   // this CTA's points
  for (int i = t; i < m * DIM; i += kSeedCtaThreads) sp[i] = pts[(size_t)g_lo * DIM + i];
  const int per = (m + kSeedCtaThreads - 1) / kSeedCtaThreads;
  const int p_lo = min(m, t * per), p_hi = min(m, p_lo + per);   // local indices of this thread's points
  if (t == 0) s_pick = min(n - 1, (int)floor((double)u[0] * (double)n));
  __syncthreads();
  for (int i = 0; i < k; ++i) {
    const int pick = s_pick;
    if (rank == 0 && t == 0) seeds[i] = pick;
    if (rank == 0 && t < DIM) cent[(size_t)i * DIM + t] = pts[(size_t)pick * DIM + t];
    if (i == k - 1) break;
    float c[DIM];
    load_point<DIM>(pts, pick, c);
    __syncthreads();                       // every thread has read s_pick
    if (t == 0) s_pick = n - 1;            // the threshold past the last running sum
    double local = 0.0;
    for (int p = p_lo; p < p_hi; ++p) {
      float x[DIM];
#pragma unroll
      for (int j = 0; j < DIM; ++j) x[j] = sp[p * DIM + j];
      const float d = dist2<DIM>(x, c);
      const float nd = i == 0 ? d : fminf(sd2[p], d);
      sd2[p] = nd;
      local += (double)nd;
    }
    const double incl = block_inclusive_scan(local, s_warp);
    s_incl[t] = incl;
    __syncthreads();
    if (t == 0) {   // this slice's total into every CTA of the cluster
      const double tot = s_incl[kSeedCtaThreads - 1];
      for (int r = 0; r < C; ++r) *cl.map_shared_rank(&s_ctot[rank], r) = tot;
    }
    cl.sync();
    double total = 0.0, before_me = 0.0;
    for (int r = 0; r < C; ++r) {
      if (r == rank) before_me = total;
      total += s_ctot[r];
    }
    const double ui = (double)u[i + 1];
    if (!(total > 0.0)) {
      if (t == 0) s_pick = min(n - 1, (int)floor(ui * (double)n));
    } else {
      const double thr = ui * total;
      const double prev = before_me + (t > 0 ? s_incl[t - 1] : 0.0);
      const double mine = before_me + incl;
      const unsigned owner = __ballot_sync(0xffffffffu, prev <= thr && mine > thr && p_lo < p_hi);
      if (owner) {   // one warp of one CTA: walk the owner's points
        const int src = __ffs(owner) - 1;
        const int q_lo = __shfl_sync(0xffffffffu, p_lo, src), q_hi = __shfl_sync(0xffffffffu, p_hi, src);
        double carry = __shfl_sync(0xffffffffu, prev, src);
        int found = g_lo + q_hi - 1;
        for (int q0 = q_lo; q0 < q_hi; q0 += 32) {
          double v = q0 + lane < q_hi ? (double)sd2[q0 + lane] : 0.0;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const double o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
          }
          const double acc = carry + v;
          const unsigned past = __ballot_sync(0xffffffffu, q0 + lane < q_hi && acc > thr);
          if (past) {
            found = g_lo + q0 + __ffs(past) - 1;
            break;
          }
          carry = __shfl_sync(0xffffffffu, acc, 31);
        }
        if (lane == 0)
          for (int r = 0; r < C; ++r) *cl.map_shared_rank(&s_pick, r) = found;
      }
    }
    cl.sync();
  }
  cl.sync();   // no CTA leaves while another may still write its shared memory
}

__global__ void to_half_kernel(const float* in, __half* out, int count) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) out[i] = __float2half_rn(in[i]);
}

template <int DIM>
void launch_assign(const float* pts, int n, const float* cent, int k, int* idx, float* dist, cudaStream_t st) {
  kmeans_assign_kernel<DIM><<<(n + kAssignThreads - 1) / kAssignThreads, kAssignThreads, 0, st>>>(pts, n, cent, k,
                                                                                                idx, dist);
}
template <int DIM>
void launch_mean(const float* pts, const int* perm, const int* start, int k, const float* c_in, float* c_out,
                 cudaStream_t st) {
  cluster_mean_kernel<DIM><<<(k + 7) / 8, 256, 0, st>>>(pts, perm, start, k, c_in, c_out);
}
constexpr size_t kSeedSliceSmemMax = 200 * 1024;   // dynamic shared memory for a CTA's slice

// Seeding: a cluster of C CTAs (the smallest C of 1, 2, 4, 8, 16 whose
// slices fit in shared memory, and that the device can schedule), else the
// one-CTA kernel that keeps D^2 in global memory.
template <int DIM>
void launch_seed(const float* pts, int n, int k, const float* u, float* d2, int* seeds, float* cent, cudaStream_t st) {
  auto kern = kmeans_seed_cluster_kernel<DIM>;
  for (int C = 1; C <= 16; C *= 2) {
    const int slice = (n + C - 1) / C;
    const size_t smem = sizeof(float) * (size_t)slice * (DIM + 1);
    if (smem > kSeedSliceSmemMax) continue;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) break;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) break;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kSeedCtaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
      (void)cudaGetLastError();
      break;
    }
    if (cudaLaunchKernelEx(&cfg, kern, pts, n, k, u, seeds, cent, slice) == cudaSuccess) return;
    (void)cudaGetLastError();
    break;
  }
  kmeans_seed_kernel<DIM><<<1, kSeedThreads, 0, st>>>(pts, n, k, u, d2, seeds, cent);
}

#define VQKV_BY_DIM(dim, fn, ...)  \
  switch (dim) {                    \
    case 2: fn<2>(__VA_ARGS__); break; \
    case 4: fn<4>(__VA_ARGS__); break; \
    default: fn<8>(__VA_ARGS__); break; \
  }

cudaError_t smoothing_launch(const void* rows, int dtype, long long n, float* s, int sms, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(s, 0, kHeadDim * sizeof(float), st);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    const long long warps = (n + 3) / 4;   // about 4 rows per warp, at most 4 CTAs per SM
    const int grid = (int)std::min<long long>((warps + 7) / 8, 4LL * sms);
    if (dtype == 0)
      absmax_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(rows), n, reinterpret_cast<unsigned*>(s));
    else
      absmax_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(rows), n, reinterpret_cast<unsigned*>(s));
  }
  smoothing_finish_kernel<<<1, kHeadDim, 0, st>>>(s);
  return cudaGetLastError();
}

cudaError_t calib_transform_launch(const void* x, int dtype, long long n, const float* s_pre, int rotate,
                                   const float* s_post, float* out, int sms, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int grid = (int)std::min<long long>((n + 7) / 8, 8LL * sms);
  if (dtype == 0)
    calib_transform_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(x), n, s_pre, rotate, s_post, out);
  else
    calib_transform_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), n, s_pre, rotate, s_post, out);
  return cudaGetLastError();
}

cudaError_t kmeans_assign_launch(const float* pts, int n, int dim, const float* cent, int k, int* idx, float* dist,
                                 cudaStream_t st) {
  VQKV_BY_DIM(dim, launch_assign, pts, n, cent, k, idx, dist, st);
  return cudaGetLastError();
}

// Scratch of the update: H [k][blocks] | start [k + 1] | perm [n] | tot [k], int32.
size_t update_scratch_bytes(int n, int k) {
  const size_t nblk = (size_t)(n + kSortBlock - 1) / kSortBlock;
  return sizeof(int) * ((size_t)k * std::max<size_t>(nblk, 1) + (size_t)k + 1 + (size_t)n + (size_t)k) + 256;
}

cudaError_t kmeans_update_launch(const float* pts, int n, int dim, const int* idx, int k, const float* c_in,
                                 float* c_out, void* scratch, cudaStream_t st) {
  const int nblk = std::max(1, (n + kSortBlock - 1) / kSortBlock);
  int* H = static_cast<int*>(scratch);
  int* start = H + (size_t)k * nblk;
  int* perm = start + k + 1;
  int* tot = perm + n;
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(H, 0, sizeof(int) * ((size_t)k * nblk), st);
    if (e != cudaSuccess) return e;
  } else {
    sort_count_kernel<<<nblk, 32, sizeof(int) * k, st>>>(idx, n, k, nblk, H);
  }
  sort_block_prefix_kernel<<<(k + 7) / 8, 256, 0, st>>>(H, k, nblk, tot);
  sort_cluster_scan_kernel<<<1, 1024, 0, st>>>(tot, k, start);
  if (n > 0) sort_scatter_kernel<<<nblk, 32, sizeof(int) * k, st>>>(idx, n, k, nblk, H, start, perm);
  VQKV_BY_DIM(dim, launch_mean, pts, perm, start, k, c_in, c_out, st);
  return cudaGetLastError();
}

cudaError_t kmeans_seed_launch(const float* pts, int n, int dim, int k, const float* u, float* d2, int* seeds,
                               float* cent, cudaStream_t st) {
  VQKV_BY_DIM(dim, launch_seed, pts, n, k, u, d2, seeds, cent, st);
  return cudaGetLastError();
}

cudaError_t to_half_launch(const float* in, void* out, int count, cudaStream_t st) {
  to_half_kernel<<<(count + 255) / 256, 256, 0, st>>>(in, static_cast<__half*>(out), count);
  return cudaGetLastError();
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up_to(size_t x, size_t a) { return (x + a - 1) / a * a; }

vqkv_status sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VQKV_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return VQKV_ERR_NO_DEVICE;
  return VQKV_OK;
}

vqkv_status status_of(cudaError_t e) { return e == cudaSuccess ? VQKV_OK : VQKV_ERR_CUDA; }

bool dim_ok(int dim) { return dim == 2 || dim == 4 || dim == 8; }

vqkv_status validate_kmeans_sizes(const vqkv_kmeans_args* a) {
  if (a == nullptr) return VQKV_ERR_INVALID_ARG;
  if (a->n < 1 || !dim_ok(a->dim) || a->k < 1 || a->k > 4096 || a->k > a->n || a->iters < 0 || a->iters > 1000)
    return VQKV_ERR_INVALID_ARG;
  if ((long long)a->n * a->dim > 0x7fffffffLL) return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

// Workspace: D^2 [n] fp32 | assignment [n] int32 | second centroid buffer
// [k][dim] fp32 | the update's sort scratch.
struct KmeansLayout {
  size_t d2 = 0, assign = 0, cent = 0, upd = 0, bytes = 0;
};
KmeansLayout kmeans_layout(const vqkv_kmeans_args* a) {
  KmeansLayout l;
  l.d2 = 0;
  l.assign = round_up_to(sizeof(float) * (size_t)a->n, 256);
  l.cent = l.assign + round_up_to(sizeof(int) * (size_t)a->n, 256);
  l.upd = l.cent + round_up_to(sizeof(float) * (size_t)a->k * a->dim, 256);
  l.bytes = l.upd + round_up_to(update_scratch_bytes(a->n, a->k), 256);
  return l;
}

vqkv_status validate_kmeans(const vqkv_kmeans_args* a, bool need_seeds) {
  vqkv_status st = validate_kmeans_sizes(a);
  if (st != VQKV_OK) return st;
  if (!a->points || !a->uniforms || !a->centroids || (need_seeds && !a->seeds)) return VQKV_ERR_INVALID_ARG;
  if (!aligned_to(a->points, 16) || !aligned_to(a->uniforms, 4) || !aligned_to(a->centroids, 16) ||
      (a->codebook && !aligned_to(a->codebook, 4)) || (a->seeds && !aligned_to(a->seeds, 4)) ||
      (a->assign && !aligned_to(a->assign, 4)))
    return VQKV_ERR_INVALID_ARG;
  if (a->workspace == nullptr || a->workspace_bytes < kmeans_layout(a).bytes) return VQKV_ERR_WORKSPACE;
  if (!aligned_to(a->workspace, 256)) return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

}  // namespace
}  // namespace vqkv

using namespace vqkv;

extern "C" {

vqkv_status vqkv_smoothing(const void* rows, int32_t dtype, int64_t n_rows, float* s, void* stream) {
  if (s == nullptr || n_rows < 0 || (dtype != 0 && dtype != 1) || (n_rows > 0 && rows == nullptr) ||
      !aligned_to(s, 16) || (rows && !aligned_to(rows, 16)))
    return VQKV_ERR_INVALID_ARG;
  int sms = 0;
  vqkv_status st = sm_count(&sms);
  if (st != VQKV_OK) return st;
  return status_of(smoothing_launch(rows, dtype, n_rows, s, sms, static_cast<cudaStream_t>(stream)));
}

vqkv_status vqkv_calib_transform(const void* x, int32_t dtype, int64_t n_rows, const float* s_pre, int32_t rotate,
                                 const float* s_post, float* out, void* stream) {
  if (n_rows < 0 || (dtype != 0 && dtype != 1)) return VQKV_ERR_INVALID_ARG;
  if (n_rows == 0) return VQKV_OK;
  if (!x || !out || !aligned_to(x, 16) || !aligned_to(out, 16) || (s_pre && !aligned_to(s_pre, 16)) ||
      (s_post && !aligned_to(s_post, 16)))
    return VQKV_ERR_INVALID_ARG;
  int sms = 0;
  vqkv_status st = sm_count(&sms);
  if (st != VQKV_OK) return st;
  return status_of(calib_transform_launch(x, dtype, n_rows, s_pre, rotate != 0, s_post, out, sms,
                                          static_cast<cudaStream_t>(stream)));
}

size_t vqkv_kmeans_workspace_bytes(const vqkv_kmeans_args* a) {
  if (validate_kmeans_sizes(a) != VQKV_OK) return 0;
  return kmeans_layout(a).bytes;
}

vqkv_status vqkv_kmeans_seed(const vqkv_kmeans_args* a, void* stream) {
  vqkv_status st = validate_kmeans(a, true);
  if (st != VQKV_OK) return st;
  unsigned char* ws = static_cast<unsigned char*>(a->workspace);
  const KmeansLayout l = kmeans_layout(a);
  return status_of(kmeans_seed_launch(a->points, a->n, a->dim, a->k, a->uniforms, reinterpret_cast<float*>(ws + l.d2),
                                      a->seeds, a->centroids, static_cast<cudaStream_t>(stream)));
}

vqkv_status vqkv_kmeans(const vqkv_kmeans_args* a, void* stream) {
  vqkv_status st = validate_kmeans(a, false);
  if (st != VQKV_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(a->workspace);
  const KmeansLayout l = kmeans_layout(a);
  float* d2 = reinterpret_cast<float*>(ws + l.d2);
  int* idx = a->assign ? a->assign : reinterpret_cast<int*>(ws + l.assign);
  // the seeding's picks go to the caller's buffer or, unused, to the assignment scratch
  int* seeds = a->seeds ? a->seeds : reinterpret_cast<int*>(ws + l.assign);
  float* cur = a->centroids;
  float* nxt = reinterpret_cast<float*>(ws + l.cent);
  cudaError_t e = kmeans_seed_launch(a->points, a->n, a->dim, a->k, a->uniforms, d2, seeds, cur, cs);
  for (int it = 0; e == cudaSuccess && it < a->iters; ++it) {
    e = kmeans_assign_launch(a->points, a->n, a->dim, cur, a->k, idx, nullptr, cs);
    if (e == cudaSuccess) e = kmeans_update_launch(a->points, a->n, a->dim, idx, a->k, cur, nxt, ws + l.upd, cs);
    float* t = cur;
    cur = nxt;
    nxt = t;
  }
  if (e == cudaSuccess && cur != a->centroids)
    e = cudaMemcpyAsync(a->centroids, cur, sizeof(float) * (size_t)a->k * a->dim, cudaMemcpyDeviceToDevice, cs);
  if (e == cudaSuccess && a->codebook) e = to_half_launch(a->centroids, a->codebook, a->k * a->dim, cs);
  return status_of(e);
}

vqkv_status vqkv_kmeans_assign(const float* points, int32_t n, int32_t dim, const float* centroids, int32_t k,
                               int32_t* assign, float* dist, void* stream) {
  if (n < 0 || !dim_ok(dim) || k < 1 || k > 4096) return VQKV_ERR_INVALID_ARG;
  if ((long long)n * dim > 0x7fffffffLL) return VQKV_ERR_INVALID_ARG;
  if (n == 0) return VQKV_OK;
  if (!points || !centroids || !assign || !aligned_to(points, 16) || !aligned_to(centroids, 16) ||
      !aligned_to(assign, 4) || (dist && !aligned_to(dist, 4)))
    return VQKV_ERR_INVALID_ARG;
  return status_of(kmeans_assign_launch(points, n, dim, centroids, k, assign, dist, static_cast<cudaStream_t>(stream)));
}

size_t vqkv_kmeans_update_workspace_bytes(int32_t n, int32_t k) {
  if (n < 0 || k < 1 || k > 4096) return 0;
  return round_up_to(update_scratch_bytes(n, k), 256);
}

vqkv_status vqkv_kmeans_update(const float* points, int32_t n, int32_t dim, const int32_t* assign, int32_t k,
                               const float* c_in, float* c_out, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (n < 0 || !dim_ok(dim) || k < 1 || k > 4096) return VQKV_ERR_INVALID_ARG;
  if ((long long)n * dim > 0x7fffffffLL) return VQKV_ERR_INVALID_ARG;
  if (!c_in || !c_out || (n > 0 && (!points || !assign)) || (points && !aligned_to(points, 16)) ||
      !aligned_to(c_in, 4) || !aligned_to(c_out, 4) || (assign && !aligned_to(assign, 4)))
    return VQKV_ERR_INVALID_ARG;
  const size_t cb = sizeof(float) * (size_t)k * dim;
  const char* i0 = reinterpret_cast<const char*>(c_in);
  const char* o0 = reinterpret_cast<const char*>(c_out);
  if (i0 < o0 + cb && o0 < i0 + cb) return VQKV_ERR_INVALID_ARG;   // overlap
  if (workspace == nullptr || workspace_bytes < vqkv_kmeans_update_workspace_bytes(n, k))
    return VQKV_ERR_WORKSPACE;
  if (!aligned_to(workspace, 256)) return VQKV_ERR_INVALID_ARG;
  return status_of(kmeans_update_launch(points, n, dim, assign, k, c_in, c_out, workspace,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
