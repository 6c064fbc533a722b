// Split-KV decode attention over a plain fp16 KV cache, for comparison with
// the quantised path on the same shapes: O = softmax(scale * q.K^T) . V.
//
// Same skeleton as the VQ kernels (split-KV, GQA grouping, online softmax,
// last-CTA merge), but K and V tiles are read from HBM as fp16 rows:
//   - each warp streams its 16-token tiles of K and V (4 KB each) through a
//     3-stage ring of 16-byte cp.async copies; chunk c of row r lands at
//     chunk c ^ (r & 7) so the ldmatrix reads below are bank-conflict free;
//     rows at or past the sequence length are zero-filled (never read);
//   - scores:  A = K tile (tokens x channels) by ldmatrix, B = q (channels x
//     heads, registers), D: tokens {gid, gid+8} x heads {2tig, 2tig+1};
//   - P:       D -> fp16 -> movmatrix.trans -> B operand of P.V;
//   - P.V:     A = V^T (channels x tokens) by ldmatrix.trans, natural
//     channel order.
#include "common.cuh"
#include "decode_common.cuh"
#include "internal.h"

namespace vqkv {
namespace {

constexpr int F_WARPS = 8;
constexpr int F_THREADS = F_WARPS * 32;
constexpr int F_TILE = 16;
constexpr int F_ROW_BYTES = 256;                      // 128 fp16 channels
constexpr int F_TILE_BYTES = F_TILE * F_ROW_BYTES;    // 4 KB per stream
constexpr int F_STAGES = 3;
constexpr int F_STAGE_BYTES = 2 * F_TILE_BYTES;       // K tile then V tile
constexpr int F_RING_BYTES = F_WARPS * F_STAGES * F_STAGE_BYTES;
constexpr size_t kF16Smem = F_RING_BYTES;             // the combine area reuses the ring
static_assert(CombineSmem<F_WARPS>::kBytes <= F_RING_BYTES, "combine area must fit in the ring");

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * F_ROW_BYTES + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(F_THREADS, 1) decode_fp16_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* s_comb = reinterpret_cast<float*>(smem);   // after the tile loop only
  __shared__ int s_last;

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int b_begin = blockIdx.z * p.bpg;
  const int b_end = min(b_begin + p.bpg, p.B);
  const uint32_t ring = smem_u32(smem) + warp * (F_STAGES * F_STAGE_BYTES);
  grid_dependency_wait();
  grid_dependents_launch();

  for (int b = b_begin; b < b_end; ++b) {
    const int L = load_len(p, b);
    const int ntiles = (L + F_TILE - 1) / F_TILE;
    const int t_begin = split * p.tps;
    const int t_end = min(t_begin + p.tps, ntiles);
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = kMInit, m1 = kMInit, l0 = 0.f, l1 = 0.f;

    if (t_begin < t_end) {
      const unsigned char* kbase = p.kc + (size_t)(b * p.Hkv + kvh) * p.stream_bytes;
      const unsigned char* vbase = p.vc + (size_t)(b * p.Hkv + kvh) * p.stream_bytes;
      const int first = t_begin + warp;
      const int n_mine = first < t_end ? (t_end - first + F_WARPS - 1) / F_WARPS : 0;
      // tile j of this warp -> stage j % F_STAGES; 16 chunks per lane, rows
      // at or past L zero-filled
      auto issue = [&](int j) {
        if (j < n_mine) {
          const int tile = first + j * F_WARPS;
          const uint32_t st = ring + (j % F_STAGES) * F_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = lane + 32 * k;                 // chunk index in the tile
            const int row = i >> 4, c = i & 15;
            const long long t = (long long)tile * F_TILE + row;
            const uint32_t n = (t < L) ? 16u : 0u;
            const size_t off = (size_t)(t < L ? t : 0) * F_ROW_BYTES + c * 16;
            cp_async16(st + swz(row, c), kbase + off, n);
            cp_async16(st + F_TILE_BYTES + swz(row, c), vbase + off, n);
          }
        }
        cp_async_commit();   // one group per step, empty ones included
      };
      issue(0);
      issue(1);
      // B operand of the score MMA: q of head gid, channels 16s + 2tig (+1, +8, +9)
      uint32_t qf[8][2];
      {
        const bool real = gid < p.g;
        const __half* qrow = p.q + ((size_t)b * p.Hq + kvh * p.g + (real ? gid : 0)) * kHeadDim;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const __half2 x = *reinterpret_cast<const __half2*>(qrow + 16 * s + 2 * tig);
          const __half2 y = *reinterpret_cast<const __half2*>(qrow + 16 * s + 2 * tig + 8);
          qf[s][0] = real ? pack_half2(__low2float(x) * p.qscale, __high2float(x) * p.qscale) : 0u;
          qf[s][1] = real ? pack_half2(__low2float(y) * p.qscale, __high2float(y) * p.qscale) : 0u;
        }
      }
      // ldmatrix row addresses of this lane (before the stage base):
      //   scores: token (lane&7) + 8*((lane>>3)&1), chunk 2s + (lane>>4)
      //   P.V:    token (lane&7) + 8*(lane>>4),     chunk 2mt + ((lane>>3)&1)
      const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1), k_hi = lane >> 4;
      const int v_row = (lane & 7) + 8 * (lane >> 4), v_hi = (lane >> 3) & 1;

      for (int j = 0; j < n_mine; ++j) {
        cp_async_wait<F_STAGES - 2>();
        __syncwarp();
        issue(j + F_STAGES - 1);   // into the stage used by step j - 1
        const uint32_t kst = ring + (j % F_STAGES) * F_STAGE_BYTES;
        const uint32_t vst = kst + F_TILE_BYTES;
        const int tile = first + j * F_WARPS;
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t a[4];
          ldmatrix_x4(a, kst + swz(k_row, 2 * s + k_hi));
          if (s & 1)
            mma_16816(sb, a[0], a[1], a[2], a[3], qf[s][0], qf[s][1]);
          else
            mma_16816(sa, a[0], a[1], a[2], a[3], qf[s][0], qf[s][1]);
        }
        float sc[4] = {sa[0] + sb[0], sa[1] + sb[1], sa[2] + sb[2], sa[3] + sb[3]};
        if ((tile + 1) * F_TILE > L) {
          const int t0 = tile * F_TILE + gid;
          if (t0 >= L) sc[0] = sc[1] = neg_inf();
          if (t0 + 8 >= L) sc[2] = sc[3] = neg_inf();
        }
        uint32_t bP0, bP1;
        softmax_tile(sc, m0, m1, l0, l1, acc, bP0, bP1);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, vst + swz(v_row, 2 * mt + v_hi));
          mma_16816(acc[mt], a[0], a[1], a[2], a[3], bP0, bP1);
        }
      }
      cp_async_wait<0>();
    }
    __syncthreads();   // every warp is done with its ring: reuse it for the combine
    stash_warp<F_WARPS, 8>(s_comb, warp, lane, acc, m0, m1, l0, l1, NaturalDim());
    __syncthreads();
    finish_sequence<F_WARPS, false, NaturalDim>(p, b, kvh, split_span(p, b, kvh, split, 0), s_comb, &s_last);
    __syncthreads();
  }
}

}  // namespace

size_t decode_fp16_smem_bytes() { return kF16Smem; }
int decode_fp16_threads() { return F_THREADS; }

cudaError_t decode_fp16_prepare() {
  return cudaFuncSetAttribute(decode_fp16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kF16Smem);
}

cudaError_t decode_fp16_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_fp16_kernel, F_THREADS, kF16Smem);
}

cudaError_t launch_decode_fp16(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  return launch_pdl(decode_fp16_kernel, grid, dim3(F_THREADS), kF16Smem, stream, p);
}

}  // namespace vqkv
