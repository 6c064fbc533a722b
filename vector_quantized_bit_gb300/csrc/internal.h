// Internal interface between the host shim (api.cu) and the kernel files.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "vqkv.h"

namespace vqkv {

// Everything a decode kernel needs; built and validated by api.cu.
struct DecodeParams {
  const __half* q;          // [B][Hq][128]
  const uint8_t* kc;        // [B][Hkv][stream_bytes]
  const uint8_t* vc;
  const int32_t* seq_lens;  // [B]
  const __half* kcb;        // [Hkv][E][d_sub]
  const __half* vcb;
  const float* s;           // [Hkv][128]
  __half* out;              // [B][Hq][128]
  float* partials;          // [B][Hkv][n_splits][g][kPartialStride]
  unsigned* tickets;        // [B][Hkv], zero between calls
  unsigned* err;            // device error word
  long long stream_bytes;
  int B, Hq, Hkv, g;
  int M = 1;                // queries per sequence (multi-query decode)
  int ncols = 0;            // softmax columns per KV head: M * g (query m, head h -> column m * g + h)
  int cgroups = 1;          // groups of up to 8 columns, one CTA each (grid.z = sequence groups x cgroups)
  int max_seq_len;
  int n_splits;             // CTAs per (sequence, KV head)
  int tps;                  // tiles per split
  int bpg;                  // sequences per CTA (grid.z = ceil(B / bpg))
  int defer_merge;          // 1: split partials are merged by the combine kernel
  int flat = 0;             // 1: flat plan (tile-ring decode, batches): n_splits CTAs per KV head share
                            // all sequences' tiles equally; partials [Hkv][n_splits + B - 1][ncols]
  float qscale;             // softmax_scale * log2(e) / sqrt(128)
  // Fused append (vqkv_decode_append): new rows [B][Hkv][128], or nullptr.
  const __half* k_new = nullptr;
  const __half* v_new = nullptr;
  uint8_t* kc_w = nullptr;  // the same caches as kc / vc, written by the append
  uint8_t* vc_w = nullptr;
  unsigned long long* near_tie = nullptr;
  // Paged cache (vqkv_decode_attn_paged): block table or nullptr.
  const int32_t* block_table = nullptr;
  int max_blocks = 0, block_tiles = 0, block_shift = 0, num_blocks = 0;   // block_tiles = 1 << block_shift
  long long block_bytes = 0;
  // Bounded waits of the 2-bit ring: polls before a wait gives up.  The
  // timeout test withholds every warp's first bulk copy so its waits run out.
  unsigned max_polls = 1u << 22;
  int withhold_first_copy = 0;
};

constexpr int kPartialStride = 132;  // O[128], m, l, pad (rows 16-byte aligned)
constexpr int kFlatMaxB = 1024;      // largest batch the flat plan takes

struct EncodeParams {
  const __half* x;          // [B][Hkv][n_rows][128]
  const int32_t* pos;       // [B]
  const float* s;           // [Hkv][128] (keys) or nullptr
  const __half* cb;         // [Hkv][E][d_sub]
  uint8_t* codes;           // [B][Hkv][stream_bytes]
  unsigned long long* near_tie;
  unsigned* err;
  long long stream_bytes;
  int B, Hkv, n_rows, cap_len, role;
  // Paged cache (vqkv_encode_paged): block table or nullptr.
  const int32_t* block_table = nullptr;
  int max_blocks = 0, block_tiles = 0, block_shift = 0, num_blocks = 0;   // block_tiles = 1 << block_shift
  long long block_bytes = 0;
};

// Decode kernels (decode.cu).  tile_tokens: 16 (VQ2) / 64 (VQ15).
int decode_tile_tokens(int mode);
int decode_tiles_per_step(int mode);   // tiles per split are a multiple of this
size_t decode_smem_bytes(int mode);
int decode_threads(int mode);
cudaError_t decode_prepare(int mode);                // set smem attributes (once per device)
cudaError_t decode_occupancy(int mode, int* blocks_per_sm);
cudaError_t launch_decode(int mode, const DecodeParams& p, dim3 grid, cudaStream_t stream);
// Merge of the split partials into O, after a decode kernel whose plan
// defers the merge (p.defer_merge, n_splits > 1).
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);

// fp16-KV comparison kernel (decode_fp16.cu); DecodeParams.kc / .vc point to
// the fp16 K / V caches, stream_bytes = cap_len * 256.
constexpr int kCodeModes = 5;  // VQKV_MODE_VQ2, VQKV_MODE_VQ15, VQKV_MODE_VQ4, VQKV_MODE_VQ3, VQKV_MODE_VQ125
constexpr int kModeFp16 = kCodeModes;   // plan index after the code modes
size_t decode_fp16_smem_bytes();
int decode_fp16_threads();
cudaError_t decode_fp16_prepare();
cudaError_t decode_fp16_occupancy(int* blocks_per_sm);
cudaError_t launch_decode_fp16(const DecodeParams& p, dim3 grid, cudaStream_t stream);

// Host-side helpers of api.cu shared with decode_static.cu.
vqkv_status decode_validate(const vqkv_decode_args* a);   // every check of vqkv_decode_attn
size_t decode_ticket_region_bytes(int B, int Hkv);       // error word + tickets, bytes

// Encode kernels (encode.cu).
cudaError_t encode_prepare(int mode);
cudaError_t encode_occupancy(int mode, int* blocks_per_sm);
cudaError_t launch_encode(int mode, const EncodeParams& p, int blocks_x, bool split_rows, cudaStream_t stream);
int encode_warps_per_cta();

}  // namespace vqkv
