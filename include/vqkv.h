/*
 * vqkv.h — C ABI of the GB300 (sm_103a) VQ KV-cache library.
 *
 * The library implements the hot path of VecInfer ("VecInfer: Efficient LLM
 * Inference with Low-Bit KV Cache via Outlier-Suppressed Vector
 * Quantization"): keys are smoothed channel-wise and rotated by a Hadamard
 * transform, every subvector of a key or value row is replaced by the index
 * of its nearest codebook centroid, and decode attention runs directly on
 * the packed indices with dequantisation fused into the score, softmax and
 * P.V loop (paper summary page, "Summary"; codebook shapes 2^8 x 4 for
 * 2 bit and 2^12 x 8 for 1.5 bit, "Key points"; the three stages
 * preprocessing -> quantisation -> fused kernel, arXiv summary page,
 * "方法详解").
 *
 * Conventions for every call:
 *   - Pointers named "device" point to memory on the current CUDA device and
 *     are owned by the caller.  The library allocates nothing, keeps no
 *     pointer after a call returns and holds no mutable global state beyond a
 *     per-device cache of device attributes.
 *   - fp16 data are passed as uint16_t bit patterns (IEEE binary16).
 *   - head_dim must be 128.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns a status and launches nothing.  Work is enqueued
 *     asynchronously on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream); no call synchronises the host.
 *   - A launch failure returns VQKV_ERR_CUDA.  Conditions that can only be
 *     seen on the device (a sequence length above max_seq_len, a cache
 *     position outside the capacity) never fault: the kernel clamps or skips
 *     and sets a bit in a caller-visible device error word.
 *   - Calls on different streams may run concurrently as long as they do not
 *     write the same buffers (workspaces included).
 *
 * Packed cache layout (the contract between vqkv_encode, vqkv_decode_attn and
 * any reader).  Each (sequence b, KV head h) owns one K stream and one V
 * stream of vqkv_code_bytes(mode, cap_len) bytes, at byte offset
 * (b * Hkv + h) * vqkv_code_bytes(mode, cap_len) of the codes buffer.  A
 * stream is a sequence of tiles; token t lives in tile t / TILE.
 *
 *   VQKV_MODE_VQ2 (256 entries x 4 dims, 8-bit codes, 32 codes per token):
 *     TILE = 16 tokens, 512 bytes.  With r = t % 16 and subvector j (0..31):
 *       K: byte 512*(t/16) + 16*(4*(r%8) + j%4) + 8*(r/8) + j/4
 *       V: byte 512*(t/16) + 16*(4*(j%8) + (r%8)/2) + 4*(j/8) + 2*(r/8) + r%2
 *     holds the code (0..255) of subvector j (channels 4j..4j+3) of token t.
 *   VQKV_MODE_VQ15 (4096 entries x 8 dims, 12-bit codes, 16 codes per token):
 *     the codes of subvectors p and p+8 (p = 0..7) of one token form a pair
 *     stored in 3 bytes: b0 = c_p & 0xFF, b1 = (c_p >> 8) | ((c_{p+8} & 0xF) << 4),
 *     b2 = c_{p+8} >> 4.  TILE = 64 tokens, 1536 bytes.  With
 *     u = (t % 64) / 16 and r = t % 16, the first byte of pair p of token t is
 *       K: 1536*(t/64) + 48*(4*(r%8) + p%4) + 12*u + 6*(r/8) + 3*(p/4)
 *       V: 1536*(t/64) + 48*(4*p + (r%8)/2) + 12*u + 3*((r%2) + 2*(r/8))
 *   VQKV_MODE_VQ4 (256 entries x 2 dims, 8-bit codes, 64 codes per token;
 *   within the 1.25-4 bit range the paper's summary page covers, "Summary"):
 *     TILE = 16 tokens, 1024 bytes.  With r = t % 16 and subvector j (0..63,
 *     channels 2j, 2j+1):
 *       K: byte 1024*(t/16) + 512*(r/8) + 16*(4*(r%8) + j%4) + 2*(j/8) + (j/4)%2
 *       V: byte 1024*(t/16) + 512*(j/32) + 16*(4*(j%8) + (r%8)/2) + 4*((j/8)%4)
 *            + 2*(r/8) + r%2
 *   VQKV_MODE_VQ3 (4096 entries x 4 dims, 12-bit codes, 32 codes per token;
 *   the same 1.25-4 bit range): the codes of subvectors p and p+16 (p =
 *   0..15, channels 4p..4p+3 and 4p+64..4p+67) form a pair stored in 3 bytes
 *   as in VQ15.  TILE = 16 tokens, 768 bytes: 32 lanes' 24-byte runs, run
 *   bytes 0..15 of lane L at 16*L and bytes 16..23 at 512 + 8*L.  With
 *   r = t % 16, byte k (0..2) of pair p of token t is run byte n of lane L:
 *       K: L = 4*(r%8) + p%4,      n = 12*(r/8) + 3*(p/4) + k
 *       V: L = 4*(p%8) + (r%8)/2,  n = 6*(2*(r/8) + r%2) + 3*(p/8) + k
 *   VQKV_MODE_VQ125 (1024 entries x 8 dims, 10-bit codes, 16 codes per
 *   token; the low end of the same range): TILE = 16 tokens, 320 bytes, a
 *   set of runs stored in two planes (plane 0 from byte 0, plane 1 from byte
 *   256).  Run bits are numbered from the least significant bit of the run's
 *   first byte; a code's bit b (LSB first) of subvector j (channels
 *   8j..8j+7) of token t, r = t % 16, is run bit B of run L / R:
 *       K: 32 runs of 10 bytes (8 at 8*L, 2 at 256 + 2*L),
 *          L = 4*(r%8) + j%4,        B = 40*(r/8) + 10*(j/4) + b
 *       V: 16 runs of 20 bytes (16 at 16*R, 4 at 256 + 4*R),
 *          R = 4*((j%8)/2) + (r%8)/2, B = 40*(2*(r/8) + r%2) + 10*(j%2 + 2*(j/8)) + b
 *     and run byte n = B/8 lies at the plane-0 offset + n while n is below
 *     the plane-0 length, else at the plane-1 offset + n - (plane-0 length).
 *   All five layouts are token-local: writing token t changes no byte of any
 *   other token.  Bits per element: 512*8/(16*128) = 2, 1536*8/(64*128) = 1.5,
 *   1024*8/(16*128) = 4, 768*8/(16*128) = 3 and 320*8/(16*128) = 1.25.
 *   (The layouts place, for each of the 32 lanes of a warp, the codes that
 *   lane needs for its tensor-core fragments in one contiguous 16-byte (VQ2)
 *   or 48-byte (VQ15) run, in two 16-byte runs 512 bytes apart (VQ4), or in
 *   a 16-byte and an 8-byte run (VQ3), so a warp reads a tile with
 *   coalesced 128-bit (and 64-bit) loads; VQ125 V runs are each read by the
 *   two lanes that share their four tokens.)
 */
#ifndef VQKV_H
#define VQKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VQKV_OK = 0,
  VQKV_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size, a misaligned pointer */
  VQKV_ERR_UNSUPPORTED = 2,   /* head_dim != 128, GQA group above 8, unknown mode */
  VQKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
  VQKV_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  VQKV_ERR_NO_DEVICE = 5      /* no usable CUDA device / device query failed */
} vqkv_status;

typedef enum {
  VQKV_MODE_VQ2 = 0,   /* 2 bit:   2^8 entries x 4 dims, 8-bit codes  */
  VQKV_MODE_VQ15 = 1,  /* 1.5 bit: 2^12 entries x 8 dims, 12-bit codes */
  VQKV_MODE_VQ4 = 2,   /* 4 bit:   2^8 entries x 2 dims, 8-bit codes */
  VQKV_MODE_VQ3 = 3,   /* 3 bit:   2^12 entries x 4 dims, 12-bit codes */
  VQKV_MODE_VQ125 = 4  /* 1.25 bit: 2^10 entries x 8 dims, 10-bit codes */
} vqkv_mode;

typedef enum {
  VQKV_ROLE_K = 0,     /* keys: x' = (x / s) . Hn before the search       */
  VQKV_ROLE_V = 1      /* values: quantised as they are                   */
} vqkv_role;

/* Bits of the device error word (see error_flags / workspace word 0). */
#define VQKV_DEVERR_SEQ_LEN   0x1u  /* a seq_lens[b] outside [0, max_seq_len]: clamped */
#define VQKV_DEVERR_POSITION  0x2u  /* an encode row outside [0, cap_len): not written */
#define VQKV_DEVERR_TIMEOUT   0x4u  /* a bounded on-chip wait gave up: see below */
#define VQKV_DEVERR_BLOCK     0x8u  /* a block-table entry outside [0, num_blocks) (paged calls) */
/*
 * VQKV_DEVERR_TIMEOUT: every on-chip wait of the decode kernels (the bulk
 * copies of the 2-bit code ring) gives up after a bounded number of polls
 * instead of hanging.  The CTA then waits, again bounded, for the copies it
 * still has in flight, sets this bit and finishes.  After it is set, the
 * launch's output O (and the shared memory of that CTA, which a late copy
 * may still write) are undefined.  A wait runs out only when a copy did not
 * complete in about 10^6 polls, which points at a fault outside the
 * library: treat the context as suspect, and do not trust later results on
 * it without checking them.
 */

/*
 * vqkv_encode — smoothing, Hadamard rotation, nearest-centroid assignment and
 * packing of new K or V rows (paper summary page, "Summary": channel-wise
 * smoothing followed by a Hadamard rotation of the keys, K-Means codebook;
 * arXiv summary page, "方法详解", stages 1-2).
 *
 * For row n (0 <= n < n_rows) of sequence b and KV head h:
 *   role K: y = x / s[h] (per channel), x' = y . Hn with Hn = H/sqrt(128),
 *           H[i][k] = (-1)^popcount(i & k), x' rounded to fp32 (computed in
 *           pairs of fp32 to about 2^-44 of its terms first, so x' is the
 *           correctly rounded value unless the exact one lies within about
 *           2^-20 ulp of a rounding boundary; such a case can change a code
 *           only between candidates whose distances are near-ties);
 *   role V: x' = x.
 *   For each subvector j of x' (d_sub = 2, 4 or 8 channels) the code is
 *   argmin_c sum_i (x'_{j,i} - C[h][c][i])^2 over the KV head's codebook C,
 *   decided on fp32 distances with ties to the lowest index, and is written
 *   at cache position pos[b] + n of stream (b, h) in the layout above.
 */
typedef struct {
  int32_t mode;        /* vqkv_mode */
  int32_t role;        /* vqkv_role */
  int32_t B;           /* sequences, >= 0 (0: nothing to do) */
  int32_t Hkv;         /* KV heads, >= 1 */
  int32_t head_dim;    /* must be 128 */
  int32_t n_rows;      /* rows per (sequence, KV head) to encode, >= 0 */
  int32_t cap_len;     /* cache capacity in tokens, >= 1 */
  const uint16_t* x;          /* device fp16 [B][Hkv][n_rows][128], 8-byte aligned */
  const int32_t* pos;         /* device [B]: position of row 0 of each sequence */
  const float* s;             /* device fp32 [Hkv][128], > 0; role K only (NULL for V) */
  const uint16_t* codebook;   /* device fp16 [Hkv][E][d_sub], 16-byte aligned, finite */
  uint8_t* codes;             /* device [B][Hkv][vqkv_code_bytes(mode, cap_len)] */
  unsigned long long* near_tie_count; /* device, optional: += subvectors whose best and
                                         second-best fp32 distances differ by less than
                                         1e-6 relative */
  uint32_t* error_flags;      /* device, optional: VQKV_DEVERR_POSITION is or-ed in when a
                                 row's position is outside [0, cap_len) (row not written) */
} vqkv_encode_args;

/*
 * vqkv_decode_attn — single-query decode attention straight from the packed
 * cache (paper summary page, "Summary": dequantisation inside the attention
 * computation; arXiv summary page, "方法详解", stage 3; the query gets the
 * matching inverse transform so scores are unchanged).
 *
 * For sequence b and query head hq (KV head h = hq / (Hq / Hkv)):
 *   q' = (q ⊙ s[h]) . Hn,  score_t = softmax_scale * q' . K'_t,
 *   O = sum_t softmax(score)_t V_t over t < seq_lens[b],
 * where K'_t and V_t are the concatenated centroids of token t's codes.
 * fp32 accumulation, fp16 output; seq_lens[b] == 0 gives a zero row.
 * The sequence is split across CTAs (split-KV); the last CTA of each
 * (b, KV head) merges the partial softmax states and writes O.
 */
typedef struct {
  int32_t mode;          /* vqkv_mode */
  int32_t B;             /* sequences, >= 0 (0: nothing to do) */
  int32_t Hq;            /* query heads, multiple of Hkv, Hq/Hkv <= 8 */
  int32_t Hkv;           /* KV heads, >= 1 */
  int32_t head_dim;      /* must be 128 */
  int32_t cap_len;       /* cache capacity in tokens (stream size), >= 1 */
  int32_t max_seq_len;   /* upper bound of seq_lens, 0 <= max_seq_len <= cap_len */
  const uint16_t* q;          /* device fp16 [B][Hq][128], 8-byte aligned */
  const uint8_t* k_codes;     /* device [B][Hkv][vqkv_code_bytes], 16-byte aligned */
  const uint8_t* v_codes;     /* device [B][Hkv][vqkv_code_bytes], 16-byte aligned */
  const int32_t* seq_lens;    /* device [B] */
  const uint16_t* k_codebook; /* device fp16 [Hkv][E][d_sub], 16-byte aligned, finite */
  const uint16_t* v_codebook; /* device fp16 [Hkv][E][d_sub], 16-byte aligned, finite */
  const float* s;             /* device fp32 [Hkv][128] key smoothing factors, > 0 */
  float softmax_scale;   /* <= 0 selects 1/sqrt(head_dim) */
  int32_t num_splits;    /* CTAs per (sequence, KV head); 0 = planned automatically */
  void* workspace;       /* device, >= vqkv_decode_workspace_bytes(args), 256-byte aligned,
                            zero-filled before its first use; every completed call leaves
                            it ready for the next.  Word 0 (uint32) is the device error
                            word (VQKV_DEVERR_SEQ_LEN, VQKV_DEVERR_TIMEOUT; sticky, the
                            caller may clear it) */
  size_t workspace_bytes;
  uint16_t* out;         /* device fp16 [B][Hq][128] */
} vqkv_decode_args;

/* Bytes of one cache stream (one of K or V of one (sequence, KV head)):
 * ceil(cap_len / TILE) * tile bytes; 0 for an unknown mode or cap_len < 0. */
size_t vqkv_code_bytes(int32_t mode, int32_t cap_len);

/* Workspace bytes vqkv_decode_attn needs for these arguments (the same split
 * plan the call will use on the current device).  Only the sizes are read
 * (mode, B, Hq, Hkv, head_dim, cap_len, max_seq_len, num_splits); pointers
 * are ignored.  0 when a size is invalid or no device is usable. */
size_t vqkv_decode_workspace_bytes(const vqkv_decode_args* args);

/* CTAs per (sequence, KV head) vqkv_decode_attn will use on the current
 * device (for the caller's bookkeeping).  Reads the sizes only, like
 * vqkv_decode_workspace_bytes; -1 when a size is invalid or no device is
 * usable. */
int32_t vqkv_decode_num_splits(const vqkv_decode_args* args);

/* Kernels one vqkv_decode_attn call with these arguments enqueues on the
 * current device: 1, or 2 when the plan merges the split partials in a
 * second kernel (CTAs that cover several sequences).  Reads the sizes only;
 * 0 for B == 0, -1 when a size is invalid or no device is usable. */
int32_t vqkv_decode_kernel_count(const vqkv_decode_args* args);

vqkv_status vqkv_encode(const vqkv_encode_args* args, void* stream);
vqkv_status vqkv_decode_attn(const vqkv_decode_args* args, void* stream);

/*
 * vqkv_decode_append — one decode step of the path in one call: the encode
 * of the step's new K and V rows (as vqkv_encode) fused into the decode
 * attention that reads them (as vqkv_decode_attn).
 *
 * For every sequence b with L = seq_lens[b] > 0 (clamped to max_seq_len as
 * in vqkv_decode_attn), k_new[b][h] and v_new[b][h] are encoded exactly as
 * vqkv_encode with n_rows = 1 and pos[b] = L - 1 would encode them, and their
 * codes are written at position L - 1 of the K and V streams of
 * decode.k_codes / decode.v_codes (which this call therefore writes, despite
 * their const type).  O is then what vqkv_decode_attn returns for the same
 * arguments over the L tokens including the new one.  Inside the kernel the
 * CTA that holds position L - 1 writes the new codes before it starts
 * streaming that tile, so one kernel does the whole step.  Workspace, error
 * word, alignment and failure rules are those of vqkv_decode_attn.  2-bit and
 * 4-bit modes (VQKV_ERR_UNSUPPORTED for the 1.5-, 3- and 1.25-bit modes,
 * whose multi-byte codes the in-kernel encode does not write).
 */
typedef struct {
  vqkv_decode_args decode;    /* as for vqkv_decode_attn (seq_lens include the new token) */
  const uint16_t* k_new;      /* device fp16 [B][Hkv][128], 8-byte aligned: new key rows */
  const uint16_t* v_new;      /* device fp16 [B][Hkv][128], 8-byte aligned: new value rows */
  unsigned long long* near_tie_count; /* device, optional: as in vqkv_encode_args, for both rows */
} vqkv_decode_append_args;

vqkv_status vqkv_decode_append(const vqkv_decode_append_args* args, void* stream);

/*
 * vqkv_decode_attn_multi — several queries per sequence over the packed
 * cache: the M = n_queries newest tokens of each sequence attend at once
 * (chunked prefill or speculative decoding on a VQ cache; attention over
 * the dequantised cache, paper summary page, "Summary").
 *
 * decode.q and decode.out are fp16 [B][M][Hq][128].  Query m of sequence b
 * is the token at position L - M + m (L = seq_lens[b], clamped as in
 * vqkv_decode_attn) and attends causally: it sees the cached tokens
 * t <= L - M + m, and is a zero row when it sees none.  The M x (Hq / Hkv)
 * queries of a KV head are its softmax columns; each group of up to 8
 * columns shares every code it reads (one CTA per group and token range).
 * M * (Hq / Hkv) <= 64 (VQKV_ERR_UNSUPPORTED otherwise).  The workspace must hold
 * n_queries * vqkv_decode_workspace_bytes(&args->decode) bytes; everything
 * else is as in vqkv_decode_attn, which is this call with n_queries = 1.
 */
typedef struct {
  vqkv_decode_args decode;  /* q, out: [B][n_queries][Hq][128] */
  int32_t n_queries;        /* M >= 1 */
} vqkv_decode_multi_args;

vqkv_status vqkv_decode_attn_multi(const vqkv_decode_multi_args* args, void* stream);

/*
 * Paged cache: one pool of fixed-size blocks per role, shared by all
 * sequences through a block table, as serving engines lay out their KV
 * caches (the pages name serving-framework integration as future work,
 * paper summary page, "Key points").
 *
 * In the paged calls, codes (encode) and k_codes / v_codes (decode) point to
 * pools of num_blocks * Hkv * vqkv_code_bytes(mode, block_tokens) bytes:
 * block n of KV head h starts at byte (n * Hkv + h) * vqkv_code_bytes(mode,
 * block_tokens) and holds block_tokens tokens in the layout above (a stream
 * of block_tokens tokens).  Logical token t of sequence b lives at position
 * t % block_tokens of block block_table[b * max_blocks + t / block_tokens].
 * cap_len must not exceed max_blocks * block_tokens.  A table entry outside
 * [0, num_blocks) is never dereferenced: the encode skips that row, the
 * decode reads block 0 instead (its O is then meaningless), and both set
 * VQKV_DEVERR_BLOCK in the error word.  Everything else is as in the
 * contiguous calls, which give the same results for the same tokens.
 */
typedef struct {
  const int32_t* block_table; /* device [B][max_blocks], 4-byte aligned */
  int32_t max_blocks;         /* entries per sequence, >= 1 */
  int32_t block_tokens;       /* tokens per block: a power of two, >= 64 */
  int32_t num_blocks;         /* blocks in each pool, >= 1 */
} vqkv_paging;

vqkv_status vqkv_encode_paged(const vqkv_encode_args* args, const vqkv_paging* paging, void* stream);
vqkv_status vqkv_decode_attn_paged(const vqkv_decode_args* args, const vqkv_paging* paging, void* stream);

/*
 * vqkv_decode_attn_fp16 — the same decode attention over a plain fp16 KV
 * cache, the comparison point for the quantised path on the same shapes
 * (the paper measures its speed-up against FP16 attention, summary page,
 * "Key points"):  O = softmax(softmax_scale * q . K_t^T) . V_t, t < seq_lens[b],
 * no smoothing, no rotation, no codebooks.  Same split-KV plan, GQA grouping
 * and workspace rules as vqkv_decode_attn (vqkv_fp16_decode_workspace_bytes
 * gives the size).
 */
typedef struct {
  int32_t B, Hq, Hkv, head_dim, cap_len, max_seq_len;
  const uint16_t* q;          /* device fp16 [B][Hq][128], 4-byte aligned */
  const uint16_t* k;          /* device fp16 [B][Hkv][cap_len][128], 16-byte aligned */
  const uint16_t* v;          /* device fp16 [B][Hkv][cap_len][128], 16-byte aligned */
  const int32_t* seq_lens;    /* device [B] */
  float softmax_scale;        /* <= 0 selects 1/sqrt(head_dim) */
  int32_t num_splits;         /* 0 = planned automatically */
  void* workspace;            /* as for vqkv_decode_attn */
  size_t workspace_bytes;
  uint16_t* out;              /* device fp16 [B][Hq][128] */
} vqkv_fp16_decode_args;

size_t vqkv_fp16_decode_workspace_bytes(const vqkv_fp16_decode_args* args);
vqkv_status vqkv_decode_attn_fp16(const vqkv_fp16_decode_args* args, void* stream);

/* Size of the scratch array compiled into the library for
 * vqkv_decode_attn_static (8 MiB, held on every GPU that loads the library
 * until the process exits). */
#define VQKV_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * vqkv_decode_attn_static — vqkv_decode_attn for callers that cannot
 * allocate device memory.  The paper has no counterpart: this is a
 * deployment variant of this library, not a step of the method.
 *
 * Some callers cannot obtain a workspace: a serving engine whose memory pool
 * has reserved all device memory up front and forbids allocation after
 * start-up, a plugin whose host framework owns every allocation and offers
 * no scratch buffer in its interface, or code that must not call cudaMalloc
 * on its hot path.  This entry point computes exactly what vqkv_decode_attn
 * computes (same kernels, same split plan) but keeps the split-KV scratch in
 * a fixed array of VQKV_STATIC_SCRATCH_BYTES inside the library, so it
 * allocates nothing and calls no allocating routine; the caller still
 * passes every input and the output.  args->workspace and
 * args->workspace_bytes are ignored.
 *
 *   - Arguments are checked exactly as in vqkv_decode_attn.  When the split
 *     plan needs more scratch than VQKV_STATIC_SCRATCH_BYTES
 *     (vqkv_decode_workspace_bytes(args) tells how much), the call returns
 *     VQKV_ERR_WORKSPACE and enqueues nothing.
 *   - Every call looks up the array's device address in the current
 *     device's context (cudaGetSymbolAddress, which allocates nothing), so
 *     the address stays right after a context is torn down and rebuilt.  The
 *     first call in a context may load the library's device code into it:
 *     make that first call before any stream capture.
 *   - Each call clears the scratch's error word and tickets with
 *     cudaMemsetAsync on `stream`, then launches.  The array is shared by
 *     every call on a device and keeps the last call's contents: calls whose
 *     execution overlaps on the GPU (different streams, not ordered) race on
 *     it and must be serialised by the caller.  The device error bits of the
 *     last call (VQKV_DEVERR_SEQ_LEN, VQKV_DEVERR_TIMEOUT) stay in the
 *     scratch's error word until the next call clears it:
 *     vqkv_decode_static_error reads them.
 */
vqkv_status vqkv_decode_attn_static(const vqkv_decode_args* args, void* stream);

/*
 * vqkv_decode_static_error — the device error word of the last
 * vqkv_decode_attn_static call on the current device (VQKV_DEVERR_* bits,
 * 0 when none was raised).  Enqueues a 4-byte copy from the scratch array to
 * *host_flags (host memory, pageable or pinned) on `stream` after the work
 * already queued there, then waits for `stream`; allocates nothing.  Call it
 * on the stream of the decode call it should observe.  Returns
 * VQKV_ERR_INVALID_ARG for a NULL host_flags, VQKV_ERR_CUDA when the copy or
 * the wait fails.
 */
vqkv_status vqkv_decode_static_error(uint32_t* host_flags, void* stream);

/*
 * vqkv_test_decode_ring_timeout — test hook for the bounded on-chip waits of
 * the 2-bit decode (not for production use).  It runs vqkv_decode_attn, but
 * every warp withholds the first bulk copy of its code ring, and every wait
 * gives up after max_polls polls (1..4096).  So each ring wait runs out.
 * The call must set VQKV_DEVERR_TIMEOUT in the workspace error word and
 * complete normally. O is then meaningless, and later calls on the same
 * context work as usual.  2-bit mode only.
 */
vqkv_status vqkv_test_decode_ring_timeout(const vqkv_decode_args* args, uint32_t max_polls, void* stream);

/* ------------------------------------------------------------------------
 * Offline calibration: the key smoothing vector, the key transform variants
 * and K-Means codebook training.  These produce the s and codebook inputs of
 * the calls above; they are not part of a decode step.  VecInfer trains its
 * codebooks offline with K-Means on the smoothed, rotated key subvectors
 * (and on raw value subvectors) (paper summary page, "Summary"), and its
 * ablation compares smoothing, the rotation, both, and their order ("Key
 * points").  Readings where the pages are silent: s_c = sqrt(max_t |K[t][c]|)
 * with 0 -> 1; K-Means is Lloyd's algorithm seeded by k-means++ (Arthur and
 * Vassilvitskii), with the random draws passed in.
 * ------------------------------------------------------------------------ */

/*
 * vqkv_smoothing — s[c] = sqrt(max over the n_rows rows of |rows[t][c]|),
 * correctly rounded fp32, and 1 where that maximum is 0, for the 128
 * channels.  rows: device [n_rows][128], fp16 (dtype 0) or fp32 (dtype 1),
 * 16-byte aligned; s: device fp32 [128], 16-byte aligned, written only by
 * this call (it is also the call's scratch).  n_rows >= 0 (0 gives all 1).
 * Errors: VQKV_ERR_INVALID_ARG for a NULL or misaligned pointer, a negative
 * n_rows or another dtype.
 */
vqkv_status vqkv_smoothing(const void* rows, int32_t dtype, int64_t n_rows, float* s, void* stream);

/*
 * vqkv_calib_transform — out[t] = R(x[t] / s_pre) / s_post for the n_rows
 * rows of 128 channels: R is the normalised Hadamard rotation x . Hn (Hn =
 * H / sqrt(128), H[i][k] = (-1)^popcount(i & k)) when rotate is nonzero,
 * else the identity; s_pre / s_post (device fp32 [128]) may each be NULL
 * (no division).  fp32 arithmetic (one rounding per division, a fast
 * Walsh-Hadamard transform for R).  x: device [n_rows][128] fp16 (dtype 0)
 * or fp32 (dtype 1); out: device fp32 [n_rows][128] (may equal x when
 * dtype is 1).  All pointers 16-byte aligned.  The variants of the
 * ablation: none (no s, no R), smooth (s_pre), Hadamard (R), both (s_pre,
 * R: the decode path's key transform), rotate-then-smooth (R, then s_post =
 * vqkv_smoothing of the rotated rows).
 */
vqkv_status vqkv_calib_transform(const void* x, int32_t dtype, int64_t n_rows, const float* s_pre,
                                 int32_t rotate, const float* s_post, float* out, void* stream);

/*
 * K-Means on n points of dim (2, 4 or 8) fp32 coordinates into k centroids.
 *   - Seeding (k-means++): centre 0 is point floor(u[0] * n); centre i is the
 *     first point (index order) whose running sum of D^2 exceeds
 *     u[i] * sum D^2, D(x) the distance of x to its nearest chosen centre
 *     (floor(u[i] * n) when every D^2 is 0).  D^2 is fp32 (the assignment's
 *     arithmetic), the sums fp64.
 *   - Assignment: nearest centroid by fp32 squared distance from direct
 *     differences; ties go to the lowest index.
 *   - Update: each centroid becomes the fp64 mean of its points rounded to
 *     fp32; an empty cluster keeps its centroid.  Every step is
 *     deterministic: the same inputs give the same bits on every run.
 *   - vqkv_kmeans runs the seeding, then `iters` (assignment, update) steps,
 *     and writes the fp32 centroids and, if requested, their fp16 rounding.
 */
typedef struct {
  int32_t n;               /* points, >= 1 */
  int32_t dim;             /* 2, 4 or 8 */
  int32_t k;               /* centroids, 1 <= k <= min(n, 4096) */
  int32_t iters;           /* Lloyd steps, 0..1000 */
  const float* points;     /* device fp32 [n][dim], 16-byte aligned */
  const float* uniforms;   /* device fp32 [k], draws in [0, 1) */
  float* centroids;        /* device fp32 [k][dim] out, 16-byte aligned */
  uint16_t* codebook;      /* device fp16 [k][dim] out, or NULL */
  int32_t* seeds;          /* device int32 [k] out: the seeding's picks, or NULL */
  int32_t* assign;         /* device int32 [n] out: the last step's assignment (made
                              before the last update), or NULL; untouched when iters = 0 */
  void* workspace;         /* device, >= vqkv_kmeans_workspace_bytes, 256-byte aligned */
  size_t workspace_bytes;
} vqkv_kmeans_args;

/* Workspace of vqkv_kmeans (0 for invalid sizes). */
size_t vqkv_kmeans_workspace_bytes(const vqkv_kmeans_args* args);

/* The whole training.  Errors: VQKV_ERR_INVALID_ARG (sizes, NULL or
 * misaligned pointers), VQKV_ERR_WORKSPACE, VQKV_ERR_CUDA. */
vqkv_status vqkv_kmeans(const vqkv_kmeans_args* args, void* stream);

/* The seeding alone: writes args->seeds (required here) and sets
 * args->centroids to the picked points.  Uses the workspace like
 * vqkv_kmeans; args->iters, codebook and assign are ignored. */
vqkv_status vqkv_kmeans_seed(const vqkv_kmeans_args* args, void* stream);

/* One assignment: assign[i] = nearest centroid of point i (int32), and, if
 * dist is not NULL, its fp32 squared distance.  points / centroids 16-byte
 * aligned; 1 <= k <= 4096; n >= 0. */
vqkv_status vqkv_kmeans_assign(const float* points, int32_t n, int32_t dim, const float* centroids, int32_t k,
                               int32_t* assign, float* dist, void* stream);

/* One update: c_out[c] = fp64 mean of the points with assign == c rounded to
 * fp32, c_in[c] when there is none.  Assignments outside [0, k) count for no
 * centroid.  c_out must not overlap c_in.  The points are brought into
 * cluster order by a stable counting sort in the workspace (device, 256-byte
 * aligned, >= vqkv_kmeans_update_workspace_bytes(n, k); 0 for invalid
 * sizes), and each cluster is summed in point order: the result does not
 * depend on scheduling. */
size_t vqkv_kmeans_update_workspace_bytes(int32_t n, int32_t k);
vqkv_status vqkv_kmeans_update(const float* points, int32_t n, int32_t dim, const int32_t* assign, int32_t k,
                               const float* c_in, float* c_out, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Static, never NULL. */
const char* vqkv_status_string(vqkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* VQKV_H */
