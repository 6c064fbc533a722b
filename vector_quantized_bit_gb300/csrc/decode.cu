// Fused VQ decode attention for sm_103a.
//
// One CTA handles one KV head, one token range ("split") of each sequence
// in its group, and all g query heads of that KV head, so every code byte
// is read from HBM once per KV head (GQA grouping).  Per 16-token tile a
// warp computes
//   scores  S[t][h] = sum_d K'[t][d] q'[h][d]      (tensor cores, K' gathered
//                                                  from the smem codebook)
//   online softmax over t                         (exp2; q' carries
//                                                  scale*log2(e))
//   O[d][h] += sum_t V[t][d] P[t][h]              (tensor cores, V gathered
//                                                  from the smem codebook)
// Dequantisation happens only in registers: the cache layout puts each
// lane's codes for its MMA fragments in one run (16 bytes at 2 bit, two
// 16-byte planes at 4 bit, 16 + 8 bytes at 3 bit, 8 + 2 bytes of K and a
// 16 + 4-byte V run shared by two lanes at 1.25 bit, 48 bytes at 1.5 bit).
// The 2-, 3-, 4- and 1.25-bit codes reach shared memory through a per-warp
// ring of TMA bulk copies (the tile-ring kernel, decode_vq2_kernel); the
// 1.5-bit codes reach a per-lane shared-memory slot through cp.async;
// centroids are gathered from shared memory.
//
// The per-query transform is q' = (q * s) . Hn, so q'.K'^T = q.K^T
// (VecInfer paper summary page, "Summary": matching inverse operations on
// the queries keep attention scores unchanged).  Split partials (m, l, O)
// are merged by the last CTA of each (sequence, KV head), chosen with an
// atomic ticket (no waiting), or, when a CTA covers several sequences, by a
// small combine kernel launched right after the decode kernel.
//
// Fragment maps (mma.m16n8k16, lane = 4*gid + tig):
//   score MMA  A = K' tile: rows = tokens {gid, gid+8}, k = the 4 channels of
//              one subvector (VQ2, VQ3: j = 4s+tig at k-step s; VQ15, VQ125:
//              half of subvector j = 4s'+tig at k-steps 2s', 2s'+1; VQ4: two
//              2-channel subvectors), so one 8/16-byte centroid load fills
//              a0a1|a4a5 (token gid) or a2a3|a6a7;
//              B = q' (k = channels, n = heads, columns >= g are zero);
//              D: tokens {gid, gid+8} x heads {2tig, 2tig+1}.
//   P          D -> fp16 -> movmatrix.trans -> B operand of the P.V MMA
//              (k = tokens {2tig, 2tig+1, 2tig+8, 2tig+9}, n = head gid).
//   P.V MMA    A = V^T: rows = channels of subvector J (VQ2, VQ3: J = 8p+gid
//              over M-tiles 2p, 2p+1; VQ15, VQ125: J = 8p+gid over M-tiles
//              4p..4p+3; VQ4: J = 8p+gid in M-tile p),
//              k = the four tokens above; centroid halves are paired across
//              tokens with byte permutes.
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "encode_common.cuh"
#include "internal.h"

namespace vqkv {
namespace {

// ------------------------------------------------------------------ tile ring (VQ2, VQ4, VQ3, VQ125)
#ifndef VQKV_V2_WARPS
#define VQKV_V2_WARPS 16
#endif
#ifndef VQKV_V2_TPI
#define VQKV_V2_TPI 3
#endif
#ifndef VQKV_V2_STAGES
#define VQKV_V2_STAGES 2
#endif
constexpr int V2_WARPS = VQKV_V2_WARPS;             // one CTA per SM
constexpr int V2_TPI = VQKV_V2_TPI;                 // 16-token tiles per step (a "super-tile")
constexpr int V2_THREADS = V2_WARPS * 32;
constexpr int V2_TILE = 16;
// q' rows (fp32, 128 channels) at a pitch that keeps the 8 lanes of each
// quarter-warp on distinct 16-byte bank groups when the MMA fragments are
// read (lane (gid, tig) reads 4 floats at gid * pitch + 4 tig + 16 s).
constexpr int V2_Q_PITCH = 144;
constexpr int V2_STAGES = VQKV_V2_STAGES;           // per-warp ring of super-tiles (K then V)

// Geometry of the tile-ring decode, per code mode: 2 bit (256 x 4, one byte
// per code), 4 bit (256 x 2, one byte per code), 3 bit (4096 x 4, 12-bit
// codes in 3-byte pairs) and 1.25 bit (1024 x 8, 10-bit codes).  Shared
// memory starts with the codebooks (64 KB: the 256-entry ones replicated
// across banks, the 4096-entry ones once; 128 KB: the 1024-entry ones in
// four interleaved copies), then q'.  A lane's code words of a tile: 2 bit
// one 16-byte word; 4 bit two 16-byte words in planes 512 bytes apart; 3 bit
// a 16-byte and an 8-byte word (planes at 0 and 512); 1.25 bit: K an 8-byte
// and a 2-byte word, V a 16-byte and a 4-byte word (planes at 0 and 256).
template <int MODE>
struct V2Geo {
  static constexpr bool PAIRS = MODE == VQKV_MODE_VQ3;          // 12-bit codes in 3-byte pairs
  static constexpr bool TEN = MODE == VQKV_MODE_VQ125;          // 10-bit codes in bit runs
  static constexpr int DSUB = MODE == VQKV_MODE_VQ4 ? 2 : TEN ? 8 : 4;
  static constexpr int TILE_BYTES = PAIRS ? 768 : TEN ? 320 : 16 * (kHeadDim / DSUB);
  static constexpr int LW = TILE_BYTES / 32 / 4;                  // byte and pair codes: a lane's 32-bit words
  static constexpr int KW = TEN ? 3 : LW, VW = TEN ? 5 : LW;      // words a lane reads per tile, K and V
  static constexpr int TPI = MODE == VQKV_MODE_VQ4 ? 2 : V2_TPI;  // tiles per step
  static constexpr int STAGE_BYTES = 2 * TPI * TILE_BYTES;
  static constexpr int CB_BYTES = TEN ? 2 * 65536 : 65536;
  static constexpr int Q_OFF = CB_BYTES;                          // q' (fp32 [8][V2_Q_PITCH])
  static constexpr int RING_OFF = Q_OFF + 8 * V2_Q_PITCH * 4;
  static constexpr int MBAR_OFF = RING_OFF + V2_WARPS * V2_STAGES * STAGE_BYTES;
  static constexpr int REPL = PAIRS ? 1 : TEN ? 4 : 128 / (2 * DSUB);   // codebook copies (byte codes use it)
};

// ------------------------------------------------------------------ VQ15
constexpr int V15_WARPS = 16;
constexpr int V15_THREADS = V15_WARPS * 32;
constexpr int V15_TILE = 64;
constexpr int V15_TILE_BYTES = 1536;
constexpr int V15_CB_BYTES = 4096 * 16;          // 64 KB per codebook
// Per-lane code slot: the lane's 48 key-code bytes and 48 value-code bytes
// of the next tile, copied with cp.async one tile ahead (each lane copies
// and reads only its own bytes).
constexpr int V15_SLOT_OFF = 2 * V15_CB_BYTES;
constexpr int V15_SLOT_BYTES = V15_THREADS * 96;  // 48 KB
constexpr int V15_Q_OFF = V15_SLOT_OFF + V15_SLOT_BYTES;
constexpr int V15_Q_PITCH = 128;   // read once per sequence; a padded pitch measured no better

// Codebooks, q', code ring, ring barriers; the combine area reuses the
// codebook, q' and ring region after the tile loop.
// Fused append (vqkv_decode_append): per-warp partial searches.
constexpr int V2_APP_BYTES = V2_WARPS * 32 * (int)sizeof(Best);
// Paged cache: the block ids of the CTA's token range, read once per sequence.
constexpr int V2_BLK_CACHE = 512;
// Flat plan (batches): per-sequence super-tile prefix sums, B <= kFlatMaxB.
template <int MODE>
struct V2Smem {
  static constexpr int APP_OFF = (V2Geo<MODE>::MBAR_OFF + V2_WARPS * V2_STAGES * 8 + 15) / 16 * 16;
  static constexpr int BLK_OFF = APP_OFF + V2_APP_BYTES;
  static constexpr int FLAT_OFF = BLK_OFF + V2_BLK_CACHE * 4;
  static constexpr size_t BYTES = FLAT_OFF + (kFlatMaxB + 1 + 4) * 4;   // + T, S_eff, share bounds
};
constexpr size_t kV2Smem = V2Smem<VQKV_MODE_VQ2>::BYTES;
constexpr size_t kV4Smem = V2Smem<VQKV_MODE_VQ4>::BYTES;
constexpr size_t kV3Smem = V2Smem<VQKV_MODE_VQ3>::BYTES;
constexpr size_t kV125Smem = V2Smem<VQKV_MODE_VQ125>::BYTES;
static_assert(kV4Smem <= 227 * 1024 && kV3Smem <= 227 * 1024 && kV125Smem <= 227 * 1024,
              "4-bit / 3-bit / 1.25-bit decode shared memory");
static_assert(CombineSmem<V2_WARPS>::kBytes <= V2Geo<VQKV_MODE_VQ2>::MBAR_OFF,
              "combine area must fit below the ring barriers");
// The combine area (after the tile loop) and q' (before it) overlap the
// code slots, which are idle at those times.
constexpr size_t kV15Smem = 2 * V15_CB_BYTES + CombineSmem<V15_WARPS>::kBytes;
static_assert(V15_Q_OFF + 8 * V15_Q_PITCH * 4 <= (int)kV15Smem, "q' must fit in the combine area");

// The lane's 4 channels of query column col0 + warp (query c / g, head
// c % g) and their smoothing factors, for warps 0..nloc-1.
struct QueryLoad {
  uint2 q;
  float4 s;
};
__device__ __forceinline__ QueryLoad load_query(const DecodeParams& p, int b, int kvh, int warp, int lane, int col0,
                                                int nloc) {
  QueryLoad r{make_uint2(0u, 0u), make_float4(0.f, 0.f, 0.f, 0.f)};
  if (warp < nloc) {
    const int c = col0 + warp;
    const int m = c / p.g, hq = kvh * p.g + c - m * p.g;
    r.q = *reinterpret_cast<const uint2*>(p.q + (((size_t)b * p.M + m) * p.Hq + hq) * kHeadDim + 4 * lane);
    r.s = *reinterpret_cast<const float4*>(p.s + (size_t)kvh * kHeadDim + 4 * lane);
  }
  return r;
}

// q' of the CTA's softmax column col0 + warp into row `warp` of s_qp (fp32,
// scaled, rows `pitch` floats apart), by warps 0..nloc-1.
__device__ __forceinline__ void transform_query(const DecodeParams& p, const QueryLoad& r, int warp, int lane,
                                                float* s_qp, int pitch, int nloc) {
  if (warp < nloc) {
    const __half2 q01 = *reinterpret_cast<const __half2*>(&r.q.x);
    const __half2 q23 = *reinterpret_cast<const __half2*>(&r.q.y);
    float v[4] = {__low2float(q01) * r.s.x, __high2float(q01) * r.s.y, __low2float(q23) * r.s.z,
                  __high2float(q23) * r.s.w};
    fwht128_f32(v, lane);
    float4 o = make_float4(v[0] * p.qscale, v[1] * p.qscale, v[2] * p.qscale, v[3] * p.qscale);
    *reinterpret_cast<float4*>(s_qp + warp * pitch + 4 * lane) = o;
  }
}

__device__ __forceinline__ void transform_queries(const DecodeParams& p, int b, int kvh, int warp,
                                                  int lane, float* s_qp, int pitch, int col0, int nloc) {
  transform_query(p, load_query(p, b, kvh, warp, lane, col0, nloc), warp, lane, s_qp, pitch, nloc);
}

// Shared-memory offset of a gathered centroid: one byte permute puts code
// byte K of `codes` into bits 8..15 and the lane's replica offset (byte 0 of
// `lane_byte`) into bits 0..7: (code << 8) | replica offset.
template <int K>
__device__ __forceinline__ uint32_t cb_offset(uint32_t codes, uint32_t lane_byte) {
  return __byte_perm(codes, lane_byte, 0x5504 | (K << 4));
}

template <typename T>
__device__ __forceinline__ T lds_at(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const T*>(base + off);
}

// 24-bit code pair at byte b (a multiple of 3) of a lane's run of words.
template <int LW>
__device__ __forceinline__ uint32_t pair_at(const uint32_t (&w)[LW], int b) {
  const int i = b >> 2, sh = (b & 3) * 8;
  return (sh <= 8 ? (w[i] >> sh) : __funnelshift_r(w[i], w[i + 1], sh)) & 0xffffffu;
}

// One step of the tile-ring decode over T consecutive 16-token tiles.
//
// Scores: tokens are the MMA rows, heads the 8 columns; B is q' (qa).
//   2 bit: the A operand of k-step s is two 8-byte centroid gathers (tokens
//     gid and gid+8, channels 4j..4j+3 of subvector j = 4s+tig); kw[i]:
//     this lane's 16 key-code bytes (tokens gid, gid+8 x subvectors 4s+tig).
//   3 bit: the same gathers; kw[i]: the 3-byte pairs (j, j+16) of tokens gid
//     (bytes 0..11) and gid+8 (bytes 12..23) for j = tig, 4+tig, 8+tig,
//     12+tig, so subvector 4s+tig is pair s%4, low code for s < 4.
//   4 bit: four 4-byte gathers (tokens gid and gid+8 x subvectors 8s+tig and
//     8s+4+tig, i.e. channels 16s+k in k order); kw[i][0..3] / [4..7]:
//     tokens gid / gid+8, byte 2s / 2s+1 = subvector 8s+tig / 8s+4+tig.
// A 16-token tile takes 8 score MMAs.  movmatrix turns the scores into the
// P.V B operand.  P.V: A = gathered V centroids, channels x tokens (2tig,
// 2tig+1, 2tig+8, 2tig+9), paired by byte permutes: for subvector 8p+gid, the
// four tokens' codes are vw word p (2 and 4 bit), or pair (gid + 8(p%2))
// of each token's 6-byte slot, low code for p < 2 (3 bit); 2 and 3 bit:
// channels 4j..4j+3 over two M-tiles; 4 bit: channels 2j, 2j+1 in one.
// kbyte / vbyte: the lane's replica offset in the K / V half row (2 and 4
// bit), or the byte offset of the K / V codebook (3 bit).
// Softmax state m0/l0, m1/l1 belongs to heads 2tig, 2tig+1, the columns of
// this lane's O^T fragments.
template <int T, int MODE>
__device__ __forceinline__ void vq2_step(const unsigned char* s_cb, uint32_t kbyte, uint32_t vbyte,
                                         const uint32_t (&qa)[8][2], const uint32_t (&kw)[T][V2Geo<MODE>::KW],
                                         const uint32_t (&vw)[T][V2Geo<MODE>::VW], int tile0,
                                         const ColumnLimits& cl, int lane, float& m0, float& m1, float& l0, float& l1,
                                         float (&acc)[8][4]) {
  const int gid = lane >> 2;
  float sc[T][4];
#pragma unroll
  for (int i = 0; i < T; ++i) {
    float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (MODE == VQKV_MODE_VQ2) {
#define VQKV_SCORE_STEP(S, ACC)                                                                        \
  {                                                                                                    \
    const uint2 c = lds_at<uint2>(s_cb, cb_offset<(S)&3>((S) < 4 ? kw[i][0] : kw[i][1], kbyte));         \
    const uint2 d = lds_at<uint2>(s_cb, cb_offset<(S)&3>((S) < 4 ? kw[i][2] : kw[i][3], kbyte));         \
    mma_16816(ACC, c.x, d.x, c.y, d.y, qa[S][0], qa[S][1]);                                             \
  }
      VQKV_SCORE_STEP(0, da) VQKV_SCORE_STEP(1, db) VQKV_SCORE_STEP(2, da) VQKV_SCORE_STEP(3, db)
      VQKV_SCORE_STEP(4, da) VQKV_SCORE_STEP(5, db) VQKV_SCORE_STEP(6, da) VQKV_SCORE_STEP(7, db)
#undef VQKV_SCORE_STEP
    } else if constexpr (MODE == VQKV_MODE_VQ3) {
#pragma unroll
      for (int S = 0; S < 8; ++S) {
        const uint32_t pg = pair_at(kw[i], 3 * (S & 3)), ph = pair_at(kw[i], 12 + 3 * (S & 3));
        const uint32_t cg = S < 4 ? (pg & 0xfffu) : (pg >> 12), ch = S < 4 ? (ph & 0xfffu) : (ph >> 12);
        const uint2 c = lds_at<uint2>(s_cb, kbyte + (cg << 3));
        const uint2 d = lds_at<uint2>(s_cb, kbyte + (ch << 3));
        mma_16816((S & 1) ? db : da, c.x, d.x, c.y, d.y, qa[S][0], qa[S][1]);
      }
    } else {
#define VQKV_SCORE_STEP4(S, ACC)                                                          \
  {                                                                                       \
    const uint32_t wg = kw[i][(S) >> 1], wh = kw[i][4 + ((S) >> 1)];                      \
    const uint32_t ag = lds_at<uint32_t>(s_cb, cb_offset<((S)&1) * 2>(wg, kbyte));        \
    const uint32_t bg = lds_at<uint32_t>(s_cb, cb_offset<((S)&1) * 2 + 1>(wg, kbyte));    \
    const uint32_t ah = lds_at<uint32_t>(s_cb, cb_offset<((S)&1) * 2>(wh, kbyte));        \
    const uint32_t bh = lds_at<uint32_t>(s_cb, cb_offset<((S)&1) * 2 + 1>(wh, kbyte));    \
    mma_16816(ACC, ag, ah, bg, bh, qa[S][0], qa[S][1]);                                   \
  }
      VQKV_SCORE_STEP4(0, da) VQKV_SCORE_STEP4(1, db) VQKV_SCORE_STEP4(2, da) VQKV_SCORE_STEP4(3, db)
      VQKV_SCORE_STEP4(4, da) VQKV_SCORE_STEP4(5, db) VQKV_SCORE_STEP4(6, da) VQKV_SCORE_STEP4(7, db)
#undef VQKV_SCORE_STEP4
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[i][e] = da[e] + db[e];
  }
  if ((tile0 + T) * V2_TILE > cl.lim_min) {   // tail of the sequence
#pragma unroll
    for (int i = 0; i < T; ++i) mask_scores(sc[i], (tile0 + i) * V2_TILE + gid, cl);
  }
  uint32_t bP[T][2];
  softmax_tiles<T, 8>(sc, m0, m1, l0, l1, acc, bP);
#pragma unroll
  for (int i = 0; i < T; ++i) {
    if constexpr (MODE == VQKV_MODE_VQ4) {
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const uint32_t w = vw[i][pp];
        const uint32_t R0 = lds_at<uint32_t>(s_cb, cb_offset<0>(w, vbyte));
        const uint32_t R1 = lds_at<uint32_t>(s_cb, cb_offset<1>(w, vbyte));
        const uint32_t R2 = lds_at<uint32_t>(s_cb, cb_offset<2>(w, vbyte));
        const uint32_t R3 = lds_at<uint32_t>(s_cb, cb_offset<3>(w, vbyte));
        mma_16816(acc[pp], __byte_perm(R0, R1, 0x5410), __byte_perm(R0, R1, 0x7632), __byte_perm(R2, R3, 0x5410),
                  __byte_perm(R2, R3, 0x7632), bP[i][0], bP[i][1]);
      }
    } else {
#define VQKV_PV_PAIR(PP, R0, R1, R2, R3)                                                           \
  {                                                                                                \
    mma_16816(acc[2 * (PP)], __byte_perm(R0.x, R1.x, 0x5410), __byte_perm(R0.x, R1.x, 0x7632),     \
              __byte_perm(R2.x, R3.x, 0x5410), __byte_perm(R2.x, R3.x, 0x7632), bP[i][0], bP[i][1]); \
    mma_16816(acc[2 * (PP) + 1], __byte_perm(R0.y, R1.y, 0x5410), __byte_perm(R0.y, R1.y, 0x7632), \
              __byte_perm(R2.y, R3.y, 0x5410), __byte_perm(R2.y, R3.y, 0x7632), bP[i][0], bP[i][1]); \
  }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        if constexpr (MODE == VQKV_MODE_VQ2) {
          const uint32_t w = vw[i][pp];
          const uint2 R0 = lds_at<uint2>(s_cb, cb_offset<0>(w, vbyte));
          const uint2 R1 = lds_at<uint2>(s_cb, cb_offset<1>(w, vbyte));
          const uint2 R2 = lds_at<uint2>(s_cb, cb_offset<2>(w, vbyte));
          const uint2 R3 = lds_at<uint2>(s_cb, cb_offset<3>(w, vbyte));
          VQKV_PV_PAIR(pp, R0, R1, R2, R3)
        } else {
          auto code = [&](int k) {   // the code of slot k's token (pair byte 6k + 3(pp%2))
            const uint32_t pr = pair_at(vw[i], 6 * k + 3 * (pp & 1));
            return pp < 2 ? (pr & 0xfffu) : (pr >> 12);
          };
          const uint2 R0 = lds_at<uint2>(s_cb, vbyte + (code(0) << 3));
          const uint2 R1 = lds_at<uint2>(s_cb, vbyte + (code(1) << 3));
          const uint2 R2 = lds_at<uint2>(s_cb, vbyte + (code(2) << 3));
          const uint2 R3 = lds_at<uint2>(s_cb, vbyte + (code(3) << 3));
          VQKV_PV_PAIR(pp, R0, R1, R2, R3)
        }
      }
#undef VQKV_PV_PAIR
    }
  }
}

// 10-bit code at bit b of a lane's run words (b is a constant after
// unrolling, so the word indices are too).
template <int N>
__device__ __forceinline__ uint32_t bits10(const uint32_t (&w)[N], int b) {
  const int i = b >> 5, sh = b & 31;
  return (i + 1 < N ? __funnelshift_r(w[i], w[i + 1], sh) : w[i] >> sh) & 0x3ffu;
}

// Byte offset of centroid c in copy `rep` of a 1024-entry codebook whose four
// copies are interleaved in 128-byte rows: copy r holds its even / odd
// entries in 16-byte bank groups 2r / 2r+1.
__device__ __forceinline__ uint32_t cb10_offset(uint32_t c) { return ((c >> 1) << 7) | ((c & 1u) << 4); }

// One step of the 1.25-bit decode over T consecutive 16-token tiles.
// Scores: a 16-byte gather is channels 8j..8j+7 of subvector j = 4 s2 + tig
// (s2 = 0..3) for token gid (X) and gid+8 (Y), the A operand of two MMAs
// (qa[2 s2], qa[2 s2 + 1]); kw: the lane's 80-bit K run, token gid's 4 codes
// at bits 10 s2, token gid+8's at 40 + 10 s2.  P.V: subvector 8 pp + gid of
// the four tokens (2tig, 2tig+1, 2tig+8, 2tig+9) = slots 0..3 of the V run,
// code at bit 40 slot + 20 pp once the run is shifted right by vshift
// (10 bits for odd gid); each gather feeds four M-tiles (channel pairs).
// kbyte / vbyte: this lane's codebook copy (tig) in the K / V table.
template <int T>
__device__ __forceinline__ void vq125_step(const unsigned char* s_cb, uint32_t kbyte, uint32_t vbyte,
                                           const uint32_t (&qa)[8][2], const uint32_t (&kw)[T][3],
                                           const uint32_t (&vw)[T][5], uint32_t vshift, int tile0,
                                           const ColumnLimits& cl, int lane, float& m0, float& m1, float& l0,
                                           float& l1, float (&acc)[8][4]) {
  const int gid = lane >> 2;
  float sc[T][4];
#pragma unroll
  for (int i = 0; i < T; ++i) {
    float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      const uint4 X = lds_at<uint4>(s_cb, kbyte + cb10_offset(bits10(kw[i], 10 * s2)));
      const uint4 Y = lds_at<uint4>(s_cb, kbyte + cb10_offset(bits10(kw[i], 40 + 10 * s2)));
      mma_16816(da, X.x, Y.x, X.y, Y.y, qa[2 * s2][0], qa[2 * s2][1]);
      mma_16816(db, X.z, Y.z, X.w, Y.w, qa[2 * s2 + 1][0], qa[2 * s2 + 1][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[i][e] = da[e] + db[e];
  }
  if ((tile0 + T) * V2_TILE > cl.lim_min) {   // tail of the sequence
#pragma unroll
    for (int i = 0; i < T; ++i) mask_scores(sc[i], (tile0 + i) * V2_TILE + gid, cl);
  }
  uint32_t bP[T][2];
  softmax_tiles<T, 8>(sc, m0, m1, l0, l1, acc, bP);
#pragma unroll
  for (int i = 0; i < T; ++i) {
    uint32_t v[5];
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = __funnelshift_r(vw[i][m], vw[i][m + 1], vshift);
    v[4] = vw[i][4] >> vshift;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const uint4 R0 = lds_at<uint4>(s_cb, vbyte + cb10_offset(bits10(v, 20 * pp)));
      const uint4 R1 = lds_at<uint4>(s_cb, vbyte + cb10_offset(bits10(v, 40 + 20 * pp)));
      const uint4 R2 = lds_at<uint4>(s_cb, vbyte + cb10_offset(bits10(v, 80 + 20 * pp)));
      const uint4 R3 = lds_at<uint4>(s_cb, vbyte + cb10_offset(bits10(v, 120 + 20 * pp)));
      mma_16816(acc[4 * pp + 0], __byte_perm(R0.x, R1.x, 0x5410), __byte_perm(R0.x, R1.x, 0x7632),
                __byte_perm(R2.x, R3.x, 0x5410), __byte_perm(R2.x, R3.x, 0x7632), bP[i][0], bP[i][1]);
      mma_16816(acc[4 * pp + 1], __byte_perm(R0.y, R1.y, 0x5410), __byte_perm(R0.y, R1.y, 0x7632),
                __byte_perm(R2.y, R3.y, 0x5410), __byte_perm(R2.y, R3.y, 0x7632), bP[i][0], bP[i][1]);
      mma_16816(acc[4 * pp + 2], __byte_perm(R0.z, R1.z, 0x5410), __byte_perm(R0.z, R1.z, 0x7632),
                __byte_perm(R2.z, R3.z, 0x5410), __byte_perm(R2.z, R3.z, 0x7632), bP[i][0], bP[i][1]);
      mma_16816(acc[4 * pp + 3], __byte_perm(R0.w, R1.w, 0x5410), __byte_perm(R0.w, R1.w, 0x7632),
                __byte_perm(R2.w, R3.w, 0x5410), __byte_perm(R2.w, R3.w, 0x7632), bP[i][0], bP[i][1]);
    }
  }
}

// Merged search state of this lane's subvector over the 8 warps of its role
// (valid in the role's first warp).
__device__ __forceinline__ Best merge_role_slices(Best part, int warp, int lane, int slice, Best* s_part) {
  s_part[warp * 32 + lane] = part;
  __syncthreads();
  Best bst = part;
  if (slice == 0) {
#pragma unroll
    for (int w = 1; w < 8; ++w) bst = best_merge(bst, s_part[(warp + w) * 32 + lane]);
  }
  __syncthreads();   // s_part is reused
  return bst;
}

// Encode of the new K row (warps 0-7) and V row (warps 8-15) of one
// (sequence, KV head) for the fused append, from the lane's 4 transformed
// channels x of its row: each warp searches 32 of the 256 candidates
// (replica 0 of the shared codebook, one broadcast per load), the slices are
// merged as in the encode kernel, and warps 0 / 8 write the codes to the
// cache at token t_new (2 bit: lane j writes subvector j; 4 bit: lane j
// writes subvectors 2j and 2j+1).  The writes are made visible to the bulk
// copies (async proxy) that the CTA issues after the closing barrier.
// Called by every thread of the CTA after the codebook is in shared memory.
template <int DSUB>
__device__ __noinline__ void append_rows(float4 xv, uint8_t* k_stream, uint8_t* v_stream,
                                         unsigned long long* near_tie, int t_new, const unsigned char* s_cb,
                                         Best* s_part) {
  static_assert(V2_WARPS == 16, "two roles x 8 candidate slices");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int role = warp >> 3, slice = warp & 7;
  const float x[4] = {xv.x, xv.y, xv.z, xv.w};
  const unsigned char* cb_role = s_cb + role * 128;
  uint8_t* stream = role ? v_stream : k_stream;
  if constexpr (DSUB == 4) {
    const Best part = vq2_search(x, slice * 32, slice * 32 + 32, [&](int c) {
      const uint2 raw = *reinterpret_cast<const uint2*>(cb_role + c * 256);
      const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x);
      const __half2 hi = *reinterpret_cast<const __half2*>(&raw.y);
      return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
    });
    const Best bst = merge_role_slices(part, warp, lane, slice, s_part);
    if (slice == 0) {
      count_near_ties(near_tie, is_near_tie(bst.d, bst.s), lane, 0xffffffffu);
      stream[vq2_code_offset(role, t_new, lane)] = (uint8_t)bst.i;
      fence_proxy_async_global();
    }
  } else {
    Best pa, pb;
    vq4_search(x, slice * 32, slice * 32 + 32, [&](int c) {
      const __half2 v = *reinterpret_cast<const __half2*>(cb_role + c * 256);
      return make_float2(__low2float(v), __high2float(v));
    }, pa, pb);
    const Best ba = merge_role_slices(pa, warp, lane, slice, s_part);
    const Best bb = merge_role_slices(pb, warp, lane, slice, s_part);
    if (slice == 0) {
      count_near_ties(near_tie, is_near_tie(ba.d, ba.s), lane, 0xffffffffu);
      count_near_ties(near_tie, is_near_tie(bb.d, bb.s), lane, 0xffffffffu);
      stream[vq4_code_offset(role, t_new, 2 * lane)] = (uint8_t)ba.i;
      stream[vq4_code_offset(role, t_new, 2 * lane + 1)] = (uint8_t)bb.i;
      fence_proxy_async_global();
    }
  }
  __syncthreads();
}

// Flat plan: s_pref[b] = super-tiles (TPI tiles of 16 tokens) of sequences
// 0 .. b-1 at their clamped lengths, for b = 0 .. B.  All threads.
template <int TPI>
__device__ __forceinline__ void flat_prefix(const DecodeParams& p, int* s_pref) {
  const int lane = threadIdx.x & 31;
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
    const int raw = p.seq_lens[b], L = min(max(raw, 0), p.max_seq_len);
    if (raw != L && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(p.err, VQKV_DEVERR_SEQ_LEN);
    s_pref[b + 1] = ((L + V2_TILE - 1) / V2_TILE + TPI - 1) / TPI;
  }
  if (threadIdx.x == 0) s_pref[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {   // inclusive scan of s_pref[1..B], 32 entries per step
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int i = base + lane;
      int v = i < p.B ? s_pref[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i < p.B) s_pref[i + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

// Flat plan: the CTA (of S_eff) whose share [T s / S_eff, T (s+1) / S_eff)
// of the T super-tiles holds super-tile x.
__device__ __forceinline__ int flat_cta_of(long long x, long long T, int S_eff) {
  return (int)(((x + 1) * S_eff - 1) / T);
}

// Q: one query per sequence (kOneQuery: one limit, L, for every column),
// several (kQueries: per-column causal limits, all columns in the CTA) or
// several in column groups of up to 8, one CTA each (kQueryGroups).  PAGED:
// tiles are found through the block table (at most two bulk copies per
// step).
template <int Q, bool PAGED, int MODE, bool FLAT>
__global__ void __launch_bounds__(V2_THREADS, 1) decode_vq2_kernel(const DecodeParams p) {
  constexpr bool MULTI = Q != kOneQuery, GROUPS = Q == kQueryGroups;
  using G = V2Geo<MODE>;
  using Sm = V2Smem<MODE>;
  using Dim = typename std::conditional<MODE == VQKV_MODE_VQ4, Vq4Dim,
                                        typename std::conditional<G::TEN, Vq15Dim, Vq2Dim>::type>::type;
  constexpr bool APPEND = !G::PAIRS && !G::TEN;   // the fused append encodes one-byte codes only
  extern __shared__ __align__(128) unsigned char smem[];
  // Codebooks.  256 entries: centroid c at row c (256 bytes), K replicas at
  // c*256 + r*2*DSUB, V replicas at c*256 + 128 + r*2*DSUB; 2 bit: lane l
  // reads replica l % 16 (8 bytes), so each half-warp phase of a 64-bit
  // gather hits 16 bank pairs; 4 bit: lane l reads replica l (4 bytes), one
  // bank per lane.  4096 entries (3 bit): K centroid c at 8c, V at 32768 + 8c.
  // 1024 entries (1.25 bit): K copy r of centroid c at cb10_offset(c) + 32 r,
  // V at 65536 + the same; lane (gid, tig) reads copy tig.
  const unsigned char* s_cb = smem;
  float* s_qp = reinterpret_cast<float*>(smem + G::Q_OFF);
  float* s_comb = reinterpret_cast<float*>(smem);   // after the tile loop only
  __shared__ int s_last;

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int b_begin = (GROUPS ? cta_bgroup(p) : (int)blockIdx.z) * p.bpg;
  const int b_end = min(b_begin + p.bpg, p.B);
  // this CTA's softmax columns
  const int col0 = GROUPS ? cta_col0(p) : 0, nloc = GROUPS ? min(8, p.ncols - col0) : p.ncols;
  const uint32_t kbyte = G::PAIRS ? 0u
                        : G::TEN   ? (uint32_t)tig << 5
                        : G::DSUB == 4 ? (uint32_t)(lane & 15) << 3
                                       : (uint32_t)lane << 2;
  const uint32_t vbyte = G::PAIRS ? 32768u : G::TEN ? 65536u + kbyte : 128u | kbyte;
  // this warp's ring: stage st holds the K super-tile, then the V super-tile
  const uint32_t ring = smem_u32(smem + G::RING_OFF) + warp * (V2_STAGES * G::STAGE_BYTES);
  const uint32_t mbar = smem_u32(smem + G::MBAR_OFF) + warp * (V2_STAGES * 8);
  if (lane == 0) {
    for (int st = 0; st < V2_STAGES; ++st) mbar_init(mbar + 8 * st, 1);
    mbar_init_fence();
  }
  __syncwarp();
  grid_dependency_wait();
  grid_dependents_launch();
  uint32_t uses = 0;        // super-tiles this warp has taken through its ring (all sequences)

  // Flat plan (batches of ragged sequences): the KV head's T super-tiles,
  // all sequences in order, are cut into S_eff = min(n_splits, T) equal
  // shares, CTA `split` taking [T split / S_eff, T (split+1) / S_eff); each
  // overlap with a sequence is a piece, merged like a split.  Split 0 also
  // writes the zero rows of empty sequences.
  int* s_pref = reinterpret_cast<int*>(smem + Sm::FLAT_OFF);
  int* s_flat = s_pref + kFlatMaxB + 1;   // T, S_eff, r0, r1 (read at piece boundaries only)
  int b = b_begin, b_stop = b_end;
  if (FLAT) {
    flat_prefix<G::TPI>(p, s_pref);
    const int T = s_pref[p.B], S_eff = min(p.n_splits, T);
    b = p.B;
    if (split < S_eff) {
      const int r0 = (int)((long long)T * split / S_eff), r1 = (int)((long long)T * (split + 1) / S_eff);
      if (threadIdx.x == 0) s_flat[0] = T, s_flat[1] = S_eff, s_flat[2] = r0, s_flat[3] = r1;
      b = 0;
      while (s_pref[b + 1] <= r0) ++b;   // the first sequence reaching into the share
    }
    b_stop = p.B;
    if (split == 0) {
      for (int i = threadIdx.x; i < p.B * nloc * kHeadDim; i += V2_THREADS) {
        const int bb = i / (nloc * kHeadDim), c = col0 + (i / kHeadDim) % nloc;
        if (s_pref[bb + 1] == s_pref[bb]) p.out[out_row(p, bb, kvh, c) + (i & (kHeadDim - 1))] = __float2half_rn(0.f);
      }
    }
    __syncthreads();
  }

  for (; b < b_stop; ++b) {
    int piece_t0 = 0, piece_t1 = 0;   // flat plan: this CTA's tiles of sequence b
    if (FLAT) {
      const int lo = s_pref[b], hi = s_pref[b + 1], r0 = s_flat[2], r1 = s_flat[3];
      if (lo >= r1) break;
      if (hi == lo) continue;   // empty sequence
      piece_t0 = (max(r0, lo) - lo) * G::TPI;
      piece_t1 = (min(r1, hi) - lo) * G::TPI;
    }
    // Every input load of the prologue is issued before the first one is
    // used (the sequence length decides the rest): this warp's codebook
    // entry, its query column, and the new K / V row of a fused append.
    // (4096 entries: eight 16-byte pieces of the two 32-KB codebooks per thread)
    // (1024 entries: four 16-byte centroids of the two codebooks per thread)
    using CbEntry = typename std::conditional<
        G::PAIRS, uint4[8],
        typename std::conditional<G::TEN, uint4[4],
                                  typename std::conditional<G::DSUB == 4, uint2, uint32_t>::type>::type>::type;
    CbEntry cb_entry;
    if constexpr (G::TEN) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        cb_entry[i] = __ldg(reinterpret_cast<const uint4*>(i < 2 ? p.kcb : p.vcb) + (size_t)kvh * 1024 +
                            (i & 1) * V2_THREADS + threadIdx.x);
    } else if constexpr (G::PAIRS) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        cb_entry[i] = __ldg(reinterpret_cast<const uint4*>(i < 4 ? p.kcb : p.vcb) + (size_t)kvh * 2048 +
                            (i & 3) * V2_THREADS + threadIdx.x);
    } else {
      cb_entry = __ldg(reinterpret_cast<const CbEntry*>((threadIdx.x >> 8) ? p.vcb : p.kcb) + (size_t)kvh * 256 +
                       (threadIdx.x & 255));
    }
    const QueryLoad qload = load_query(p, b, kvh, warp, lane, col0, nloc);
    uint2 xraw = make_uint2(0u, 0u);
    float4 xs = make_float4(1.f, 1.f, 1.f, 1.f);
    if (APPEND && p.k_new != nullptr) {
      const size_t row = ((size_t)b * p.Hkv + kvh) * kHeadDim + 4 * lane;
      xraw = *reinterpret_cast<const uint2*>((warp < 8 ? p.k_new : p.v_new) + row);
      if (warp < 8) xs = *reinterpret_cast<const float4*>(p.s + (size_t)kvh * kHeadDim + 4 * lane);
    }
    const int L = load_len(p, b);
    const int ntiles = (L + V2_TILE - 1) / V2_TILE;
    const int t_begin = FLAT ? piece_t0 : split * p.tps;
    const int t_end = min(FLAT ? piece_t1 : t_begin + p.tps, ntiles);
    const ColumnLimits cl = MULTI ? column_limits(p, L, tig, col0) : ColumnLimits{L, L, L};
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = kMInit, m1 = kMInit, l0 = 0.f, l1 = 0.f;

    if (t_begin < t_end) {
      // super-tiles of G::TPI tiles: this warp takes k = warp + j * V2_WARPS,
      // j < n_mine, starting at tile t_begin + k * G::TPI.  The split length is
      // a multiple of G::TPI, so a super-tile never reaches into the next split;
      // tiles past the sequence end are masked, tiles past the capacity are not
      // copied.
      const int cap_tiles = (int)(p.stream_bytes / G::TILE_BYTES);
      const int blk_first = PAGED ? t_begin >> p.block_shift : 0;
      // blocks of this split's tiles [t_begin, t_end) held in s_blk
      const int n_blk = PAGED ? min(((t_end - 1) >> p.block_shift) - blk_first + 1, V2_BLK_CACHE) : 0;
      int* s_blk = reinterpret_cast<int*>(smem + Sm::BLK_OFF);
      const int n_super = (t_end - t_begin + G::TPI - 1) / G::TPI;
      const int n_mine = warp < n_super ? (n_super - warp + V2_WARPS - 1) / V2_WARPS : 0;
      auto issue = [&](int j) {
        const uint32_t st = (uses + j) % V2_STAGES;
        const int tile0 = t_begin + (warp + j * V2_WARPS) * G::TPI;
        // paged: never past the sequence's last tile, whose table entries
        // beyond it need not be valid (those slots are masked anyway)
        const int nt = min(G::TPI, (PAGED ? t_end : cap_tiles) - tile0);
        mbar_expect_tx(mbar + 8 * st, 2 * (uint32_t)nt * G::TILE_BYTES);
        bool bad = false;
        if (!PAGED) {   // the super-tile is contiguous
          const long long off = tile_offset<false>(p, b, kvh, tile0, G::TILE_BYTES, &bad);
          tma_load_1d(ring + st * G::STAGE_BYTES, p.kc + off, nt * G::TILE_BYTES, mbar + 8 * st);
          tma_load_1d(ring + st * G::STAGE_BYTES + G::TPI * G::TILE_BYTES, p.vc + off, nt * G::TILE_BYTES,
                      mbar + 8 * st);
        } else {
          // a step spans at most two blocks (nt <= 3 <= block_tiles); block ids
          // come from the shared-memory list when this split's fit in it
          static_assert(G::TPI <= 4, "a step must not span more than two blocks of >= 4 tiles");
          auto blk_off = [&](int tile) -> long long {
            const int lb = (tile >> p.block_shift) - blk_first;
            if (lb < n_blk) return ((long long)s_blk[lb] * p.Hkv + kvh) * p.block_bytes;
            bool bb = false;
            const long long off = tile_offset<true>(p, b, kvh, tile & ~(p.block_tiles - 1), G::TILE_BYTES, &bb);
            if (bb) atomicOr(p.err, VQKV_DEVERR_BLOCK);
            return off;
          };
          const int in_blk = tile0 & (p.block_tiles - 1);
          const int n0 = min(nt, p.block_tiles - in_blk);
          const long long off0 = blk_off(tile0) + (long long)in_blk * G::TILE_BYTES;
          tma_load_1d(ring + st * G::STAGE_BYTES, p.kc + off0, n0 * G::TILE_BYTES, mbar + 8 * st);
          tma_load_1d(ring + st * G::STAGE_BYTES + G::TPI * G::TILE_BYTES, p.vc + off0, n0 * G::TILE_BYTES,
                      mbar + 8 * st);
          if (n0 < nt) {   // the rest starts its next block
            const long long off1 = blk_off(tile0 + n0);
            tma_load_1d(ring + st * G::STAGE_BYTES + n0 * G::TILE_BYTES, p.kc + off1, (nt - n0) * G::TILE_BYTES,
                        mbar + 8 * st);
            tma_load_1d(ring + st * G::STAGE_BYTES + (G::TPI + n0) * G::TILE_BYTES, p.vc + off1,
                        (nt - n0) * G::TILE_BYTES, mbar + 8 * st);
          }
        }
      };
      if (PAGED) {   // block ids of this split's tiles, checked once
        for (int i = threadIdx.x; i < n_blk; i += V2_THREADS) {
          int blk = __ldg(p.block_table + (size_t)b * p.max_blocks + blk_first + i);
          if (blk < 0 || blk >= p.num_blocks) {
            atomicOr(p.err, VQKV_DEVERR_BLOCK);
            blk = 0;
          }
          s_blk[i] = blk;
        }
        __syncthreads();
      }
      // Fused append: the CTA whose split holds position L - 1 encodes the
      // new rows in its prologue and writes their codes before any copy of
      // that tile is issued, so the ring reads them like any other code.
      const int t_new = L - 1;
      const bool append = APPEND && p.k_new != nullptr && t_new >= 0 && (t_new >> 4) >= t_begin && (t_new >> 4) < t_end;
      const int k_new = append ? ((t_new >> 4) - t_begin) / G::TPI : 0;   // super-tile of the new token
      const bool late_start = append && k_new % V2_WARPS == warp && k_new / V2_WARPS < V2_STAGES - 1;
      // start the ring before the prologue so the copies overlap it (after
      // the append for the one warp whose first copies hold the new token)
      if (lane == 0 && !late_start)
        for (int j = 0; j < min(V2_STAGES - 1, n_mine); ++j)
          if (!(p.withhold_first_copy && j == 0)) issue(j);
      // the new row's transform (warps 0-7: smoothed, rotated key) before
      // the codebook fill, which only the search needs
      float4 xnew = make_float4(0.f, 0.f, 0.f, 0.f);
      if (append) {
        float x[4];
        transform_loaded(xraw, warp < 8, xs, lane, x);
        xnew = make_float4(x[0], x[1], x[2], x[3]);
      }
      if constexpr (G::TEN) {
        // the four copies of each centroid; copy (k + c/2) % 4 at step k keeps
        // the 8 lanes of each store phase on distinct 16-byte bank groups
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t c = (uint32_t)((i & 1) * V2_THREADS + threadIdx.x);
          unsigned char* row = smem + (i >> 1) * 65536 + cb10_offset(c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(row + 32 * ((k + (c >> 1)) & 3)) = cb_entry[i];
        }
      } else if constexpr (G::PAIRS) {
#pragma unroll
        for (int i = 0; i < 8; ++i) reinterpret_cast<uint4*>(smem)[i * V2_THREADS + threadIdx.x] = cb_entry[i];
      } else {
        // thread t writes the G::REPL replicas of centroid t & 255 of K
        // (t < 256) or V (t >= 256), loaded above; replica (i + lane) % REPL
        // at step i keeps the lanes of each store phase on distinct banks
        static_assert(V2_THREADS == 512, "one thread per K and V centroid");
        const int c = threadIdx.x & 255, role = threadIdx.x >> 8;
        CbEntry* row = reinterpret_cast<CbEntry*>(smem + c * 256 + role * 128);
#pragma unroll 1
        for (int i = 0; i < G::REPL; ++i) row[(i + lane) & (G::REPL - 1)] = cb_entry;
      }
      transform_query(p, qload, warp, lane, s_qp, V2_Q_PITCH, nloc);
      __syncthreads();
      if constexpr (APPEND) if (append) {
        const size_t stream = (size_t)(b * p.Hkv + kvh) * p.stream_bytes;
        append_rows<G::DSUB>(xnew, p.kc_w + stream, p.vc_w + stream, p.near_tie, t_new, smem,
                    reinterpret_cast<Best*>(smem + Sm::APP_OFF));
        if (lane == 0 && late_start)
          for (int j = 0; j < min(V2_STAGES - 1, n_mine); ++j)
            if (!(p.withhold_first_copy && j == 0)) issue(j);
      }
      // B operand of the score MMA: head gid; 2 and 3 bit: channels
      // 4j..4j+3 of j = 4s+tig; 4 bit: channels 16s+2tig, +1 and
      // 16s+8+2tig, +1; 1.25 bit: channels 8j + 4(s%2) .. +3 of j = 4(s/2)+tig
      uint32_t qa[8][2];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        if (gid < nloc) {
          if constexpr (G::TEN) {
            const float4 v = *reinterpret_cast<const float4*>(s_qp + gid * V2_Q_PITCH +
                                                              8 * (4 * (s >> 1) + tig) + 4 * (s & 1));
            qa[s][0] = pack_half2(v.x, v.y);
            qa[s][1] = pack_half2(v.z, v.w);
          } else if constexpr (G::DSUB == 4) {
            const float4 v = *reinterpret_cast<const float4*>(s_qp + gid * V2_Q_PITCH + 4 * (4 * s + tig));
            qa[s][0] = pack_half2(v.x, v.y);
            qa[s][1] = pack_half2(v.z, v.w);
          } else {
            const float2 v0 = *reinterpret_cast<const float2*>(s_qp + gid * V2_Q_PITCH + 16 * s + 2 * tig);
            const float2 v1 = *reinterpret_cast<const float2*>(s_qp + gid * V2_Q_PITCH + 16 * s + 8 + 2 * tig);
            qa[s][0] = pack_half2(v0.x, v0.y);
            qa[s][1] = pack_half2(v1.x, v1.y);
          }
        } else {
          qa[s][0] = qa[s][1] = 0u;
        }
      }

      int stalled = -1;   // ring index whose wait gave up
      for (int j = 0; j < n_mine; ++j) {
        const uint32_t st = (uses + j) % V2_STAGES;
        const uint32_t par = ((uses + j) / V2_STAGES) & 1u;
        if (!mbar_wait_bounded(mbar + 8 * st, par, p.max_polls)) {
          stalled = j;
          break;
        }
        // the lane's code words: plane w (every lane's 16- or 8-byte piece
        // of it, contiguous) at 512 w; 1.25 bit: planes at 0 and 256, V run
        // 4 (gid / 2) + tig shared by the lanes gid and gid ^ 1
        uint32_t kq[G::TPI][G::KW], vq[G::TPI][G::VW];
#pragma unroll
        for (int i = 0; i < G::TPI; ++i) {
          const uint32_t kt = ring + st * G::STAGE_BYTES + i * G::TILE_BYTES;
          const uint32_t vt = kt + G::TPI * G::TILE_BYTES;
          if constexpr (G::TEN) {
            const uint2 a = lds64(kt + 8 * lane);
            kq[i][0] = a.x, kq[i][1] = a.y, kq[i][2] = lds16(kt + 256 + 2 * lane);
            const uint32_t run = 4 * (gid >> 1) + tig;
            const uint4 c = lds128(vt + 16 * run);
            vq[i][0] = c.x, vq[i][1] = c.y, vq[i][2] = c.z, vq[i][3] = c.w, vq[i][4] = lds32(vt + 256 + 4 * run);
          } else {
#pragma unroll
            for (int w = 0; w < G::LW / 4; ++w) {
              const uint4 a = lds128(kt + 512 * w + lane * 16), c = lds128(vt + 512 * w + lane * 16);
              kq[i][4 * w] = a.x, kq[i][4 * w + 1] = a.y, kq[i][4 * w + 2] = a.z, kq[i][4 * w + 3] = a.w;
              vq[i][4 * w] = c.x, vq[i][4 * w + 1] = c.y, vq[i][4 * w + 2] = c.z, vq[i][4 * w + 3] = c.w;
            }
            if constexpr (G::LW % 4 != 0) {
              const uint2 a = lds64(kt + 512 + lane * 8), c = lds64(vt + 512 + lane * 8);
              kq[i][G::LW - 2] = a.x, kq[i][G::LW - 1] = a.y;
              vq[i][G::LW - 2] = c.x, vq[i][G::LW - 1] = c.y;
            }
          }
        }
        __syncwarp();
        // refill the stage this warp finished with in the previous step
        if (lane == 0 && j + V2_STAGES - 1 < n_mine) issue(j + V2_STAGES - 1);
        if constexpr (G::TEN)
          vq125_step<G::TPI>(s_cb, kbyte, vbyte, qa, kq, vq, 10u * (gid & 1), t_begin + (warp + j * V2_WARPS) * G::TPI,
                             cl, lane, m0, m1, l0, l1, acc);
        else
          vq2_step<G::TPI, MODE>(s_cb, kbyte, vbyte, qa, kq, vq, t_begin + (warp + j * V2_WARPS) * G::TPI, cl,
                                 lane, m0, m1, l0, l1, acc);
      }
      if (stalled >= 0) {
        // The copies in flight are exactly the ring indices issued but not
        // consumed: index `stalled` and the refills issued ahead of it, i.e.
        // stalled .. min(stalled + V2_STAGES - 2, n_mine - 1) (index j + S - 1
        // is issued only after index j is consumed).  Give each of them a
        // bounded chance to land, on its own stage and phase, before the
        // ring is reused or the CTA exits, and report the failure.
        const int last = min(stalled + V2_STAGES - 2, n_mine - 1);
        for (int j = stalled; j <= last; ++j)
          mbar_wait_bounded(mbar + 8 * ((uses + j) % V2_STAGES), ((uses + j) / V2_STAGES) & 1u, p.max_polls);
        if (lane == 0) atomicOr(p.err, VQKV_DEVERR_TIMEOUT);
      }
      uses += n_mine;
    }
    __syncthreads();   // every warp is done with the codebooks: reuse them for the combine
    stash_warp<V2_WARPS, 8>(s_comb, warp, lane, acc, m0, m1, l0, l1, Dim());
    __syncthreads();
    MergeSpan span = split_span(p, b, kvh, split, col0);
    if (FLAT) {   // CTAs s_first .. s_last share sequence b; piece ids s + b
      const int T = s_flat[0], S_eff = s_flat[1];
      const int s_first = flat_cta_of(s_pref[b], T, S_eff), s_last = flat_cta_of(s_pref[b + 1] - 1, T, S_eff);
      span = {split - s_first, s_last - s_first + 1,
              (((size_t)kvh * (p.n_splits + p.B - 1) + s_first + b) * p.ncols + col0) * kPartialStride};
    }
    finish_sequence<V2_WARPS, GROUPS, Dim>(p, b, kvh, span, s_comb, &s_last);
    __syncthreads();   // (a warp that timed out still takes part in every barrier)
  }
}

// 24-bit code pair k (bytes 3k..3k+2) of a lane's 12-byte run (3 words).
__device__ __forceinline__ uint32_t pair24(uint32_t w0, uint32_t w1, uint32_t w2, int k) {
  if (k == 0) return w0 & 0xffffffu;
  if (k == 1) return __funnelshift_r(w0, w1, 24) & 0xffffffu;
  if (k == 2) return __funnelshift_r(w1, w2, 16) & 0xffffffu;
  return w2 >> 8;
}

template <int Q, bool PAGED>
__global__ void __launch_bounds__(V15_THREADS, 1) decode_vq15_kernel(const DecodeParams p) {
  constexpr bool MULTI = Q != kOneQuery, GROUPS = Q == kQueryGroups;
  extern __shared__ __align__(128) unsigned char smem[];
  uint4* s_kcb = reinterpret_cast<uint4*>(smem);
  uint4* s_vcb = reinterpret_cast<uint4*>(smem + V15_CB_BYTES);
  float* s_comb = reinterpret_cast<float*>(smem + 2 * V15_CB_BYTES);
  float* s_qp = reinterpret_cast<float*>(smem + V15_Q_OFF);
  const uint32_t slot = smem_u32(smem + V15_SLOT_OFF) + threadIdx.x * 96;
  __shared__ int s_last;

  const int split = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int b_begin = (GROUPS ? cta_bgroup(p) : (int)blockIdx.z) * p.bpg;
  const int b_end = min(b_begin + p.bpg, p.B);
  // this CTA's softmax columns
  const int col0 = GROUPS ? cta_col0(p) : 0, nloc = GROUPS ? min(8, p.ncols - col0) : p.ncols;
  const uint32_t kcb_s = smem_u32(s_kcb);
  const uint32_t vcb_s = smem_u32(s_vcb);
  bool have_cb = false;
  grid_dependency_wait();
  grid_dependents_launch();

  for (int b = b_begin; b < b_end; ++b) {
    const int L = load_len(p, b);
    const int ntiles = (L + V15_TILE - 1) / V15_TILE;
    const int t_begin = split * p.tps;
    const int t_end = min(t_begin + p.tps, ntiles);
    const ColumnLimits cl = MULTI ? column_limits(p, L, tig, col0) : ColumnLimits{L, L, L};
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = kMInit, m1 = kMInit, l0 = 0.f, l1 = 0.f;

    if (t_begin < t_end) {
      // this lane's 48 + 48 code bytes of `tile` into its slot
      auto copy_codes = [&](int tile) {
        bool bad = false;
        const long long off = tile_offset<PAGED>(p, b, kvh, tile, V15_TILE_BYTES, &bad) + lane * 48;
        if (PAGED && bad && lane == 0) atomicOr(p.err, VQKV_DEVERR_BLOCK);
        const uint8_t* kp = p.kc + off;
        const uint8_t* vp = p.vc + off;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          cp_async16(slot + 16 * i, kp + 16 * i, 16);
          cp_async16(slot + 48 + 16 * i, vp + 16 * i, 16);
        }
        cp_async_commit();
      };
      // the first tile's copy overlaps the prologue
      if (t_begin + warp < t_end) copy_codes(t_begin + warp);
      if (!have_cb) {
        const uint4* gk = reinterpret_cast<const uint4*>(p.kcb) + (size_t)kvh * 4096;
        const uint4* gv = reinterpret_cast<const uint4*>(p.vcb) + (size_t)kvh * 4096;
#pragma unroll 4
        for (int k = threadIdx.x; k < 4096; k += V15_THREADS) {
          s_kcb[k] = __ldg(gk + k);
          s_vcb[k] = __ldg(gv + k);
        }
        have_cb = true;
      }
      transform_queries(p, b, kvh, warp, lane, s_qp, V15_Q_PITCH, col0, nloc);
      __syncthreads();
      uint32_t qf[8][2];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int j = 4 * (s >> 1) + tig;     // subvector
        const int c = 8 * j + 4 * (s & 1);    // first channel of this half
        if (gid < nloc) {
          const float4 v = *reinterpret_cast<const float4*>(s_qp + gid * V15_Q_PITCH + c);
          qf[s][0] = pack_half2(v.x, v.y);
          qf[s][1] = pack_half2(v.z, v.w);
        } else {
          qf[s][0] = qf[s][1] = 0u;
        }
      }
      __syncthreads();

      for (int tile = t_begin + warp; tile < t_end; tile += V15_WARPS) {
        uint32_t kw[12], vw[12];
        cp_async_wait<0>();
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const uint4 a = lds128(slot + 16 * i);
          kw[4 * i] = a.x; kw[4 * i + 1] = a.y; kw[4 * i + 2] = a.z; kw[4 * i + 3] = a.w;
          const uint4 c = lds128(slot + 48 + 16 * i);
          vw[4 * i] = c.x; vw[4 * i + 1] = c.y; vw[4 * i + 2] = c.z; vw[4 * i + 3] = c.w;
        }
        if (tile + V15_WARPS < t_end) {
          // the slot is overwritten only after every word above has arrived
          asm volatile("" ::"r"(kw[0]), "r"(kw[1]), "r"(kw[2]), "r"(kw[3]), "r"(kw[4]), "r"(kw[5]),
                       "r"(kw[6]), "r"(kw[7]), "r"(kw[8]), "r"(kw[9]), "r"(kw[10]), "r"(kw[11]));
          asm volatile("" ::"r"(vw[0]), "r"(vw[1]), "r"(vw[2]), "r"(vw[3]), "r"(vw[4]), "r"(vw[5]),
                       "r"(vw[6]), "r"(vw[7]), "r"(vw[8]), "r"(vw[9]), "r"(vw[10]), "r"(vw[11]));
          copy_codes(tile + V15_WARPS);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tq = tile * V15_TILE + 16 * u;   // first token of this quarter
          if (tq >= L) break;
          const uint32_t k0 = kw[3 * u], k1 = kw[3 * u + 1], k2 = kw[3 * u + 2];
          // pairs: token gid -> bytes 0..5 (pair index tig, tig+4), token gid+8 -> bytes 6..11
          const uint32_t pa0 = pair24(k0, k1, k2, 0), pa1 = pair24(k0, k1, k2, 1);
          const uint32_t pb0 = pair24(k0, k1, k2, 2), pb1 = pair24(k0, k1, k2, 3);
          float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2) {
            // subvector j = 4*s2 + tig: s2 0 -> lo(pair0), 1 -> lo(pair1), 2 -> hi(pair0), 3 -> hi(pair1)
            const uint32_t va = (s2 & 1) ? pa1 : pa0;
            const uint32_t vb = (s2 & 1) ? pb1 : pb0;
            const uint32_t ca = (s2 < 2) ? (va & 0xfffu) : (va >> 12);
            const uint32_t cb = (s2 < 2) ? (vb & 0xfffu) : (vb >> 12);
            const uint4 X = lds128(kcb_s + ca * 16);
            const uint4 Y = lds128(kcb_s + cb * 16);
            mma_16816(sc, X.x, Y.x, X.y, Y.y, qf[2 * s2][0], qf[2 * s2][1]);
            mma_16816(sc, X.z, Y.z, X.w, Y.w, qf[2 * s2 + 1][0], qf[2 * s2 + 1][1]);
          }
          if (tq + 16 > cl.lim_min) mask_scores(sc, tq + gid, cl);
          uint32_t bP0, bP1;
          softmax_tile(sc, m0, m1, l0, l1, acc, bP0, bP1);

          const uint32_t v0 = vw[3 * u], v1 = vw[3 * u + 1], v2 = vw[3 * u + 2];
          const uint32_t q0 = pair24(v0, v1, v2, 0), q1 = pair24(v0, v1, v2, 1);
          const uint32_t q2 = pair24(v0, v1, v2, 2), q3 = pair24(v0, v1, v2, 3);
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            // subvector J = gid + 8*pp: low code of each pair for pp = 0, high for pp = 1
            const uint32_t c0 = pp ? (q0 >> 12) : (q0 & 0xfffu);
            const uint32_t c1 = pp ? (q1 >> 12) : (q1 & 0xfffu);
            const uint32_t c2 = pp ? (q2 >> 12) : (q2 & 0xfffu);
            const uint32_t c3 = pp ? (q3 >> 12) : (q3 & 0xfffu);
            const uint4 R0 = lds128(vcb_s + c0 * 16);
            const uint4 R1 = lds128(vcb_s + c1 * 16);
            const uint4 R2 = lds128(vcb_s + c2 * 16);
            const uint4 R3 = lds128(vcb_s + c3 * 16);
            mma_16816(acc[4 * pp + 0], __byte_perm(R0.x, R1.x, 0x5410), __byte_perm(R0.x, R1.x, 0x7632),
                      __byte_perm(R2.x, R3.x, 0x5410), __byte_perm(R2.x, R3.x, 0x7632), bP0, bP1);
            mma_16816(acc[4 * pp + 1], __byte_perm(R0.y, R1.y, 0x5410), __byte_perm(R0.y, R1.y, 0x7632),
                      __byte_perm(R2.y, R3.y, 0x5410), __byte_perm(R2.y, R3.y, 0x7632), bP0, bP1);
            mma_16816(acc[4 * pp + 2], __byte_perm(R0.z, R1.z, 0x5410), __byte_perm(R0.z, R1.z, 0x7632),
                      __byte_perm(R2.z, R3.z, 0x5410), __byte_perm(R2.z, R3.z, 0x7632), bP0, bP1);
            mma_16816(acc[4 * pp + 3], __byte_perm(R0.w, R1.w, 0x5410), __byte_perm(R0.w, R1.w, 0x7632),
                      __byte_perm(R2.w, R3.w, 0x5410), __byte_perm(R2.w, R3.w, 0x7632), bP0, bP1);
          }
        }
      }
    }
    __syncthreads();   // every warp is done with its code slot: the combine area overlaps them
    stash_warp<V15_WARPS, 8>(s_comb, warp, lane, acc, m0, m1, l0, l1, Vq15Dim());
    __syncthreads();
    finish_sequence<V15_WARPS, GROUPS, Vq15Dim>(p, b, kvh, split_span(p, b, kvh, split, col0), s_comb, &s_last);
    __syncthreads();
  }
}

// One CTA per (query head, sequence), one thread per channel.
__global__ void __launch_bounds__(kHeadDim) decode_combine_kernel(const DecodeParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  combine_splits(p);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  return launch_pdl(decode_combine_kernel, dim3(p.Hkv * p.ncols, p.B), dim3(kHeadDim), 0, stream, p);
}

int decode_tile_tokens(int mode) { return mode == VQKV_MODE_VQ15 ? V15_TILE : V2_TILE; }
int decode_tiles_per_step(int mode) {
  return mode == VQKV_MODE_VQ2   ? V2Geo<VQKV_MODE_VQ2>::TPI
         : mode == VQKV_MODE_VQ4 ? V2Geo<VQKV_MODE_VQ4>::TPI
         : mode == VQKV_MODE_VQ3 ? V2Geo<VQKV_MODE_VQ3>::TPI
         : mode == VQKV_MODE_VQ125 ? V2Geo<VQKV_MODE_VQ125>::TPI
                                 : 1;
}
size_t decode_smem_bytes(int mode) {
  return mode == VQKV_MODE_VQ2     ? kV2Smem
         : mode == VQKV_MODE_VQ4   ? kV4Smem
         : mode == VQKV_MODE_VQ3   ? kV3Smem
         : mode == VQKV_MODE_VQ125 ? kV125Smem
                                   : kV15Smem;
}
int decode_threads(int mode) { return mode == VQKV_MODE_VQ15 ? V15_THREADS : V2_THREADS; }

namespace {
using DecodeKernel = void (*)(DecodeParams);

// [flat][paged][query layout] instantiations of one mode's decode kernel.
template <int MODE>
struct ByteCodeKernels {
  static constexpr DecodeKernel k[2][2][3] = {
      {{decode_vq2_kernel<kOneQuery, false, MODE, false>, decode_vq2_kernel<kQueries, false, MODE, false>,
        decode_vq2_kernel<kQueryGroups, false, MODE, false>},
       {decode_vq2_kernel<kOneQuery, true, MODE, false>, decode_vq2_kernel<kQueries, true, MODE, false>,
        decode_vq2_kernel<kQueryGroups, true, MODE, false>}},
      {{decode_vq2_kernel<kOneQuery, false, MODE, true>, decode_vq2_kernel<kQueries, false, MODE, true>,
        decode_vq2_kernel<kQueryGroups, false, MODE, true>},
       {decode_vq2_kernel<kOneQuery, true, MODE, true>, decode_vq2_kernel<kQueries, true, MODE, true>,
        decode_vq2_kernel<kQueryGroups, true, MODE, true>}}};
};
struct Vq15Kernels {
  static constexpr DecodeKernel k[2][2][3] = {
      {{decode_vq15_kernel<kOneQuery, false>, decode_vq15_kernel<kQueries, false>,
        decode_vq15_kernel<kQueryGroups, false>},
       {decode_vq15_kernel<kOneQuery, true>, decode_vq15_kernel<kQueries, true>,
        decode_vq15_kernel<kQueryGroups, true>}},
      {{nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr}}};   // no flat plan at 1.5 bit
};

const DecodeKernel (*kernels_of(int mode))[2][3] {
  return mode == VQKV_MODE_VQ2   ? ByteCodeKernels<VQKV_MODE_VQ2>::k
         : mode == VQKV_MODE_VQ4 ? ByteCodeKernels<VQKV_MODE_VQ4>::k
         : mode == VQKV_MODE_VQ3 ? ByteCodeKernels<VQKV_MODE_VQ3>::k
         : mode == VQKV_MODE_VQ125 ? ByteCodeKernels<VQKV_MODE_VQ125>::k
                                 : Vq15Kernels::k;
}
}  // namespace

cudaError_t decode_prepare(int mode) {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const auto ks = kernels_of(mode);
  cudaError_t e = cudaSuccess;
  for (int fl = 0; fl < 2; ++fl)
    for (int pg = 0; pg < 2; ++pg)
      for (int q = 0; q < 3; ++q)
        if (e == cudaSuccess && ks[fl][pg][q] != nullptr)
          e = cudaFuncSetAttribute(ks[fl][pg][q], a, (int)decode_smem_bytes(mode));
  return e;
}

cudaError_t decode_occupancy(int mode, int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kernels_of(mode)[0][0][kOneQuery],
                                                       decode_threads(mode), decode_smem_bytes(mode));
}

cudaError_t launch_decode(int mode, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  const int q = p.M == 1 ? kOneQuery : p.cgroups == 1 ? kQueries : kQueryGroups;
  const bool paged = p.block_table != nullptr;
  const DecodeKernel k = kernels_of(mode)[p.flat ? 1 : 0][paged][q];
  if (k == nullptr) return cudaErrorInvalidValue;
  return launch_pdl(k, grid, dim3(decode_threads(mode)), decode_smem_bytes(mode), stream, p);
}

}  // namespace vqkv
