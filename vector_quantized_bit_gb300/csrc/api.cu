// Host side of the C ABI declared in include/vqkv.h: argument validation,
// the split-KV plan, workspace layout and kernel launches.  Nothing here
// allocates device memory or synchronises the host.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "vqkv.h"

namespace vqkv {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kWsHeader = 256;   // word 0: device error flags

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int decode_bpsm[kCodeModes + 1] = {};   // resident decode CTAs per SM: each code mode, then fp16
  int encode_bpsm[kCodeModes] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device attributes, queried once (kernel attributes set here too).
vqkv_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VQKV_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return VQKV_ERR_NO_DEVICE;
    for (int m = 0; m < kCodeModes; ++m) {
      if (decode_prepare(m) != cudaSuccess || encode_prepare(m) != cudaSuccess) return VQKV_ERR_CUDA;
      if (decode_occupancy(m, &d.decode_bpsm[m]) != cudaSuccess) return VQKV_ERR_CUDA;
      if (encode_occupancy(m, &d.encode_bpsm[m]) != cudaSuccess) return VQKV_ERR_CUDA;
      if (d.decode_bpsm[m] < 1) d.decode_bpsm[m] = 1;
      if (d.encode_bpsm[m] < 1) d.encode_bpsm[m] = 1;
    }
    if (decode_fp16_prepare() != cudaSuccess || decode_fp16_occupancy(&d.decode_bpsm[kModeFp16]) != cudaSuccess)
      return VQKV_ERR_CUDA;
    if (d.decode_bpsm[kModeFp16] < 1) d.decode_bpsm[kModeFp16] = 1;
    d.ready = true;
  }
  *out = d;
  return VQKV_OK;
}

bool is_code_mode(int m) {
  return m == VQKV_MODE_VQ2 || m == VQKV_MODE_VQ15 || m == VQKV_MODE_VQ4 || m == VQKV_MODE_VQ3 ||
         m == VQKV_MODE_VQ125;
}
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sizes only (what the split plan and the workspace size depend on).
vqkv_status validate_decode_sizes(const vqkv_decode_args* a) {
  if (a == nullptr) return VQKV_ERR_INVALID_ARG;
  if (!is_code_mode(a->mode)) return VQKV_ERR_UNSUPPORTED;
  if (a->head_dim != 128) return VQKV_ERR_UNSUPPORTED;
  if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->cap_len < 1) return VQKV_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return VQKV_ERR_INVALID_ARG;
  if (a->Hq / a->Hkv > 8) return VQKV_ERR_UNSUPPORTED;
  if (a->max_seq_len < 0 || a->max_seq_len > a->cap_len) return VQKV_ERR_INVALID_ARG;
  if (a->num_splits < 0) return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

vqkv_status validate_decode(const vqkv_decode_args* a) {
  if (a == nullptr) return VQKV_ERR_INVALID_ARG;
  if (!is_code_mode(a->mode)) return VQKV_ERR_UNSUPPORTED;
  if (a->head_dim != 128) return VQKV_ERR_UNSUPPORTED;
  if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->cap_len < 1) return VQKV_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return VQKV_ERR_INVALID_ARG;
  if (a->Hq / a->Hkv > 8) return VQKV_ERR_UNSUPPORTED;
  if (a->max_seq_len < 0 || a->max_seq_len > a->cap_len) return VQKV_ERR_INVALID_ARG;
  if (a->num_splits < 0) return VQKV_ERR_INVALID_ARG;
  if (!(std::isfinite(a->softmax_scale))) return VQKV_ERR_INVALID_ARG;
  if (a->B == 0) return VQKV_OK;
  if (!a->q || !a->k_codes || !a->v_codes || !a->seq_lens || !a->k_codebook || !a->v_codebook || !a->s ||
      !a->out)
    return VQKV_ERR_INVALID_ARG;
  if (!aligned(a->q, 8) || !aligned(a->k_codes, 16) || !aligned(a->v_codes, 16) || !aligned(a->k_codebook, 16) ||
      !aligned(a->v_codebook, 16) || !aligned(a->s, 16) || !aligned(a->seq_lens, 4) || !aligned(a->out, 2))
    return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

// Block-table arguments of the paged calls: sizes and alignment only.
vqkv_status validate_paging(const vqkv_paging* pg, int mode, int cap_len) {
  if (pg == nullptr) return VQKV_ERR_INVALID_ARG;
  if (pg->max_blocks < 1 || pg->num_blocks < 1 || pg->block_tokens < 64 ||
      (pg->block_tokens & (pg->block_tokens - 1)) != 0)
    return VQKV_ERR_INVALID_ARG;
  if ((long long)pg->max_blocks * pg->block_tokens < cap_len) return VQKV_ERR_INVALID_ARG;
  if ((long long)pg->num_blocks * vqkv_code_bytes(mode, pg->block_tokens) > (1LL << 46)) return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

template <typename P>
void set_paging(P& p, const vqkv_paging* pg, int mode) {
  if (pg == nullptr) return;
  p.block_table = pg->block_table;
  p.max_blocks = pg->max_blocks;
  p.block_tiles = pg->block_tokens / decode_tile_tokens(mode);
  p.block_shift = 0;
  while ((1 << p.block_shift) < p.block_tiles) ++p.block_shift;
  p.num_blocks = pg->num_blocks;
  p.block_bytes = (long long)vqkv_code_bytes(mode, pg->block_tokens);
}

}  // namespace
size_t decode_ticket_region_bytes(int B, int Hkv);
namespace {

struct DecodePlan {
  int n_splits = 1, tps = 1, bpg = 1, n_bgroups = 1, cgroups = 1, flat = 0;
  size_t tickets_off = 0, partials_off = 0, ws_bytes = 0;
};

// Split-KV plan.  Work is (sequence group, KV head, split); every CTA of a
// split processes `tps` tiles of each sequence in its group.  The plan picks
// the split count that minimises (waves of CTAs) x (tiles per CTA + a fixed
// per-CTA setup cost), assuming full-length sequences; short sequences make
// some CTAs finish early, which the hardware scheduler backfills.
struct PlanInput {
  int mode;   // a code mode or kModeFp16
  int B, Hq, Hkv, max_seq_len, num_splits;
  int M = 1;  // queries per sequence
  // Tiles' worth of extra work in the CTA whose split holds a sequence's
  // last token (the fused append encodes the new rows there first).  When
  // every CTA of the plan runs at once, the splits are sized for
  // max_seq_len + credit_tiles, so that split comes out this much shorter.
  int credit_tiles = 0;
};

vqkv_status plan_decode(const PlanInput* a, DecodePlan* pl) {
  DeviceInfo di;
  vqkv_status st = device_info(&di);
  if (st != VQKV_OK) return st;
  const int T = a->mode == kModeFp16 ? 16 : decode_tile_tokens(a->mode);
  const int unit_tiles = a->mode == kModeFp16 ? 1 : decode_tiles_per_step(a->mode);
  const int g = a->Hq / a->Hkv;
  const long long tiles_max = std::max(1, (a->max_seq_len + T - 1) / T);
  const long long slots = (long long)di.sms * di.decode_bpsm[a->mode];
  const int B = std::max(a->B, 1);
  // 1.5-bit CTAs load 128 KB of codebooks: keep one CTA per KV head and split
  // across sequences only when the batch alone cannot fill the GPU.
  int bpg = 1;
  if (a->mode == VQKV_MODE_VQ15 && (long long)B * a->Hkv < slots) bpg = B;
  const int cgroups = (g * a->M + 7) / 8;   // CTAs per (sequence group, KV head, split)
  // Flat plan for batches on the tile-ring decode: one wave of CTAs per (KV
  // head, column group), each taking an equal share of all sequences' tiles,
  // balanced by the actual lengths on the device (ragged batches leave no CTA
  // idle).  Explicit split counts keep the split plan.
  const bool ring = a->mode == VQKV_MODE_VQ2 || a->mode == VQKV_MODE_VQ4 || a->mode == VQKV_MODE_VQ3 ||
                    a->mode == VQKV_MODE_VQ125;
  const long long super_max = (tiles_max + unit_tiles - 1) / unit_tiles;
  if (ring && a->num_splits == 0 && a->B > 1 && a->B <= kFlatMaxB && (long long)a->B * super_max < (1LL << 30)) {
    const long long S = std::max<long long>(1, slots / ((long long)a->Hkv * cgroups));
    pl->flat = 1;
    pl->n_splits = (int)S;
    pl->tps = 0;
    pl->bpg = 1;
    pl->n_bgroups = 1;
    pl->cgroups = cgroups;
    pl->tickets_off = kWsHeader;
    pl->partials_off = decode_ticket_region_bytes(B, a->Hkv * cgroups);
    pl->ws_bytes = pl->partials_off +
                   sizeof(float) * (size_t)a->Hkv * (S + a->B - 1) * g * a->M * kPartialStride;
    return VQKV_OK;
  }
  const long long pairs = (long long)a->Hkv * ((B + bpg - 1) / bpg) * cgroups;
  // per-CTA prologue + merge in tile units
  const double setup_tiles = (a->mode == VQKV_MODE_VQ15) ? 24.0 : (a->mode == kModeFp16) ? 4.0 : 12.0;
  long long best_n = 1;
  double best_cost = 1e300;
  if (a->num_splits > 0) {
    best_n = std::min<long long>(a->num_splits, tiles_max);
  } else {
    const long long n_hi = std::min<long long>(tiles_max, 4 * ((slots + pairs - 1) / pairs) + 64);
    for (long long n = 1; n <= n_hi; ++n) {
      const long long tps = (tiles_max + n - 1) / n;
      const long long waves = (pairs * n + slots - 1) / slots;
      const double cost = (double)waves * ((double)tps * bpg + setup_tiles);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best_n = n;
      }
    }
  }
  const long long unit = unit_tiles;
  const bool one_wave = pairs * best_n <= slots;
  const long long credit = (a->num_splits == 0 && one_wave) ? a->credit_tiles : 0;
  const long long tps = ((tiles_max + credit + best_n - 1) / best_n + unit - 1) / unit * unit;
  pl->tps = (int)tps;
  pl->n_splits = (int)((tiles_max + tps - 1) / tps);
  pl->bpg = bpg;
  pl->n_bgroups = (B + bpg - 1) / bpg;
  pl->cgroups = cgroups;
  pl->tickets_off = kWsHeader;
  pl->partials_off = decode_ticket_region_bytes(B, a->Hkv * cgroups);
  pl->ws_bytes = pl->partials_off +
                 sizeof(float) * (size_t)B * a->Hkv * pl->n_splits * g * a->M * kPartialStride;
  return VQKV_OK;
}

vqkv_status validate_encode(const vqkv_encode_args* a) {
  if (a == nullptr) return VQKV_ERR_INVALID_ARG;
  if (!is_code_mode(a->mode)) return VQKV_ERR_UNSUPPORTED;
  if (a->role != VQKV_ROLE_K && a->role != VQKV_ROLE_V) return VQKV_ERR_INVALID_ARG;
  if (a->head_dim != 128) return VQKV_ERR_UNSUPPORTED;
  if (a->B < 0 || a->Hkv < 1 || a->n_rows < 0 || a->cap_len < 1) return VQKV_ERR_INVALID_ARG;
  if (a->B == 0 || a->n_rows == 0) return VQKV_OK;
  if (!a->x || !a->pos || !a->codebook || !a->codes) return VQKV_ERR_INVALID_ARG;
  if (a->role == VQKV_ROLE_K && !a->s) return VQKV_ERR_INVALID_ARG;
  if (!aligned(a->x, 8) || !aligned(a->codebook, 16) || !aligned(a->pos, 4) ||
      (a->role == VQKV_ROLE_K && !aligned(a->s, 16)) || (a->near_tie_count && !aligned(a->near_tie_count, 8)) ||
      (a->error_flags && !aligned(a->error_flags, 4)))
    return VQKV_ERR_INVALID_ARG;
  if ((long long)a->B * a->n_rows > 0x7fffffffLL) return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

PlanInput plan_input(const vqkv_decode_args* a) {
  return PlanInput{a->mode, a->B, a->Hq, a->Hkv, a->max_seq_len, a->num_splits};
}

vqkv_status validate_fp16(const vqkv_fp16_decode_args* a, bool sizes_only) {
  if (a == nullptr) return VQKV_ERR_INVALID_ARG;
  if (a->head_dim != 128) return VQKV_ERR_UNSUPPORTED;
  if (a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->cap_len < 1) return VQKV_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return VQKV_ERR_INVALID_ARG;
  if (a->Hq / a->Hkv > 8) return VQKV_ERR_UNSUPPORTED;
  if (a->max_seq_len < 0 || a->max_seq_len > a->cap_len) return VQKV_ERR_INVALID_ARG;
  if (a->num_splits < 0 || !std::isfinite(a->softmax_scale)) return VQKV_ERR_INVALID_ARG;
  if (sizes_only || a->B == 0) return VQKV_OK;
  if (!a->q || !a->k || !a->v || !a->seq_lens || !a->out) return VQKV_ERR_INVALID_ARG;
  if (!aligned(a->q, 4) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->seq_lens, 4) ||
      !aligned(a->out, 2))
    return VQKV_ERR_INVALID_ARG;
  return VQKV_OK;
}

PlanInput plan_input(const vqkv_fp16_decode_args* a) {
  return PlanInput{kModeFp16, a->B, a->Hq, a->Hkv, a->max_seq_len, a->num_splits};
}

}  // namespace

vqkv_status decode_validate(const vqkv_decode_args* a) { return validate_decode(a); }

namespace {
// Both decode entry points: ap == nullptr for vqkv_decode_attn.
vqkv_status decode_launch(const vqkv_decode_args* a, const vqkv_decode_append_args* ap, int M, void* stream,
                          const vqkv_paging* pg = nullptr, unsigned test_polls = 0);
vqkv_status encode_launch(const vqkv_encode_args* a, void* stream, const vqkv_paging* pg = nullptr);
}  // namespace

size_t decode_ticket_region_bytes(int B, int Hkv) {
  return round_up(kWsHeader + sizeof(unsigned) * (size_t)std::max(B, 1) * Hkv, 256);
}

}  // namespace vqkv

using namespace vqkv;

extern "C" {

size_t vqkv_code_bytes(int32_t mode, int32_t cap_len) {
  if (cap_len < 0) return 0;
  if (mode == VQKV_MODE_VQ2) return (size_t)((cap_len + 15) / 16) * 512;
  if (mode == VQKV_MODE_VQ15) return (size_t)((cap_len + 63) / 64) * 1536;
  if (mode == VQKV_MODE_VQ4) return (size_t)((cap_len + 15) / 16) * 1024;
  if (mode == VQKV_MODE_VQ3) return (size_t)((cap_len + 15) / 16) * 768;
  if (mode == VQKV_MODE_VQ125) return (size_t)((cap_len + 15) / 16) * 320;
  return 0;
}

size_t vqkv_decode_workspace_bytes(const vqkv_decode_args* a) {
  if (validate_decode_sizes(a) != VQKV_OK) return 0;
  DecodePlan pl;
  const PlanInput in = plan_input(a);
  if (plan_decode(&in, &pl) != VQKV_OK) return 0;
  return pl.ws_bytes;
}

int32_t vqkv_decode_num_splits(const vqkv_decode_args* a) {
  if (validate_decode_sizes(a) != VQKV_OK) return -1;
  DecodePlan pl;
  const PlanInput in = plan_input(a);
  if (plan_decode(&in, &pl) != VQKV_OK) return -1;
  return pl.n_splits;
}

int32_t vqkv_decode_kernel_count(const vqkv_decode_args* a) {
  if (validate_decode_sizes(a) != VQKV_OK) return -1;
  if (a->B == 0) return 0;
  DecodePlan pl;
  const PlanInput in = plan_input(a);
  if (plan_decode(&in, &pl) != VQKV_OK) return -1;
  return (pl.bpg > 1 && pl.n_splits > 1) ? 2 : 1;
}

vqkv_status vqkv_decode_attn(const vqkv_decode_args* a, void* stream) { return decode_launch(a, nullptr, 1, stream); }

vqkv_status vqkv_decode_attn_multi(const vqkv_decode_multi_args* am, void* stream) {
  if (am == nullptr || am->n_queries < 1) return VQKV_ERR_INVALID_ARG;
  return decode_launch(&am->decode, nullptr, am->n_queries, stream);
}

vqkv_status vqkv_decode_append(const vqkv_decode_append_args* ap, void* stream) {
  if (ap == nullptr) return VQKV_ERR_INVALID_ARG;
  return decode_launch(&ap->decode, ap, 1, stream);
}

}  // extern "C"

namespace vqkv {
namespace {

vqkv_status decode_launch(const vqkv_decode_args* a, const vqkv_decode_append_args* ap, int M, void* stream,
                          const vqkv_paging* pg, unsigned test_polls) {
  if (ap != nullptr && a->mode != VQKV_MODE_VQ2 && a->mode != VQKV_MODE_VQ4) return VQKV_ERR_UNSUPPORTED;
  vqkv_status st = validate_decode(a);
  if (st != VQKV_OK) return st;
  if (pg != nullptr) {
    st = validate_paging(pg, a->mode, a->cap_len);
    if (st != VQKV_OK) return st;
    if (a->B > 0 && (!pg->block_table || !aligned(pg->block_table, 4))) return VQKV_ERR_INVALID_ARG;
  }
  if (M > 64 || (long long)M * (a->Hq / a->Hkv) > 64) return VQKV_ERR_UNSUPPORTED;   // <= 8 column groups
  if (ap != nullptr) {
    if (a->B > 0 && (!ap->k_new || !ap->v_new || !aligned(ap->k_new, 8) || !aligned(ap->v_new, 8) ||
                     (ap->near_tie_count && !aligned(ap->near_tie_count, 8))))
      return VQKV_ERR_INVALID_ARG;
  }
  if (a->B == 0) return VQKV_OK;
  DecodePlan pl;
  PlanInput in = plan_input(a);
  in.M = M;
  // the fused append costs its CTA about 60 tiles of streaming (2-bit, one
  // CTA per SM); a split of at most the plain plan's size, so the workspace
  // of vqkv_decode_workspace_bytes still covers it
  if (ap != nullptr) in.credit_tiles = 60;
  st = plan_decode(&in, &pl);
  if (st != VQKV_OK) return st;
  if (a->workspace == nullptr || a->workspace_bytes < pl.ws_bytes) return VQKV_ERR_WORKSPACE;
  if (!aligned(a->workspace, 256)) return VQKV_ERR_INVALID_ARG;
  DecodeParams p;
  unsigned char* ws = static_cast<unsigned char*>(a->workspace);
  p.q = reinterpret_cast<const __half*>(a->q);
  p.kc = a->k_codes;
  p.vc = a->v_codes;
  p.seq_lens = a->seq_lens;
  p.kcb = reinterpret_cast<const __half*>(a->k_codebook);
  p.vcb = reinterpret_cast<const __half*>(a->v_codebook);
  p.s = a->s;
  p.out = reinterpret_cast<__half*>(a->out);
  p.err = reinterpret_cast<unsigned*>(ws);
  p.tickets = reinterpret_cast<unsigned*>(ws + pl.tickets_off);
  p.partials = reinterpret_cast<float*>(ws + pl.partials_off);
  p.stream_bytes = (long long)vqkv_code_bytes(a->mode, a->cap_len);
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.g = a->Hq / a->Hkv;
  p.M = M;
  p.ncols = M * p.g;
  p.max_seq_len = a->max_seq_len;
  p.n_splits = pl.n_splits;
  p.tps = pl.tps;
  p.bpg = pl.bpg;
  p.defer_merge = pl.bpg > 1 ? 1 : 0;
  p.flat = pl.flat;
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt(128.0f);
  p.qscale = scale * 1.4426950408889634f / std::sqrt(128.0f);
  if (ap != nullptr) {
    p.k_new = reinterpret_cast<const __half*>(ap->k_new);
    p.v_new = reinterpret_cast<const __half*>(ap->v_new);
    p.kc_w = const_cast<uint8_t*>(a->k_codes);
    p.vc_w = const_cast<uint8_t*>(a->v_codes);
    p.near_tie = ap->near_tie_count;
  }
  set_paging(p, pg, a->mode);
  if (test_polls > 0) {
    p.max_polls = test_polls;
    p.withhold_first_copy = 1;
  }
  p.cgroups = pl.cgroups;
  const dim3 grid(pl.n_splits, a->Hkv, pl.n_bgroups * pl.cgroups);
  if (launch_decode(a->mode, p, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return VQKV_ERR_CUDA;
  if (p.defer_merge && p.n_splits > 1 && launch_combine(p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VQKV_ERR_CUDA;
  return VQKV_OK;
}

}  // namespace
}  // namespace vqkv

extern "C" {

vqkv_status vqkv_encode(const vqkv_encode_args* a, void* stream) { return encode_launch(a, stream); }

vqkv_status vqkv_encode_paged(const vqkv_encode_args* a, const vqkv_paging* pg, void* stream) {
  if (pg == nullptr) return VQKV_ERR_INVALID_ARG;
  return encode_launch(a, stream, pg);
}

vqkv_status vqkv_test_decode_ring_timeout(const vqkv_decode_args* a, uint32_t max_polls, void* stream) {
  if (a == nullptr || a->mode != VQKV_MODE_VQ2) return a == nullptr ? VQKV_ERR_INVALID_ARG : VQKV_ERR_UNSUPPORTED;
  if (max_polls < 1 || max_polls > 4096) return VQKV_ERR_INVALID_ARG;
  return decode_launch(a, nullptr, 1, stream, nullptr, max_polls);
}

vqkv_status vqkv_decode_attn_paged(const vqkv_decode_args* a, const vqkv_paging* pg, void* stream) {
  if (pg == nullptr) return VQKV_ERR_INVALID_ARG;
  return decode_launch(a, nullptr, 1, stream, pg);
}

}  // extern "C"

namespace vqkv {
namespace {

vqkv_status encode_launch(const vqkv_encode_args* a, void* stream, const vqkv_paging* pg) {
  vqkv_status st = validate_encode(a);
  if (st != VQKV_OK) return st;
  if (pg != nullptr) {
    st = validate_paging(pg, a->mode, a->cap_len);
    if (st != VQKV_OK) return st;
    if (a->B > 0 && a->n_rows > 0 && (!pg->block_table || !aligned(pg->block_table, 4))) return VQKV_ERR_INVALID_ARG;
  }
  if (a->B == 0 || a->n_rows == 0) return st;
  DeviceInfo di;
  st = device_info(&di);
  if (st != VQKV_OK) return st;
  EncodeParams p;
  p.x = reinterpret_cast<const __half*>(a->x);
  p.pos = a->pos;
  p.s = a->s;
  p.cb = reinterpret_cast<const __half*>(a->codebook);
  p.codes = a->codes;
  p.near_tie = a->near_tie_count;
  p.err = a->error_flags;
  p.stream_bytes = (long long)vqkv_code_bytes(a->mode, a->cap_len);
  p.B = a->B;
  p.Hkv = a->Hkv;
  p.n_rows = a->n_rows;
  p.cap_len = a->cap_len;
  p.role = a->role;
  const long long rows = (long long)a->B * a->n_rows;   // per KV head
  // Few rows (a decode-step append): one row per CTA, its candidates split
  // over the CTA's warps, for latency.  Many rows: one row per warp.
  const bool split_rows = rows * a->Hkv * encode_warps_per_cta() <= (long long)di.sms * 8;
  int blocks_x;
  if (split_rows) {
    blocks_x = (int)rows;
  } else {
    const long long want = (rows + encode_warps_per_cta() - 1) / encode_warps_per_cta();
    // every mode but 4 bit: persistent tensor-memory CTAs over tiles of 8 or
    // 4 rows, one wave; 4 bit: one warp per row, 4 waves
    const int waves = a->mode == VQKV_MODE_VQ4 ? 4 : 1;
    long long cap = ((long long)di.sms * di.encode_bpsm[a->mode] * waves + a->Hkv - 1) / a->Hkv;
    if (cap < 1) cap = 1;
    blocks_x = (int)std::min(want, cap);
  }
  set_paging(p, pg, a->mode);
  if (launch_encode(a->mode, p, blocks_x, split_rows, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VQKV_ERR_CUDA;
  return VQKV_OK;
}

}  // namespace
}  // namespace vqkv

extern "C" {

size_t vqkv_fp16_decode_workspace_bytes(const vqkv_fp16_decode_args* a) {
  if (validate_fp16(a, true) != VQKV_OK) return 0;
  DecodePlan pl;
  const PlanInput in = plan_input(a);
  if (plan_decode(&in, &pl) != VQKV_OK) return 0;
  return pl.ws_bytes;
}

vqkv_status vqkv_decode_attn_fp16(const vqkv_fp16_decode_args* a, void* stream) {
  vqkv_status st = validate_fp16(a, false);
  if (st != VQKV_OK || a->B == 0) return st;
  DecodePlan pl;
  const PlanInput in = plan_input(a);
  st = plan_decode(&in, &pl);
  if (st != VQKV_OK) return st;
  if (a->workspace == nullptr || a->workspace_bytes < pl.ws_bytes) return VQKV_ERR_WORKSPACE;
  if (!aligned(a->workspace, 256)) return VQKV_ERR_INVALID_ARG;
  unsigned char* ws = static_cast<unsigned char*>(a->workspace);
  DecodeParams p{};
  p.q = reinterpret_cast<const __half*>(a->q);
  p.kc = reinterpret_cast<const uint8_t*>(a->k);
  p.vc = reinterpret_cast<const uint8_t*>(a->v);
  p.seq_lens = a->seq_lens;
  p.out = reinterpret_cast<__half*>(a->out);
  p.err = reinterpret_cast<unsigned*>(ws);
  p.tickets = reinterpret_cast<unsigned*>(ws + pl.tickets_off);
  p.partials = reinterpret_cast<float*>(ws + pl.partials_off);
  p.stream_bytes = (long long)a->cap_len * 256;
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.g = a->Hq / a->Hkv;
  p.M = 1;
  p.ncols = p.g;
  p.max_seq_len = a->max_seq_len;
  p.n_splits = pl.n_splits;
  p.tps = pl.tps;
  p.bpg = pl.bpg;
  p.defer_merge = pl.bpg > 1 ? 1 : 0;
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt(128.0f);
  p.qscale = scale * 1.4426950408889634f;
  const dim3 grid(pl.n_splits, a->Hkv, pl.n_bgroups);
  if (launch_decode_fp16(p, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return VQKV_ERR_CUDA;
  if (p.defer_merge && p.n_splits > 1 && launch_combine(p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VQKV_ERR_CUDA;
  return VQKV_OK;
}

const char* vqkv_status_string(vqkv_status s) {
  switch (s) {
    case VQKV_OK: return "ok";
    case VQKV_ERR_INVALID_ARG: return "invalid argument";
    case VQKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case VQKV_ERR_WORKSPACE: return "workspace missing or too small";
    case VQKV_ERR_CUDA: return "CUDA error";
    case VQKV_ERR_NO_DEVICE: return "no usable CUDA device";
  }
  return "unknown status";
}

}  // extern "C"
