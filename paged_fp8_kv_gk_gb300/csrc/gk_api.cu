// gk_api.cu -- extern "C" entry points declared in include/gk.h: argument
// validation, workspace layout and kernel launches.  No allocation.
#include <cuda_runtime.h>
#include <string.h>

#include "gk_internal.h"
#include "../../include/gk_testing.h"

namespace gk {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by all entry points.  Returns GK_OK, GK_ERR_INVALID_ARG
// (inconsistent) or GK_ERR_UNSUPPORTED (valid but outside version 1).
static gk_status check_shape(const gk_shape* s) {
  if (!s) return GK_ERR_INVALID_ARG;
  if (s->num_layers < 2 || (s->num_layers & 1) || s->batch < 1 || s->num_q_heads < 1 ||
      s->num_kv_heads < 1 || s->head_dim < 2 || s->block_size < 2 || (s->block_size & 1) ||
      s->num_blocks < 1 || s->window < 1 || s->max_blocks_full < 1 || s->max_blocks_swa < 1 ||
      s->num_q_heads % s->num_kv_heads != 0)
    return GK_ERR_INVALID_ARG;
  if (s->num_layers > 2 * kMaxGroups || s->batch > kMaxBatch || s->head_dim != kHeadDim ||
      s->num_q_heads / s->num_kv_heads != kGroup ||
      !(s->block_size == 16 || (s->block_size % kStageTok == 0 && s->block_size <= 1024)))
    return GK_ERR_UNSUPPORTED;
  // the trimmed window row must hold every block a window can touch
  const int64_t need_swa = (int64_t(s->window) + s->block_size - 1 + s->block_size - 1) / s->block_size;
  if (s->max_blocks_swa < need_swa) return GK_ERR_INVALID_ARG;
  // flat slots (block * B + offset) are int32
  if (int64_t(s->num_blocks) * s->block_size > INT32_MAX) return GK_ERR_UNSUPPORTED;
  if (int64_t(s->max_blocks_full) * s->block_size > INT32_MAX / 2) return GK_ERR_UNSUPPORTED;
  return GK_OK;
}

static int64_t recommended_cap(const gk_shape& s) {
  const int64_t max_tok = int64_t(s.max_blocks_full) * s.block_size;
  if (max_tok <= kMinSplit) return 0;
  const int64_t per_row = (max_tok + kMinSplit - 1) / kMinSplit;
  const int64_t a = int64_t(s.batch) * (per_row < kMaxSplitsPerRow ? per_row : kMaxSplitsPerRow);
  const int64_t b = 2 * int64_t(s.batch) + 256;
  return a < b ? a : b;
}

// The cache descriptor -> per-group K and V base pointers.  Exactly one of
// the two forms must be present ("Kernel contract": the kernel asserts it).
static gk_status resolve_kv(const gk_shape& s, const gk_kv_cache* kv, uint8_t** kb, uint8_t** vb,
                            int* k_packed) {
  if (!kv) return GK_ERR_INVALID_ARG;
  const bool per_group = kv->k_bufs != nullptr || kv->v_bufs != nullptr;
  const bool stacked = kv->k_cache != nullptr || kv->v_cache != nullptr;
  if (per_group == stacked) return GK_ERR_INVALID_ARG;
  if (kv->k_layout != GK_K_PACKED && kv->k_layout != GK_K_PLAIN) return GK_ERR_INVALID_ARG;
  const int groups = s.num_layers / 2;
  if (per_group) {
    if (!kv->k_bufs || !kv->v_bufs) return GK_ERR_INVALID_ARG;
    for (int j = 0; j < groups; ++j) {
      if (!kv->k_bufs[j] || !kv->v_bufs[j] || !aligned16(kv->k_bufs[j]) ||
          !aligned16(kv->v_bufs[j]))
        return GK_ERR_INVALID_ARG;
      kb[j] = static_cast<uint8_t*>(kv->k_bufs[j]);
      vb[j] = static_cast<uint8_t*>(kv->v_bufs[j]);
    }
  } else {
    if (!kv->k_cache || !kv->v_cache || !aligned16(kv->k_cache) || !aligned16(kv->v_cache))
      return GK_ERR_INVALID_ARG;
    // one half of a group buffer: a multiple of 16 bytes (D = 64), so every
    // group's base stays 16-byte aligned
    const int64_t half = int64_t(s.num_blocks) * s.num_kv_heads * s.block_size * s.head_dim;
    for (int j = 0; j < groups; ++j) {
      kb[j] = static_cast<uint8_t*>(kv->k_cache) + int64_t(j) * half;
      vb[j] = static_cast<uint8_t*>(kv->v_cache) + int64_t(j) * half;
    }
  }
  *k_packed = kv->k_layout == GK_K_PACKED ? 1 : 0;
  return GK_OK;
}

static int64_t cmax_of(const gk_shape& s) { return int64_t(s.batch) * kMaxSplitsPerRow; }

WsLayout ws_layout(const gk_shape& s, size_t ws_bytes) {
  WsLayout L;
  const int64_t planes = int64_t(s.num_layers / 2) * s.num_kv_heads;
  const size_t rec = size_t(kPartialFloats) * sizeof(float);
  // fixed part, with the entry list sized for `cap` extra entries below
  size_t off = 0;
  L.hdr = off;
  off = align256(off + kHdrWords * sizeof(int32_t));
  const size_t after_hdr = off;
  auto place = [&](int64_t cap) {
    size_t o = after_hdr;
    L.edesc = o;  // full-layer entries (at most batch + cap), then one window entry per row
    o = align256(o + size_t(2 * s.batch + cap) * sizeof(int4));
    L.zero_list = o;
    o = align256(o + size_t(s.batch) * sizeof(int32_t));
    L.part_base = o;
    o = align256(o + size_t(s.batch) * sizeof(int32_t));
    L.split_rows = o;
    o = align256(o + size_t(s.batch) * sizeof(int32_t));
    L.partials = o;
    o = align256(o + size_t(cap) * size_t(planes) * rec);
    L.total = o;
    L.cap = cap;
    L.max_entries = s.batch + cap;
  };
  if (ws_bytes == 0) {
    place(recommended_cap(s));
    return L;
  }
  place(0);
  const size_t fixed = L.total;
  int64_t cap = 0;
  if (ws_bytes > fixed + 512)
    cap = int64_t((ws_bytes - fixed - 512) / (size_t(planes) * rec + sizeof(int4)));
  // the estimate above can fall one record short (alignment slack): start
  // two above it and step down to the largest capacity that fits
  cap = cap + 2 < cmax_of(s) ? cap + 2 : cmax_of(s);
  place(cap);
  while (cap > 0 && L.total > ws_bytes) place(--cap);
  return L;
}

}  // namespace gk

using namespace gk;

extern "C" {

const char* gk_status_str(gk_status st) {
  switch (st) {
    case GK_OK: return "GK_OK";
    case GK_ERR_INVALID_ARG: return "GK_ERR_INVALID_ARG";
    case GK_ERR_UNSUPPORTED: return "GK_ERR_UNSUPPORTED";
    case GK_ERR_WORKSPACE: return "GK_ERR_WORKSPACE";
    case GK_ERR_CUDA: return "GK_ERR_CUDA";
    case GK_ERR_DEVICE_BOUNDS: return "GK_ERR_DEVICE_BOUNDS";
    case GK_ERR_BUDGET: return "GK_ERR_BUDGET";
  }
  return "GK_ERR_UNKNOWN";
}

int32_t gk_abi_version(void) { return 3; }

gk_status gk_kv_append(const gk_shape* shape, const void* k_new, const void* v_new,
                       const float* cos, const float* sin, const float* k_scale,
                       const float* v_scale, const int32_t* upd_full, const int32_t* upd_swa,
                       const uint8_t* active, const gk_kv_cache* kv, void* stream) {
  gk_status st = check_shape(shape);
  if (st != GK_OK) return st;
  if (!k_new || !v_new || !cos || !sin || !k_scale || !v_scale || !upd_full || !upd_swa ||
      !active)
    return GK_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(cos) || !aligned16(sin))
    return GK_ERR_INVALID_ARG;
  AppendParams p;
  memset(&p, 0, sizeof(p));
  st = resolve_kv(*shape, kv, p.kb, p.vb, &p.k_packed);
  if (st != GK_OK) return st;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.cosb = cos;
  p.sinb = sin;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.upd_full = upd_full;
  p.upd_swa = upd_swa;
  p.active = active;
  p.NL = shape->num_layers;
  p.Bt = shape->batch;
  p.Hkv = shape->num_kv_heads;
  p.B = shape->block_size;
  p.nb = shape->num_blocks;
  return launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GK_OK : GK_ERR_CUDA;
}

size_t gk_attn_workspace_bytes(const gk_shape* shape, const int32_t* host_positions) {
  (void)host_positions;
  if (check_shape(shape) != GK_OK) return 0;
  return ws_layout(*shape, 0).total;
}

size_t gk_attn_workspace_min_bytes(const gk_shape* shape) {
  if (check_shape(shape) != GK_OK) return 0;
  WsLayout L = ws_layout(*shape, 1);  // smallest layout: no partial capacity
  return L.total;
}

}  // extern "C"

namespace gk {

struct AppendInputs {
  const void* k_new;
  const void* v_new;
  const int32_t* upd_full;
  const int32_t* upd_swa;
};

// Validation and launch shared by gk_decode_attn_stack and gk_decode_step
// (app != nullptr: gk_decode_step, whose planner grid also appends).
static gk_status decode_attention(const gk_shape* shape, const void* q, const gk_kv_cache* kv,
                                  const float* k_scale, const float* v_scale,
                                  const float* cos, const float* sin, const int32_t* bt_full,
                                  const int32_t* bt_swa, const int32_t* pos, const int32_t* pos_w,
                                  const uint8_t* active, const float* sinks, void* out,
                                  float* out_f32, void* workspace, size_t ws_bytes, void* stream,
                                  const AppendInputs* app, int force_split_log = -1) {
  gk_status st = check_shape(shape);
  if (st != GK_OK) return st;
  if (!q || !k_scale || !v_scale || !cos || !sin || !bt_full || !bt_swa ||
      !pos || !pos_w || !active || !out)
    return GK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (out_f32 && !aligned16(out_f32)) || !aligned16(cos) ||
      !aligned16(sin) || (reinterpret_cast<uintptr_t>(sinks) & 3u))
    return GK_ERR_INVALID_ARG;
  if (app && (!app->k_new || !app->v_new || !app->upd_full || !app->upd_swa ||
              !aligned16(app->k_new) || !aligned16(app->v_new)))
    return GK_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return GK_ERR_WORKSPACE;
  const WsLayout L = ws_layout(*shape, ws_bytes);
  if (L.total > ws_bytes) return GK_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  AttnParams p;
  memset(&p, 0, sizeof(p));
  {
    uint8_t* kb[kMaxGroups];
    uint8_t* vb[kMaxGroups];
    st = resolve_kv(*shape, kv, kb, vb, &p.k_packed);
    if (st != GK_OK) return st;
    for (int j = 0; j < shape->num_layers / 2; ++j) {
      p.kb[j] = kb[j];
      p.vb[j] = vb[j];
    }
  }
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.out_f32 = out_f32;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.cosb = cos;
  p.sinb = sin;
  p.sinks = sinks;
  p.bt_full = bt_full;
  p.bt_swa = bt_swa;
  p.hdr = reinterpret_cast<const int32_t*>(ws + L.hdr);
  p.queue = reinterpret_cast<int32_t*>(ws + L.hdr) + kHdrQueue;
  p.edesc = reinterpret_cast<const int4*>(ws + L.edesc);
  p.zero_list = reinterpret_cast<const int32_t*>(ws + L.zero_list);
  p.part_base = reinterpret_cast<const int32_t*>(ws + L.part_base);
  p.split_rows = reinterpret_cast<const int32_t*>(ws + L.split_rows);
  p.partials = reinterpret_cast<float*>(ws + L.partials);
  p.cap = L.cap;
  p.NL = shape->num_layers;
  p.Bt = shape->batch;
  p.Hq = shape->num_q_heads;
  p.Hkv = shape->num_kv_heads;
  p.B = shape->block_size;
  p.nb = shape->num_blocks;
  p.W = shape->window;
  p.MBF = shape->max_blocks_full;
  p.MBS = shape->max_blocks_swa;
  p.fd_planes = make_fastdiv(uint32_t(shape->num_layers / 2) * uint32_t(shape->num_kv_heads));
  p.fd_hkv = make_fastdiv(uint32_t(shape->num_kv_heads));
  p.fd_nl = make_fastdiv(uint32_t(shape->num_layers));
  p.fd_b = make_fastdiv(uint32_t(shape->block_size));

  PlanParams pl;
  memset(&pl, 0, sizeof(pl));
  pl.pos = pos;
  pl.pos_w = pos_w;
  pl.active = active;
  pl.hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  pl.edesc = reinterpret_cast<int4*>(ws + L.edesc);
  pl.zero_list = reinterpret_cast<int32_t*>(ws + L.zero_list);
  pl.part_base = reinterpret_cast<int32_t*>(ws + L.part_base);
  pl.split_rows = reinterpret_cast<int32_t*>(ws + L.split_rows);
  pl.cap = L.cap;
  pl.NL = shape->num_layers;
  pl.Bt = shape->batch;
  pl.Hkv = shape->num_kv_heads;
  pl.W = shape->window;
  pl.max_tokens_full = shape->max_blocks_full * shape->block_size;
  pl.max_tokens_swa = shape->max_blocks_swa * shape->block_size;
  pl.force_split_log = force_split_log;
  AppendParams ap;
  if (app) {
    // gk_decode_step: the append runs in the planner's grid
    memset(&ap, 0, sizeof(ap));
    ap.k_new = static_cast<const uint16_t*>(app->k_new);
    ap.v_new = static_cast<const uint16_t*>(app->v_new);
    ap.cosb = cos;
    ap.sinb = sin;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.upd_full = app->upd_full;
    ap.upd_swa = app->upd_swa;
    ap.active = active;
    for (int j = 0; j < shape->num_layers / 2; ++j) {
      ap.kb[j] = const_cast<uint8_t*>(p.kb[j]);
      ap.vb[j] = const_cast<uint8_t*>(p.vb[j]);
    }
    ap.k_packed = p.k_packed;
    ap.NL = shape->num_layers;
    ap.Bt = shape->batch;
    ap.Hkv = shape->num_kv_heads;
    ap.B = shape->block_size;
    ap.nb = shape->num_blocks;
  }
  return launch_attention(pl, p, static_cast<cudaStream_t>(stream), app ? &ap : nullptr) ==
                 cudaSuccess
             ? GK_OK
             : GK_ERR_CUDA;
}

}  // namespace gk

extern "C" {

gk_status gk_decode_attn_stack(const gk_shape* shape, const void* q, const gk_kv_cache* kv,
                               const float* k_scale, const float* v_scale,
                               const float* cos, const float* sin, const int32_t* bt_full,
                               const int32_t* bt_swa, const int32_t* pos, const int32_t* pos_w,
                               const uint8_t* active, const float* sinks, void* out,
                               float* out_f32, void* workspace, size_t ws_bytes, void* stream) {
  return decode_attention(shape, q, kv, k_scale, v_scale, cos, sin, bt_full, bt_swa, pos, pos_w,
                          active, sinks, out, out_f32, workspace, ws_bytes, stream, nullptr);
}

gk_status gk_decode_step(const gk_shape* shape, const void* q, const void* k_new,
                         const void* v_new, const float* cos, const float* sin,
                         const float* k_scale, const float* v_scale, const int32_t* upd_full,
                         const int32_t* upd_swa, const int32_t* bt_full, const int32_t* bt_swa,
                         const int32_t* pos, const int32_t* pos_w, const uint8_t* active,
                         const float* sinks, const gk_kv_cache* kv, void* out, float* out_f32,
                         void* workspace, size_t ws_bytes, void* stream) {
  const AppendInputs app = {k_new, v_new, upd_full, upd_swa};
  return decode_attention(shape, q, kv, k_scale, v_scale, cos, sin, bt_full, bt_swa, pos, pos_w,
                          active, sinks, out, out_f32, workspace, ws_bytes, stream, &app);
}

gk_status gk_kv_budget(uint64_t total_bytes, uint64_t used_bytes, double gmu, double cap_fraction,
                       double min_budget_gib, const gk_shape* shape, uint64_t* available_bytes,
                       int64_t* num_blocks) {
  if (!available_bytes || (shape && !num_blocks)) return GK_ERR_INVALID_ARG;
  if (!(gmu > 0.0 && gmu <= 1.0) || !(cap_fraction > 0.0 && cap_fraction <= 1.0) ||
      !(min_budget_gib >= 0.0))
    return GK_ERR_INVALID_ARG;
  // integer truncation of the double products, as the page's int() does
  const uint64_t total_budget = uint64_t(double(total_bytes) * gmu);
  const uint64_t kv_budget = total_budget > used_bytes ? total_budget - used_bytes : 0;
  const uint64_t cap = uint64_t(double(total_budget) * cap_fraction);
  const uint64_t available = kv_budget < cap ? kv_budget : cap;
  *available_bytes = available;
  bool too_small = double(available) < min_budget_gib * 1073741824.0;
  if (shape) {
    if (shape->num_layers < 2 || (shape->num_layers & 1) || shape->num_kv_heads < 1 ||
        shape->block_size < 1 || shape->head_dim < 1)
      return GK_ERR_INVALID_ARG;
    const uint64_t per_block = uint64_t(shape->num_layers / 2) * 2 * uint64_t(shape->num_kv_heads) *
                               uint64_t(shape->block_size) * uint64_t(shape->head_dim);
    *num_blocks = int64_t(available / per_block);
    too_small = too_small || *num_blocks < 2;
  }
  return too_small ? GK_ERR_BUDGET : GK_OK;
}

gk_status gk_kv_regions(const gk_shape* shape, void* const* layer_k, void* const* layer_v,
                        gk_kv_region* out, int32_t capacity, int32_t* count) {
  const gk_status st = check_shape(shape);
  if (st != GK_OK) return st;
  if (!layer_k || !layer_v || !count || capacity < 0 || (capacity > 0 && !out))
    return GK_ERR_INVALID_ARG;
  const uint64_t block_len =
      uint64_t(shape->num_kv_heads) * uint64_t(shape->block_size) * uint64_t(shape->head_dim);
  const uint64_t length = uint64_t(shape->num_blocks) * block_len;
  const void* seen[2 * 2 * kMaxGroups];
  int n = 0;
  for (int i = 0; i < shape->num_layers; ++i) {
    for (int half = 0; half < 2; ++half) {
      const void* a = half ? layer_v[i] : layer_k[i];
      if (!a || !aligned16(a)) {
        *count = 0;
        return GK_ERR_INVALID_ARG;
      }
      bool dup = false;
      for (int k = 0; k < n && !dup; ++k) dup = seen[k] == a;
      if (dup) continue;
      if (n < capacity) {
        out[n].base = const_cast<void*>(a);
        out[n].length = length;
        out[n].block_len = block_len;
      }
      seen[n++] = a;
    }
  }
  *count = n;
  return n > capacity ? GK_ERR_INVALID_ARG : GK_OK;
}

gk_status gk_kv_ingest(const gk_kv_region* regions, int32_t n_regions, const int32_t* dst_region,
                       const int32_t* dst_block, int64_t n, const void* src, void* stream) {
  if (n < 0) return GK_ERR_INVALID_ARG;
  if (n == 0) return GK_OK;
  if (!regions || n_regions < 1 || n_regions > kMaxRegions || !dst_region || !dst_block || !src ||
      !aligned16(src) || (reinterpret_cast<uintptr_t>(dst_region) & 3u) ||
      (reinterpret_cast<uintptr_t>(dst_block) & 3u))
    return GK_ERR_INVALID_ARG;
  IngestParams p;
  memset(&p, 0, sizeof(p));
  const uint64_t block_len = regions[0].block_len;
  if (block_len == 0 || (block_len & 15u) || block_len > (uint64_t(1) << 40))
    return GK_ERR_INVALID_ARG;
  for (int r = 0; r < n_regions; ++r) {
    const gk_kv_region& g = regions[r];
    if (g.block_len != block_len || !g.base || !aligned16(g.base) || g.length % block_len)
      return GK_ERR_INVALID_ARG;
    p.base[r] = static_cast<uint8_t*>(g.base);
    p.nblocks[r] = int64_t(g.length / block_len);
  }
  // The source must be memory the device can address: device memory, or host
  // memory that is pinned and mapped (translated to its device address).
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, src) != cudaSuccess) {
    cudaGetLastError();
    return GK_ERR_INVALID_ARG;
  }
  const void* dsrc = nullptr;
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    dsrc = src;
  } else if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    dsrc = a.devicePointer;
  } else {
    return GK_ERR_INVALID_ARG;
  }
  p.src = static_cast<const uint8_t*>(dsrc);
  p.dst_region = dst_region;
  p.dst_block = dst_block;
  p.n = n;
  p.block_len = int64_t(block_len);
  p.n_regions = n_regions;
  return launch_ingest(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GK_OK : GK_ERR_CUDA;
}

gk_status gk_di_blocks(int64_t num_tokens, int32_t block_size, int32_t window,
                       int64_t* full_count, int64_t* swa_first, int64_t* swa_count) {
  if (num_tokens < 1 || block_size < 1 || window < 1 || !full_count || !swa_first || !swa_count)
    return GK_ERR_INVALID_ARG;
  // both engines operate at N - 1: transferred keys are 0 .. N-2
  const int64_t last = num_tokens - 2;
  *full_count = (num_tokens - 1 + block_size - 1) / block_size;
  const int64_t lo = num_tokens - window > 0 ? num_tokens - window : 0;  // window of N - 1
  *swa_first = lo / block_size;
  *swa_count = last >= lo ? last / block_size - *swa_first + 1 : 0;
  return GK_OK;
}

gk_status gk_e4m3_quantize(const float* x, float scale, uint8_t* codes, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !codes))) return GK_ERR_INVALID_ARG;
  return launch_quantize(x, scale, codes, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GK_OK
             : GK_ERR_CUDA;
}

gk_status gk_selftest_decode_attn_split(const gk_shape* shape, const void* q,
                                        const gk_kv_cache* kv, const float* k_scale,
                                        const float* v_scale, const float* cos, const float* sin,
                                        const int32_t* bt_full, const int32_t* bt_swa,
                                        const int32_t* pos, const int32_t* pos_w,
                                        const uint8_t* active, const float* sinks, void* out,
                                        float* out_f32, void* workspace, size_t ws_bytes,
                                        int32_t split_tokens, void* stream) {
  int k = -1;
  for (int c = 0; c < 22; ++c)
    if ((kMinSplit << c) == split_tokens) k = c;
  if (k < 0) return GK_ERR_INVALID_ARG;
  return decode_attention(shape, q, kv, k_scale, v_scale, cos, sin, bt_full, bt_swa, pos, pos_w,
                          active, sinks, out, out_f32, workspace, ws_bytes, stream, nullptr, k);
}

gk_status gk_selftest_wait_timeout(uint64_t limit_ns, void* stream, uint32_t* bits) {
  if (!bits || limit_ns < 1000ull || limit_ns > 1000000000ull) return GK_ERR_INVALID_ARG;
  if (launch_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GK_ERR_CUDA;
  return gk_read_device_error(stream, bits, 1);
}

gk_status gk_read_device_error(void* stream, uint32_t* bits, int clear) {
  if (!bits) return GK_ERR_INVALID_ARG;
  *bits = 0;
  if (read_device_error(static_cast<cudaStream_t>(stream), bits, clear != 0) != cudaSuccess)
    return GK_ERR_CUDA;
  uint32_t ingest_bits = 0;
  if (read_ingest_error(&ingest_bits, clear != 0) != cudaSuccess) return GK_ERR_CUDA;
  *bits |= ingest_bits;
  return *bits ? GK_ERR_DEVICE_BOUNDS : GK_OK;
}

}  // extern "C"
