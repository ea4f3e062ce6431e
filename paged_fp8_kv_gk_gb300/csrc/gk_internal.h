// gk_internal.h -- parameter blocks, workspace layout and launchers shared by
// the host API (gk_api.cu) and the kernels (gk_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <vector_types.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gk.h"

namespace gk {

constexpr int kMaxGroups = 64;        // group buffers -> at most 128 layers
constexpr int kHeadDim = 64;          // D
constexpr int kGroup = 8;             // q heads per kv head (one MMA N tile)
constexpr int kMaxBatch = 8192;
constexpr int kStageTok = 32;         // tokens per pipeline stage
constexpr int kStageKBytes = kStageTok * kHeadDim;   // 2 KB of K codes
constexpr int kStageBytes = 2 * kStageKBytes;        // K + V
constexpr int kMinSplit = 512;        // smallest split-KV chunk, tokens (power of two)
constexpr int kMaxSplitsPerRow = 64;  // cap on chunks per (layer, row, kv head)
constexpr int kPartialFloats = 2 * kGroup + kGroup * kHeadDim;  // m[8], l[8], o[8][64]

// n / d for 0 <= n < 2^31 by multiply and shift (d >= 1 fixed per launch):
// shift = ceil(log2 d), mul = floor(2^32 (2^shift - d) / d) + 1,
// n / d = (umulhi(n, mul) + n) >> shift.
struct FastDiv {
  uint32_t mul, shift, d;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t s = 0;
  while ((uint64_t(1) << s) < d) ++s;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1;
  return FastDiv{uint32_t(m), s, d};
}
#ifdef __CUDACC__
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  const uint32_t hi = __umulhi(uint32_t(n), f.mul);
  return int((hi + uint32_t(n)) >> f.shift);
}
#endif

// Header words at the start of the attention workspace.
enum HdrWord {
  kHdrQueue = 0,        // work counter (atomic)
  kHdrNUnits = 1,       // units with a descriptor (full-layer, then sliding-window)
  kHdrNZero = 3,        // zero-fill units (inactive rows)
  kHdrSplit = 4,        // split length in tokens
  kHdrNEntries = 5,
  kHdrTotalSplits = 6,
  kHdrPieces = 7,       // pieces cut from chunks of long rows for the last wave (0: none)
  kHdrSplitRows = 9,    // rows with split-KV partials (entries of the split-row list)
  kHdrWords = 64
};

struct WsLayout {
  size_t hdr, edesc, zero_list, part_base, split_rows, partials, total;
  int64_t cap;          // partial records per (layer pair, kv head) plane
  int64_t max_entries;
};

// Offsets for a workspace of `ws_bytes` (0 -> the recommended size).
WsLayout ws_layout(const gk_shape& s, size_t ws_bytes);

struct AppendParams {
  const uint16_t* k_new;
  const uint16_t* v_new;
  const float* cosb;
  const float* sinb;
  const float* k_scale;
  const float* v_scale;
  const int32_t* upd_full;
  const int32_t* upd_swa;
  const uint8_t* active;
  uint8_t* kb[kMaxGroups];
  uint8_t* vb[kMaxGroups];
  int k_packed;  // 1: K through the packed view, 0: K laid out like V
  int NL, Bt, Hkv, B, nb;
};

struct PlanParams {
  const int32_t* pos;
  const int32_t* pos_w;
  const uint8_t* active;
  int32_t* hdr;
  int4* edesc;
  int32_t* zero_list;
  int32_t* part_base;
  int32_t* split_rows;  // rows with split-KV partials: b | ns << 16
  int64_t cap;
  int NL, Bt, Hkv, W, n_warps;
  int max_tokens_full, max_tokens_swa;  // table row lengths in tokens
  // test hook: split length kMinSplit << force_split_log (-1: the planner's
  // choice), still raised if a row would need more than kMaxSplitsPerRow
  // chunks or the records would not fit; no last-wave pieces
  int force_split_log;
};

// gk_decode_step's planner grid: CTA 0 plans, the others append.
struct PlanAppendParams {
  PlanParams plan;
  AppendParams app;
};

struct AttnParams {
  const uint16_t* q;
  uint16_t* out;
  float* out_f32;
  const uint8_t* kb[kMaxGroups];
  const uint8_t* vb[kMaxGroups];
  const float* k_scale;
  const float* v_scale;
  const float* cosb;
  const float* sinb;
  const float* sinks;  // [NL, Hq] attention-sink logits or nullptr
  const int32_t* bt_full;
  const int32_t* bt_swa;
  const int32_t* hdr;
  int32_t* queue;
  const int4* edesc;
  const int32_t* zero_list;
  const int32_t* part_base;
  const int32_t* split_rows;
  float* partials;
  int64_t cap;  // partial records per (layer pair, kv head) plane
  // 36 bytes unused: they keep the offsets of the fields below, on which the
  // attention kernel's measured speed depends
  uint8_t reserved[36];
  int k_packed;  // 1: K through the packed view, 0: K laid out like V
  int NL, Bt, Hq, Hkv, B, nb, W, MBF, MBS;
  FastDiv fd_planes, fd_hkv, fd_nl, fd_b;  // (NL/2)*Hkv, Hkv, NL, B
};

constexpr int kMaxRegions = 2 * kMaxGroups;

struct IngestParams {
  uint8_t* base[kMaxRegions];
  int64_t nblocks[kMaxRegions];
  const int32_t* dst_region;
  const int32_t* dst_block;
  const uint8_t* src;
  int64_t n;
  int64_t block_len;
  int n_regions;
};

// Launchers (gk_kernels.cu).  They return the launch status.
cudaError_t launch_append(const AppendParams& p, cudaStream_t st);
cudaError_t launch_quantize(const float* x, float scale, uint8_t* codes, int64_t n, cudaStream_t st);
// app: gk_decode_step's append, done in the planner's grid (or null).
cudaError_t launch_attention(const PlanParams& plan, const AttnParams& p, cudaStream_t st,
                             const AppendParams* app = nullptr);
// Resident warps of the persistent attention grid on the current device.
int attention_resident_warps();
cudaError_t read_device_error(cudaStream_t st, uint32_t* bits, bool clear);
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t st);
// gk_ingest.cu: the landing copy and its own device error word (read after
// the stream has been synchronised).
cudaError_t launch_ingest(const IngestParams& p, cudaStream_t st);
cudaError_t read_ingest_error(uint32_t* bits, bool clear);

}  // namespace gk
