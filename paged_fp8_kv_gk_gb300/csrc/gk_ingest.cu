// gk_ingest.cu -- the DI landing copy ("GPT-OSS-120B giga-kernel decode",
// section "DI wiring (NIXL)": a transferred block b of a group buffer's K or V
// region lands at base + b * block_len, block_len = kv * block * d).
//
// Grid-stride over descriptors, one CTA per descriptor at a time: 16-byte
// streaming loads of the source block (each thread issues all of its loads
// before its stores), written to base[region] + block * block_len.  A
// descriptor out of range is skipped and reported in this file's own error
// word, which gk_read_device_error merges with the decode kernels' word.
#include <cuda_runtime.h>

#include "gk_internal.h"

namespace gk {

__device__ uint32_t g_ingest_error;

constexpr int kIngestThreads = 256;
constexpr int kIngestUnroll = 4;

__global__ void __launch_bounds__(kIngestThreads)
    ingest_kernel(const __grid_constant__ IngestParams p) {
  const int64_t chunks = p.block_len >> 4;
  for (int64_t d = blockIdx.x; d < p.n; d += gridDim.x) {
    const int32_t r = __ldg(p.dst_region + d);
    const int32_t b = __ldg(p.dst_block + d);
    if (r < 0 || r >= p.n_regions || b < 0 || b >= p.nblocks[r]) {
      if (threadIdx.x == 0) atomicOr(&g_ingest_error, GK_DEVERR_INGEST);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(p.src + d * p.block_len);
    uint4* dst = reinterpret_cast<uint4*>(p.base[r] + int64_t(b) * p.block_len);
    for (int64_t c0 = threadIdx.x; c0 < chunks; c0 += kIngestThreads * kIngestUnroll) {
      uint4 v[kIngestUnroll];
#pragma unroll
      for (int u = 0; u < kIngestUnroll; ++u) {
        const int64_t c = c0 + int64_t(u) * kIngestThreads;
        if (c < chunks) v[u] = __ldcs(src + c);
      }
#pragma unroll
      for (int u = 0; u < kIngestUnroll; ++u) {
        const int64_t c = c0 + int64_t(u) * kIngestThreads;
        if (c < chunks) __stcs(dst + c, v[u]);
      }
    }
  }
}

cudaError_t launch_ingest(const IngestParams& p, cudaStream_t st) {
  if (p.n <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t cap = int64_t(sms) * 8;
  const int64_t blocks = p.n < cap ? p.n : cap;
  ingest_kernel<<<unsigned(blocks), kIngestThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t read_ingest_error(uint32_t* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_ingest_error, sizeof(uint32_t));
  if (e != cudaSuccess || !clear) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_ingest_error, &zero, sizeof(uint32_t));
}

}  // namespace gk
