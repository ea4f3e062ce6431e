// gk_kernels.cu -- sm_103a kernels of the stack-wide paged-FP8 decode step.
//
//   kv_append_kernel   RoPE(k) in IEEE fp32, / scale, E4M3 (RNE, satfinite),
//                      scatter into the packed K and plain V layouts.
//   plan_kernel        one CTA: split-KV chunk length, work-unit order
//                      (largest first), per-row split bookkeeping; for
//                      gk_decode_step, further CTAs of the same grid do the
//                      KV append beside it (plan_append_kernel).
//   attn_kernel        persistent: each warp takes (layer, row, kv head, split)
//                      units from an atomic counter, streams 32-token stages of
//                      K and V through a private ring of 1-D bulk copies, and
//                      runs QK^T and PV on the tensor cores (mma.sync m16n8k16,
//                      N = the 8 q heads of the GQA group) with an online
//                      softmax.  Split units write (m, l, o) partials.
//   combine_kernel     the split-KV (flash-decoding) combine: one warp per
//                      (row with partials, layer pair, kv head) merges them.
//
// Page references: "GPT-OSS-120B giga-kernel decode", sections "Kernel
// contract" (layer parity i % 2 selects table / index / position, buffer
// i / 2) and "KV-cache layout" (packed K view [.., block/2, d, 2], plain V).
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include "gk_device.cuh"
#include "gk_internal.h"

namespace gk {

__device__ uint32_t g_dev_error;

__device__ __forceinline__ void set_error(uint32_t bits) { atomicOr(&g_dev_error, bits); }

// 1/s when s is a power of two whose reciprocal is a normal float (then
// x * (1/s) is exactly the correctly rounded x / s for every x); 0 otherwise.
__device__ __forceinline__ float exact_reciprocal(float s) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t e = (u >> 23) & 0xffu;
  if ((u & 0x7fffffu) != 0 || e < 2 || e > 252) return 0.f;
  return __uint_as_float((u & 0x80000000u) | ((254u - e) << 23));
}

// x / s with IEEE round-to-nearest; r = exact_reciprocal(s) when nonzero.
__device__ __forceinline__ float div_scale(float x, float s, float r) {
  return r != 0.f ? x * r : __fdiv_rn(x, s);
}

// =========================================================================
// KV append
// =========================================================================
// One warp per (layer i, row b); kv heads in groups of 8.  Lane l rotates
// the pair (l, l + 32) of k and converts channels 2l, 2l + 1 of v.  All of a
// group's loads are issued before any of them is used (one memory round trip
// per group rather than a chain of dependent ones).  Used by the append kernel
// and by the append CTAs of gk_decode_step's planner launch; ib = i * Bt + b.
constexpr int kAppendHeads = 8;

__device__ __forceinline__ void append_row(const AppendParams& p, int64_t ib, int lane) {
  const int b = int(ib % p.Bt);
  const int i = int(ib / p.Bt);
  const uint16_t* kr = p.k_new + ib * p.Hkv * kHeadDim;
  const uint32_t* vr = reinterpret_cast<const uint32_t*>(p.v_new + ib * p.Hkv * kHeadDim);
  // layer parity: even = sliding window (upd_swa), odd = full (upd_full)
  const uint8_t act = p.active[b];
  const int32_t slot = (i & 1) ? p.upd_full[b] : p.upd_swa[b];
  const float c = p.cosb[b * (kHeadDim / 2) + lane];
  const float s = p.sinb[b * (kHeadDim / 2) + lane];
  const float ks = p.k_scale[i];
  const float vs = p.v_scale[i];
  for (int h0 = 0; h0 < p.Hkv; h0 += kAppendHeads) {
    const int nh = min(kAppendHeads, p.Hkv - h0);
    uint32_t kx[kAppendHeads], ky[kAppendHeads], vw[kAppendHeads];
#pragma unroll
    for (int k = 0; k < kAppendHeads; ++k) {
      if (k < nh) {
        kx[k] = kr[(h0 + k) * kHeadDim + lane];
        ky[k] = kr[(h0 + k) * kHeadDim + lane + 32];
        vw[k] = vr[(h0 + k) * (kHeadDim / 2) + lane];
      }
    }
    if (!act) return;
    if (slot < 0 || int64_t(slot) >= int64_t(p.nb) * p.B) {
      if (lane == 0) set_error(GK_DEVERR_SLOT);
      return;
    }
    const int64_t pb = slot / p.B;
    const int t = slot % p.B;
    const float kr_inv = exact_reciprocal(ks), vr_inv = exact_reciprocal(vs);
    // packed K: tokens 2p and 2p+1 interleaved per channel (channel e at byte
    // 2e of the pair row); plain K: laid out like V.  Either way a head's block
    // is B * D bytes.
    uint8_t* kbase = p.kb[i >> 1];
    uint8_t* kdst = p.k_packed
                        ? kbase + ((pb * p.Hkv + h0) * (p.B >> 1) + (t >> 1)) * (2 * kHeadDim) + (t & 1)
                        : kbase + ((pb * p.Hkv + h0) * p.B + t) * kHeadDim;
    const int estep = p.k_packed ? 2 : 1;
    uint8_t* vdst = p.vb[i >> 1] + ((pb * p.Hkv + h0) * p.B + t) * kHeadDim;
    const int64_t kstride = int64_t(p.B) * kHeadDim, vstride = int64_t(p.B) * kHeadDim;
#pragma unroll
    for (int k = 0; k < kAppendHeads; ++k) {
      if (k < nh) {
        const float x = __uint_as_float(kx[k] << 16);
        const float y = __uint_as_float(ky[k] << 16);
        // fixed fp32 sequence, every operation rounded on its own (no contraction)
        const float xr = __fsub_rn(__fmul_rn(x, c), __fmul_rn(y, s));
        const float yr = __fadd_rn(__fmul_rn(y, c), __fmul_rn(x, s));
        const uint32_t kc =
            f32x2_to_e4m3x2(div_scale(xr, ks, kr_inv), div_scale(yr, ks, kr_inv));
        kdst[k * kstride + estep * lane] = uint8_t(kc & 0xffu);
        kdst[k * kstride + estep * (lane + 32)] = uint8_t(kc >> 8);
        const uint32_t vc = f32x2_to_e4m3x2(div_scale(bf16lo_to_f32(vw[k]), vs, vr_inv),
                                            div_scale(bf16hi_to_f32(vw[k]), vs, vr_inv));
        reinterpret_cast<uint16_t*>(vdst + k * vstride)[lane] = uint16_t(vc);
      }
    }
  }
}

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendParams p) {
  // The decode-attention planner may launch now: it reads only positions and
  // the active mask, and waits for this grid before it exits.
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int64_t ib = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (ib >= int64_t(p.NL) * p.Bt) return;
  append_row(p, ib, lane);
}

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ x, float scale,
                                                       uint8_t* __restrict__ codes, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x * 2;
  const float r = exact_reciprocal(scale);
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 2; i < n; i += stride) {
    if (i + 1 < n) {
      const uint32_t c = f32x2_to_e4m3x2(div_scale(x[i], scale, r), div_scale(x[i + 1], scale, r));
      codes[i] = uint8_t(c & 0xffu);
      codes[i + 1] = uint8_t(c >> 8);
    } else {
      codes[i] = uint8_t(f32x2_to_e4m3x2(div_scale(x[i], scale, r), 0.f) & 0xffu);
    }
  }
}

// =========================================================================
// Planner (one CTA)
// =========================================================================
constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kUnitsPerWarp = 8;   // minimum work units per resident warp
constexpr int kMinPiece = 512;     // shortest piece cut from a chunk for the last wave
constexpr int kShortSplit = 1024;  // chunks this short ...
constexpr int kShortMerge = 8;     // ... are not chosen if a row would need more of them
constexpr int kSplitCands = 22;    // candidate split lengths kMinSplit << k
constexpr int kRemBuckets = 256;   // remainder size classes for the largest-first order

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ long long warp_sum64(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Work entries are int4 descriptors: {row b, t_begin, t_end, w} with
// w = s | ns << 16 | kind << 30 (kind 1 = sliding-window layer).  One entry
// covers the (layer pair, kv head) planes of one row's chunk: unit u is plane
// u % planes of entry u / planes.  Full-layer entries come first, largest
// first; then one sliding-window entry per active row; then zero-fill units
// (one per inactive row and layer).

// The planner's work, done by one CTA.
__device__ __forceinline__ void plan_body(const PlanParams& p) {
  extern __shared__ int32_t plan_sm[];
  int32_t* Ls = plan_sm;          // clamped context length per row (0 = no work)
  int32_t* Pw = plan_sm + p.Bt;   // window-frame position per row
  __shared__ long long s_units[kSplitCands], s_need[kSplitCands];
  __shared__ long long s_full[kSplitCands], s_remtok[kSplitCands];
  __shared__ int s_ne[kSplitCands], s_maxnf[kSplitCands];
  __shared__ int s_conv[3];  // chunks cut per eligible row, rows cutting one more, pieces
  __shared__ int s_erank[kPlanWarps];
  __shared__ long long s_red[3][kPlanWarps];
  __shared__ int s_bucket[kRemBuckets];
  __shared__ int4 s_scan[kPlanWarps];
  __shared__ int s_nsr[kPlanWarps];
  __shared__ int s_S_log;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int chunk = (p.Bt + kPlanThreads - 1) / kPlanThreads;
  const int b_lo = min(p.Bt, tid * chunk), b_hi = min(p.Bt, b_lo + chunk);

  long long tsum = 0;
  int lmax = 0, nact = 0;
  for (int b = b_lo; b < b_hi; ++b) {
    int L = 0;
    const int act = p.active[b], pos = p.pos[b];   // one round trip for all three
    Pw[b] = p.pos_w[b];
    if (act) {
      if (pos < 0) {
        set_error(GK_DEVERR_POS);
      } else {
        L = pos + 1;
        if (L > p.max_tokens_full) {
          set_error(GK_DEVERR_POS);
          L = p.max_tokens_full;
        }
        ++nact;
      }
    }
    Ls[b] = L;
    tsum += L;
    lmax = max(lmax, L);
  }
  for (int k = tid; k < kRemBuckets; k += kPlanThreads) s_bucket[k] = 0;
  tsum = warp_sum64(tsum);
  nact = warp_sum(nact);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(kFull, lmax, o));
  if (lane == 0) {
    s_red[0][wid] = tsum;
    s_red[1][wid] = lmax;
    s_red[2][wid] = nact;
  }
  __syncthreads();
  long long T = 0, NAct = 0;
  int Lmax = 0;
  for (int w = 0; w < kPlanWarps; ++w) {
    T += s_red[0][w];
    Lmax = max(Lmax, int(s_red[1][w]));
    NAct += s_red[2][w];
  }

  // unit counts and split-record needs of every candidate split length,
  // one candidate per warp at a time
  for (int k = wid; k < kSplitCands; k += kPlanWarps) {
    const int sh = 9 + k;  // log2 of kMinSplit << k
    const long long S = 1ll << sh;
    long long units = 0, need = 0, full = 0, remtok = 0;
    int ne = 0, maxnf = 0;
    for (int b = lane; b < p.Bt; b += 32) {
      const int L = Ls[b];
      if (L > 0) {
        const long long c = (L + S - 1) >> sh;
        const int nf = int(L >> sh);
        units += c;
        if (L > S) need += c;
        full += nf;
        remtok += L & (S - 1);
        ne += nf >= 2;
        maxnf = max(maxnf, nf);
      }
    }
    units = warp_sum64(units);
    need = warp_sum64(need);
    full = warp_sum64(full);
    remtok = warp_sum64(remtok);
    ne = warp_sum(ne);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxnf = max(maxnf, __shfl_xor_sync(kFull, maxnf, o));
    if (lane == 0) {
      s_units[k] = units;
      s_need[k] = need;
      s_full[k] = full;
      s_remtok[k] = remtok;
      s_ne[k] = ne;
      s_maxnf[k] = maxnf;
    }
  }
  __syncthreads();
  const int planes = (p.NL >> 1) * p.Hkv;
  const long long warps = max(1, p.n_warps);
  if (tid == 0) {
    // Split length S = kMinSplit << k.  Start near a quarter of one warp's
    // share of the full-layer work, then halve while there are fewer than
    // kUnitsPerWarp units per resident warp (uniform long rows need many
    // chunks; mixed rows balance through largest-first order).  Then cap the
    // chunks per row and fit the partial records into the workspace.
    const long long share = (T * planes) / (warps * 4);
    int k = 0;
    while (k < kSplitCands - 1 && ((long long)kMinSplit << k) < share) ++k;
    while (k > 0 && (s_units[k] + NAct) * planes < kUnitsPerWarp * warps) --k;
    // no short chunks that would give a row more than kShortMerge partials:
    // the per-unit cost of the extra partials outweighs the balance they buy
    while (k < kSplitCands - 1 && ((long long)kMinSplit << k) <= kShortSplit &&
           (Lmax - 1) / ((long long)kMinSplit << k) + 1 > kShortMerge)
      ++k;
    if (p.force_split_log >= 0) k = p.force_split_log;  // test hook: a fixed split length
    while (k < kSplitCands - 1 && ((long long)kMinSplit << k) * kMaxSplitsPerRow < Lmax) ++k;
    while (k < kSplitCands - 1 && s_need[k] > p.cap) ++k;
    s_S_log = k;
    // Last wave.  Equal chunks give full * planes units of one size; when
    // that is at least one wave but not a whole number of waves over the
    // warps and the smaller
    // units (remainders, window units) cannot fill the idle part of the last
    // wave, cut the last chunks of the rows with two or more of them into
    // p pieces (largest-first order runs them at the end), keeping whole
    // waves of full chunks.  Rows stay within kMaxSplitsPerRow chunks and
    // the partial records within the workspace.
    int conv_c = 0, conv_x = 0, conv_p = 0;
    const long long Sk = (long long)kMinSplit << k;
    const long long cunits = s_full[k] * planes;
    const long long q = cunits / warps, rem = cunits - q * warps;
    const long long gap = (warps - rem) * Sk;                    // idle token slots
    const long long small = (s_remtok[k] + NAct * p.W) * planes;  // work in smaller units
    if (p.force_split_log < 0 && q >= 1 && rem > 0 && small < gap && s_ne[k] > 0) {
      // cv chunks in all, spread over the eligible rows in row order (fewer
      // if a row would pass kMaxSplitsPerRow chunks or the records the
      // workspace holds)
      const long long cv = s_full[k] - (q * warps) / planes;
      for (int pp = int(min(8ll, Sk / kMinPiece)); pp >= 2; pp >>= 1) {
        const long long per_row = (kMaxSplitsPerRow - 1 - s_maxnf[k]) / (pp - 1);
        const long long room = (p.cap - s_need[k]) / (pp - 1);
        const long long cvp = min(cv, min(per_row * s_ne[k], room));
        if (cvp >= 1) {
          conv_c = int(cvp / s_ne[k]);
          conv_x = int(cvp - conv_c * s_ne[k]);
          conv_p = pp;
          break;
        }
      }
    }
    s_conv[0] = conv_c;
    s_conv[1] = conv_x;
    s_conv[2] = conv_p;
  }
  __syncthreads();
  const int conv_c = s_conv[0], conv_x = s_conv[1], conv_p = s_conv[2];
  // rank of this thread's first row among the rows with two or more full
  // chunks (the first conv_x of them cut one chunk more)
  int erank = 0;
  if (conv_p > 0) {
    int e = 0;
    for (int b = b_lo; b < b_hi; ++b) e += (Ls[b] >> (9 + s_S_log)) >= 2;
    int inc = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) s_erank[wid] = inc;
    __syncthreads();
    erank = inc - e;
    for (int w = 0; w < wid; ++w) erank += s_erank[w];
  }
  const int S_log = s_S_log;
  const int S_sh = 9 + S_log;  // S = 2^S_sh
  const long long S = 1ll << S_sh;
  static_assert(kMinSplit == 512, "split lengths are 2^(9 + k)");
  const int bshift = max(0, S_log + 9 - 8);  // remainder -> one of 256 classes

  // per-thread counts -> one packed exclusive scan: (full chunks, split
  // records, active rows, remainders)
  // a row's chunks: nf - cut full chunks, then cut * conv_p pieces, then the
  // remainder; split indices follow the keys
  const int piece_len = conv_p > 0 ? int(S) / conv_p : 0;
  const int piece_bucket = conv_p > 0 ? kRemBuckets - 1 - (piece_len >> bshift) : 0;
  auto cut_of = [&](int nf, int& rank) {
    if (conv_p == 0 || nf < 2) return 0;
    const int c = conv_c + (rank < conv_x ? 1 : 0);
    ++rank;
    return min(c, nf);
  };
  int4 cnt = make_int4(0, 0, 0, 0);
  int nsr = 0;  // rows with split-KV partials
  int rk = erank;
  for (int b = b_lo; b < b_hi; ++b) {
    const int L = Ls[b];
    if (L > 0) {
      const int nf = int(L >> S_sh), r = int(L & (S - 1)), cut = cut_of(nf, rk);
      const int ns = nf + cut * (conv_p - 1) + (r > 0);
      cnt.x += nf - cut;
      cnt.y += ns > 1 ? ns : 0;
      nsr += ns > 1;
      cnt.z += 1;
      if (r > 0) {
        cnt.w += 1;
        atomicAdd(&s_bucket[kRemBuckets - 1 - (r >> bshift)], 1);  // largest first
      }
      if (cut > 0) {
        cnt.w += cut * conv_p;
        atomicAdd(&s_bucket[piece_bucket], cut * conv_p);
      }
    }
  }
  int4 inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, inc.x, o), y = __shfl_up_sync(kFull, inc.y, o);
    const int z = __shfl_up_sync(kFull, inc.z, o), w = __shfl_up_sync(kFull, inc.w, o);
    if (lane >= o) {
      inc.x += x;
      inc.y += y;
      inc.z += z;
      inc.w += w;
    }
  }
  int nsr_inc = nsr;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, nsr_inc, o);
    if (lane >= o) nsr_inc += y;
  }
  if (lane == 31) {
    s_scan[wid] = inc;
    s_nsr[wid] = nsr_inc;
  }
  __syncthreads();
  int srp = nsr_inc - nsr, n_split_rows = 0;  // this thread's first slot in the split-row list
  for (int w = 0; w < kPlanWarps; ++w) {
    if (w < wid) srp += s_nsr[w];
    n_split_rows += s_nsr[w];
  }
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
  for (int w = 0; w < kPlanWarps; ++w) {
    const int4 v = s_scan[w];
    if (w < wid) {
      base.x += v.x;
      base.y += v.y;
      base.z += v.z;
      base.w += v.w;
    }
    tot.x += v.x;
    tot.y += v.y;
    tot.z += v.z;
    tot.w += v.w;
  }
  if (wid == 0) {  // bucket counts -> exclusive offsets: 8 buckets per lane, one warp scan
    constexpr int per = kRemBuckets / 32;
    int v[per], sum = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      v[k] = s_bucket[lane * per + k];
      sum += v[k];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    int acc = incl - sum;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      s_bucket[lane * per + k] = acc;
      acc += v[k];
    }
  }
  __syncthreads();
  int fp = base.x + inc.x - cnt.x;
  int sp = base.y + inc.y - cnt.y;
  int ap = base.z + inc.z - cnt.z;
  const int A = tot.x, TS = tot.y, NA = tot.z, R = tot.w;
  const int NEF = A + R;  // full-layer entries
  int ip = b_lo - ap;     // inactive rows before this thread's rows
  (void)R;

  rk = erank;
  for (int b = b_lo; b < b_hi; ++b) {
    const int L = Ls[b];
    if (L > 0) {
      const int nf = int(L >> S_sh), r = int(L & (S - 1)), cut = cut_of(nf, rk);
      const int ns = nf + cut * (conv_p - 1) + (r > 0);
      const int nk = nf - cut;  // full chunks kept
      for (int s = 0; s < nk; ++s)
        p.edesc[fp++] = make_int4(b, int(s * S), int((s + 1) * S), s | (ns << 16));
      if (cut > 0) {
        const int np = cut * conv_p;
        const int slot = atomicAdd(&s_bucket[piece_bucket], np);
        for (int i = 0; i < np; ++i) {
          const int t0 = int(nk * S) + i * piece_len;
          p.edesc[A + slot + i] = make_int4(b, t0, t0 + piece_len, (nk + i) | (ns << 16));
        }
      }
      if (r > 0) {
        const int slot = atomicAdd(&s_bucket[kRemBuckets - 1 - (r >> bshift)], 1);
        p.edesc[A + slot] = make_int4(b, int(nf * S), L, (ns - 1) | (ns << 16));
      }
      if (ns > 1) {
        p.part_base[b] = sp;
        sp += ns;
        p.split_rows[srp++] = b | (ns << 16);
      } else {
        p.part_base[b] = 0;
      }
      // sliding-window layer of this row: keys [max(0, pos_w - W + 1), pos_w]
      int pw = Pw[b];
      if (pw < 0 || pw >= p.max_tokens_swa) {
        set_error(GK_DEVERR_POS);
        pw = min(max(pw, 0), p.max_tokens_swa - 1);
      }
      p.edesc[NEF + ap++] = make_int4(b, max(0, pw - p.W + 1), pw + 1, (1 << 16) | (1 << 30));
    } else {
      p.part_base[b] = 0;
      p.zero_list[ip++] = b;
    }
  }
  if (tid == 0) {
    if (TS > p.cap) set_error(GK_DEVERR_PLAN);
    p.hdr[kHdrQueue] = p.n_warps;
    p.hdr[kHdrNUnits] = (NEF + NA) * planes;
    p.hdr[kHdrNZero] = (p.Bt - NA) * p.NL;
    p.hdr[kHdrSplit] = int(S);
    p.hdr[kHdrNEntries] = NEF + NA;
    p.hdr[kHdrTotalSplits] = TS;
    p.hdr[kHdrPieces] = conv_p > 0 ? (conv_c * s_ne[s_S_log] + conv_x) * conv_p : 0;
    p.hdr[kHdrSplitRows] = n_split_rows;
  }
  // This grid may have started while the kernel before it (the KV append)
  // was still running; it completes only after that kernel has, so the
  // attention grid that waits on this one also sees the appended KV.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams p) {
  // let the attention grid launch now; it waits for this grid before reading the plan
  asm volatile("griddepcontrol.launch_dependents;");
  plan_body(p);
}

// gk_decode_step: CTA 0 plans; the CTAs after it append the new token,
// warp w taking (layer, row) pairs w, w + warps, ...  The attention grid waits
// for this whole grid, so it reads the plan and the appended cache; the kernel
// before this grid must be complete before the cache is written.
__global__ void __launch_bounds__(kPlanThreads)
    plan_append_kernel(const __grid_constant__ PlanAppendParams p) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (blockIdx.x == 0) {
    plan_body(p.plan);
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t n_ib = int64_t(p.app.NL) * p.app.Bt;
  const int64_t warps = (int64_t(gridDim.x) - 1) * (kPlanThreads / 32);
  const int lane = threadIdx.x & 31;
  for (int64_t ib = (int64_t(blockIdx.x) - 1) * (kPlanThreads / 32) + (threadIdx.x >> 5);
       ib < n_ib; ib += warps)
    append_row(p.app, ib, lane);
}

// =========================================================================
// Decode attention (persistent)
// =========================================================================
constexpr int kWarps = 4;    // independent worker warps per CTA
constexpr int kStages = 3;   // ring depth per warp (stages of 32 tokens)
constexpr int kFifo = 6;     // unit descriptors in flight per warp (> kStages + 1)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per barrier wait
constexpr uint32_t kOnesF16x2 = 0x3C003C00u;        // (1.0, 1.0) in f16
constexpr float kLazyLog2 = 8.f;  // probabilities stay <= 2^8 between rescales

struct UnitDesc {
  int32_t kind;  // 1 = full layer, 2 = sliding-window layer
  int32_t layer, b, kvh, s, ns;
  int32_t t_begin, t_end;  // key range [t_begin, t_end) in the table's frame
  int32_t st_begin, n_st;  // 32-token stages covering the range
};

// q of the unit's 8 heads (bf16) followed by its row's cos and sin (fp32),
// fetched with the unit's first stage.
constexpr uint32_t kQBytes = kGroup * kHeadDim * 2;
constexpr uint32_t kRopeBytes = (kHeadDim / 2) * 4;
constexpr uint32_t kUnitHeadBytes = kQBytes + 2 * kRopeBytes;

// The FMA comparison path keeps q' in fp32 (rows padded so the eight heads
// fall in different banks) and one stage of P for the exchange between its
// token-per-lane and channel-per-lane phases.
constexpr int kQfStride = kHeadDim + 4;

// One per warp, laid out back to back: the 128-byte alignment keeps every
// warp's ring and q buffer on the 16-byte boundary bulk copies require.
template <bool kMma>
struct alignas(128) WarpSmemT {
  uint8_t ring[kStages][kStageBytes];
  uint8_t qbuf[kUnitHeadBytes];
  float qf[kMma ? 4 : kGroup * kQfStride];
  float pbuf[kMma ? 4 : kStageTok * kGroup];
  unsigned long long bar[kStages];
  const uint8_t* pu_base[2];  // the producer unit's K and V bases (its kv head's bytes)
  // the producer unit's first stage is copied from key lo, its last stage up
  // to key hi of their 32-key stages (its range rounded out to 8): lo | hi << 8
  int pu_trim;
  int4 e_next;             // work descriptor of the claimed unit (copied asynchronously)
  UnitDesc fifo[kFifo];
};
static_assert(sizeof(WarpSmemT<true>) % 128 == 0 && sizeof(WarpSmemT<false>) % 128 == 0,
              "warp areas must stay 128-byte aligned");
// 4 CTAs x 4 warps x 14 KB (+ 1 KB reserved per CTA) is the SM's 228 KB
static_assert(sizeof(WarpSmemT<true>) <= 14336, "the MMA path must keep 16 warps per SM");
static_assert(kStageBytes % 16 == 0 && kUnitHeadBytes % 16 == 0 && kStageKBytes % 16 == 0,
              "bulk-copy destinations must be 16-byte aligned");

template <bool kMma>
constexpr size_t attn_smem() { return sizeof(WarpSmemT<kMma>) * kWarps; }

__device__ __forceinline__ void zero_row(const AttnParams& p, int layer, int b, int lane) {
  const int64_t base = (int64_t(layer) * p.Bt + b) * p.Hq * kHeadDim;
  uint4* o = reinterpret_cast<uint4*>(p.out + base);
  const int n16 = p.Hq * kHeadDim * 2 / 16;
  for (int c = lane; c < n16; c += 32) o[c] = make_uint4(0, 0, 0, 0);
  if (p.out_f32) {
    float4* of = reinterpret_cast<float4*>(p.out_f32 + base);
    for (int c = lane; c < 2 * n16; c += 32) of[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Output scale of a head: v_scale / (l + 2^(sg - m)) with the head's
// attention-sink logit sg (log2 units; none when `sink` is null), l the sum of
// 2^(s - m) over its keys and m their reference maximum (log2 units).  When
// sg > m numerator and denominator are scaled by 2^-(sg - m), so nothing
// overflows.
__device__ __forceinline__ float out_scale(float l, float m, const float* sink, float vscale) {
  if (sink == nullptr) return vscale * __frcp_rn(l);
  const float d = __ldg(sink) * 1.4426950408889634f - m;
  const float e = ex2(-fabsf(d));
  return d > 0.f ? vscale * e * __frcp_rn(fmaf(l, e, 1.f)) : vscale * __frcp_rn(l + e);
}

// Unit u covers plane u % planes of work entry e = u / planes.
__device__ __forceinline__ void decode_unit(const AttnParams& p, int u, int4 e, UnitDesc& d) {
  const int pl = u - fdiv(u, p.fd_planes) * int(p.fd_planes.d);
  const int j = fdiv(pl, p.fd_hkv);
  const bool swa = ((e.w >> 30) & 1) != 0;
  d.kind = swa ? 2 : 1;
  d.layer = swa ? 2 * j : 2 * j + 1;
  d.b = e.x;
  d.kvh = pl - j * p.Hkv;
  d.s = e.w & 0xffff;
  d.ns = (e.w >> 16) & 0x3fff;
  d.t_begin = e.y;
  d.t_end = e.z;
  d.st_begin = e.y / kStageTok;
  d.n_st = (e.z + kStageTok - 1) / kStageTok - d.st_begin;
}

// kMma = true: QK^T and PV on the tensor cores (the product path).
// kMma = false: the same pipeline with both products as fp32 FMA, kept to
// measure the choice (selected with GK_ATTN_PATH=fma).
// 4 CTAs (16 warps) per SM: latency hiding across warps measured worth more
// than a deeper ring or the registers above 128.
// kPackedK: K through the packed view (tokens 2p, 2p+1 interleaved per
// channel) or laid out like V.
template <bool kMma, bool kPackedK>
__global__ void __launch_bounds__(kWarps * 32, kMma ? 4 : 3)
    attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qd = lane & 3;
  WarpSmemT<kMma>& ws = reinterpret_cast<WarpSmemT<kMma>*>(smem_raw)[warp];
  const uint32_t ring0 = smem_u32(&ws.ring[0][0]);
  const uint32_t qbuf0 = smem_u32(&ws.qbuf[0]);
  const uint32_t bar0 = smem_u32(&ws.bar[0]);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
  }
  __syncwarp();

  // the planner grid (launched just before) must be complete from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The combine grid, launched right after this one when partial records
  // exist (cap > 0), may launch now: it waits for this grid before reading.
  // Without it the next launch in the stream could be a planner, which must
  // not start (and rewrite the work queue) while this grid runs: no trigger.
  if (p.cap > 0) asm volatile("griddepcontrol.launch_dependents;");
  const int nU = p.hdr[kHdrNUnits];
  const int nAll = nU + p.hdr[kHdrNZero];  // units with a descriptor, then zero-fill units

  // ------------------------------------------------ scheduler pipeline
  // Each warp holds one claimed unit ahead of the one it streams: its
  // descriptor is loaded when it is claimed and its first block-table chunk
  // while the current unit streams.  (Claiming two ahead measured slower.)
  // the first unit of warp w is unit w (the planner starts the counter at
  // the grid's warp count): no burst of claims on one counter at the start
  int u_after = 0, u_next = int(blockIdx.x) * kWarps + warp;
  // the claimed unit's descriptor travels into shared memory by cp.async (no
  // registers held while it is in flight); read_desc waits for it
  auto claim_desc = [&](int u) {
    if (lane == 0 && u < nU) cp_async16(smem_u32(&ws.e_next), p.edesc + fdiv(u, p.fd_planes));
  };
  auto read_desc = [&]() -> int4 {
    if (lane == 0) cp_async_wait_all();
    __syncwarp();
    const int4 e = ws.e_next;
    __syncwarp();
    return e;
  };
  claim_desc(u_next);
  bool tn_ready = false;
  int32_t tbl_next = 0;
  int tbl_next_base = 0;
  // lane l: entry l of the table chunk starting at the unit's first block
  auto load_tbl = [&](int4 e, int& base) -> int32_t {
    const bool swa = ((e.w >> 30) & 1) != 0;
    const int32_t* row = swa ? p.bt_swa + int64_t(e.x) * p.MBS : p.bt_full + int64_t(e.x) * p.MBF;
    const int row_len = swa ? p.MBS : p.MBF;
    base = fdiv((e.y / kStageTok) * kStageTok, p.fd_b);
    const int idx = base + lane;
    return idx < row_len ? __ldg(row + idx) : 0;
  };

  // ------------------------------------------------ producer state
  int prod = 0, cons = 0;
  int f_head = 0, f_tail = 0;
  bool exhausted = false;
  // (the producer unit's other fields are read from its FIFO entry, the last one pushed)
  int pk = 0, pu_n_st = 0;
  // the producer's unit, advanced stage by stage: block (row index) and key
  // offset of the next stage (its K/V bases are in ws.pu_base)
  int pu_blk = 0, pu_off = 0, p_slot = 0;
  int tbl_base = -1;
  int32_t tbl = 0;
  bool failed = false;
  bool q_free = true;  // the q buffer may take the next unit's q

  // lane 0: copy the producer unit's q (8 heads) and its row's cos/sin rows
  auto issue_unit_head = [&](uint32_t bar, int layer, int b, int kvh) {
    const uint16_t* qsrc =
        p.q + ((int64_t(layer) * p.Bt + b) * p.Hq + int64_t(kvh) * kGroup) * kHeadDim;
    bulk_g2s(qbuf0, qsrc, kQBytes, bar);
    bulk_g2s(qbuf0 + kQBytes, p.cosb + int64_t(b) * (kHeadDim / 2), kRopeBytes, bar);
    bulk_g2s(qbuf0 + kQBytes + kRopeBytes, p.sinb + int64_t(b) * (kHeadDim / 2), kRopeBytes, bar);
  };

  // Next unit from the pipeline (warp-uniform); zero-fill units (inactive
  // rows) are done here.  Returns false when the queue is empty.
  auto next_unit = [&](UnitDesc& d) -> bool {
    for (;;) {
      const int u = u_next;
      if (u >= nAll) return false;
      const int4 e = u < nU ? read_desc() : make_int4(0, 0, 0, 0);
      int32_t tcur = 0;
      int tcur_base = 0;
      if (u < nU) {
        if (tn_ready) {
          tcur = tbl_next;
          tcur_base = tbl_next_base;
        } else {
          tcur = load_tbl(e, tcur_base);
        }
      }
      if (lane == 0) u_after = atomicAdd(p.queue, 1);
      u_next = __shfl_sync(kFull, u_after, 0);
      claim_desc(u_next);
      tn_ready = false;
      if (u >= nU) {
        const int v = u - nU;
        const int zr = fdiv(v, p.fd_nl);
        zero_row(p, v - zr * p.NL, p.zero_list[zr], lane);
        continue;
      }
      decode_unit(p, u, e, d);
      tbl = tcur;
      tbl_base = tcur_base;
      return true;
    }
  };

  auto issue_next = [&]() -> bool {
    if (exhausted) return false;
    int h_layer = 0, h_b = 0, h_kvh = 0;  // the unit started here (for its head copy)
    if (pk == pu_n_st) {
      if (!q_free) return false;  // the consumer has not read the buffered q yet
      UnitDesc d;
      if (!next_unit(d)) {
        exhausted = true;
        return false;
      }
      if (lane == 0) ws.fifo[f_tail % kFifo] = d;
      __syncwarp();
      ++f_tail;
      pk = 0;
      pu_n_st = d.n_st;
      h_layer = d.layer;
      h_b = d.b;
      h_kvh = d.kvh;
      {
        const int tok = d.st_begin * kStageTok;
        pu_blk = fdiv(tok, p.fd_b);
        pu_off = tok - pu_blk * p.B;
        const int last = tok + (d.n_st - 1) * kStageTok;
        if (lane == 0) ws.pu_trim = ((d.t_begin - tok) & ~7) | (((d.t_end - last + 7) & ~7) << 8);
      }
      if (lane == 0) {
        const int64_t head = int64_t(d.kvh) * p.B * kHeadDim;
        ws.pu_base[0] = p.kb[d.layer >> 1] + head;
        ws.pu_base[1] = p.vb[d.layer >> 1] + head;
      }
      q_free = false;
    } else if (!tn_ready && u_next < nU) {
      tbl_next = load_tbl(read_desc(), tbl_next_base);
      tn_ready = true;
    }
    const uint32_t head_bytes =
        pk == 0 ? kUnitHeadBytes : 0u;
    const uint32_t dst = ring0 + p_slot * kStageBytes;
    const uint32_t bar = bar0 + 8 * p_slot;
    const bool two = p.B < kStageTok;  // 16-token blocks: two per stage
    if (tbl_base < 0 || pu_blk + (two ? 1 : 0) >= tbl_base + 32) {
      const UnitDesc& du = ws.fifo[(f_tail + kFifo - 1) % kFifo];
      const int row_len = du.kind == 1 ? p.MBF : p.MBS;
      const int32_t* row = du.kind == 1 ? p.bt_full + int64_t(du.b) * p.MBF
                                        : p.bt_swa + int64_t(du.b) * p.MBS;
      tbl_base = pu_blk;
      const int idx = pu_blk + lane;
      tbl = idx < row_len ? row[idx] : 0;
    }
    const int blk_bytes = p.Hkv * p.B * kHeadDim;  // one block of all kv heads
    int32_t pb0 = __shfl_sync(kFull, tbl, pu_blk - tbl_base);
    if (uint32_t(pb0) >= uint32_t(p.nb)) {
      if (lane == 0) set_error(GK_DEVERR_BLOCK);
      pb0 = 0;
    }
    if (!two) {
      // a unit's first and last stages copy only the keys of its range
      // (rounded out to 8): a window starting inside a stage reads at most 7
      // keys before it instead of up to 31
      uint32_t lo_b = 0, kbytes = kStageKBytes;
      if (pk == 0 || pk == pu_n_st - 1) {
        const int trim = ws.pu_trim;
        const int lo = pk == 0 ? (trim & 0xff) : 0;
        const int hi = pk == pu_n_st - 1 ? (trim >> 8) : kStageTok;
        lo_b = uint32_t(lo) * kHeadDim;
        kbytes = uint32_t(hi - lo) * kHeadDim;
      }
      if (lane == 0) {
        const int64_t off = int64_t(pb0) * blk_bytes + pu_off * kHeadDim + lo_b;
        mbar_arrive_expect_tx(bar, 2 * kbytes + head_bytes);
        if (head_bytes) issue_unit_head(bar, h_layer, h_b, h_kvh);
        bulk_g2s(dst + lo_b, ws.pu_base[0] + off, kbytes, bar);
        bulk_g2s(dst + kStageKBytes + lo_b, ws.pu_base[1] + off, kbytes, bar);
      }
      pu_off += kStageTok;
      if (pu_off == p.B) {
        pu_off = 0;
        ++pu_blk;
      }
    } else {
      int32_t pb1 = __shfl_sync(kFull, tbl, min(pu_blk + 1 - tbl_base, 31));
      const UnitDesc& du = ws.fifo[(f_tail + kFifo - 1) % kFifo];
      const int row_len = du.kind == 1 ? p.MBF : p.MBS;
      const bool has1 = (pu_blk + 1) * p.B < du.t_end;
      if (has1 && (pu_blk + 1 >= row_len || uint32_t(pb1) >= uint32_t(p.nb))) {
        if (lane == 0) set_error(GK_DEVERR_BLOCK);
        pb1 = 0;
      }
      if (lane == 0) {
        const uint32_t half = uint32_t(p.B) * kHeadDim;
        mbar_arrive_expect_tx(bar, (has1 ? 4 * half : 2 * half) + head_bytes);
        if (head_bytes) issue_unit_head(bar, h_layer, h_b, h_kvh);
        const int64_t o0 = int64_t(pb0) * blk_bytes;
        bulk_g2s(dst, ws.pu_base[0] + o0, half, bar);
        bulk_g2s(dst + kStageKBytes, ws.pu_base[1] + o0, half, bar);
        if (has1) {
          const int64_t o1 = int64_t(pb1) * blk_bytes;
          bulk_g2s(dst + half, ws.pu_base[0] + o1, half, bar);
          bulk_g2s(dst + kStageKBytes + half, ws.pu_base[1] + o1, half, bar);
        }
      }
      pu_blk += 2;
    }
    p_slot = p_slot == kStages - 1 ? 0 : p_slot + 1;
    ++pk;
    ++prod;
    return true;
  };

  // ------------------------------------------------ consumer state
  // The consumer's unit: the fields the stage loop uses live in registers;
  // the others are read from its descriptor in shared memory (the slot stays
  // put while the unit runs: the FIFO holds more units than the ring can run ahead).
  struct {
    int t_begin, t_end, st_begin, n_st;
  } cd;
#define CU (ws.fifo[f_head % kFifo])
  int k_in_unit = 0;
  int c_slot = 0;        // cons % kStages
  uint32_t c_par = 0u;   // (cons / kStages) & 1
  uint32_t qhi[8], qlo[8];  // q' = qhi + qlo (f16 each): ~22-bit significand
  // Scores come out of the MMA as x * 2^e_h, x = logit in log2 units and
  // 2^e_h the per-head normalisation of q; si_h = 2^-e_h undoes it.  mr_h is
  // the running reference maximum (raw units), allowed to lag the true
  // maximum by up to kLazyLog2 so that most stages skip the rescale.
  float si0 = 0.f, si1 = 0.f, mr0 = 0.f, mr1 = 0.f, nb0 = 0.f, nb1 = 0.f, thr0 = 0.f,
        thr1 = 0.f, vscale = 0.f;
  float o[4][4];
  float lacc[4];  // softmax denominators from a ones-row MMA over the f16 P
  // FMA path: per-head reference maxima / thresholds (log2 units, warp-uniform)
  // and this lane's partial denominators (lane = token)
  float mh[kMma ? 1 : kGroup], thh[kMma ? 1 : kGroup], lsum[kMma ? 1 : kGroup];

  while (prod - cons < kStages && issue_next()) {
  }

  while (cons < prod) {
    // ---- wait for the stage (the unit's first stage also brings its q)
    const int slot = c_slot;
    const uint32_t bar = bar0 + 8 * slot;
    const uint32_t parity = c_par;
    if (!mbar_wait_bounded(bar, parity, kWaitLimitNs)) failed = true;
    if (__any_sync(kFull, failed)) {
      failed = true;
      break;
    }
    if (k_in_unit == 0) {
      cd.t_begin = CU.t_begin;
      cd.t_end = CU.t_end;
      cd.st_begin = CU.st_begin;
      cd.n_st = CU.n_st;
      // ---- unit prologue: rotated q for head (kvh*8 + g), channels 16qd..16qd+15
      const uint32_t qrow = qbuf0 + g * (kHeadDim * 2);
      const uint4 x0 = lds128(qrow + 32 * qd);
      const uint4 x1 = lds128(qrow + 32 * qd + 16);
      const uint4 y0 = lds128(qrow + 32 * (qd ^ 2));
      const uint4 y1 = lds128(qrow + 32 * (qd ^ 2) + 16);
      const uint32_t cp = qbuf0 + kQBytes + 64 * (qd & 1);
      const uint32_t sp = cp + kRopeBytes;
      const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yw[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      uint32_t cw[16], sw[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 c4 = lds128(cp + 16 * k);
        const uint4 s4 = lds128(sp + 16 * k);
        cw[4 * k] = c4.x; cw[4 * k + 1] = c4.y; cw[4 * k + 2] = c4.z; cw[4 * k + 3] = c4.w;
        sw[4 * k] = s4.x; sw[4 * k + 1] = s4.y; sw[4 * k + 2] = s4.z; sw[4 * k + 3] = s4.w;
      }
      __syncwarp();
      q_free = true;
      const float sgn = qd < 2 ? -1.f : 1.f;
      // logits in log2 units: q'.k * k_scale / sqrt(D) * log2(e), folded into q
      // (for the MMA path together with the power-of-two normalisation below)
      const float ck = p.k_scale[CU.layer] * (0.125f * 1.4426950408889634f);
      float r[16];  // rotated q, before the ck scaling
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float c0 = __uint_as_float(cw[2 * w]), c1 = __uint_as_float(cw[2 * w + 1]);
        const float s0 = __uint_as_float(sw[2 * w]), s1 = __uint_as_float(sw[2 * w + 1]);
        r[2 * w] = bf16lo_to_f32(xw[w]) * c0 + sgn * bf16lo_to_f32(yw[w]) * s0;
        r[2 * w + 1] = bf16hi_to_f32(xw[w]) * c1 + sgn * bf16hi_to_f32(yw[w]) * s1;
        amax = fmaxf(amax, fmaxf(fabsf(r[2 * w]), fabsf(r[2 * w + 1])));
      }
      if constexpr (!kMma) {
        // q' (log2 units) in fp32 to shared memory: head g, channels 16qd..16qd+15
        float* qrow_f = ws.qf + g * kQfStride + 16 * qd;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          reinterpret_cast<float4*>(qrow_f)[k] =
              make_float4(r[4 * k] * ck, r[4 * k + 1] * ck, r[4 * k + 2] * ck, r[4 * k + 3] * ck);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          mh[h] = -INFINITY;
          thh[h] = -INFINITY;
          lsum[h] = 0.f;
        }
        si0 = si1 = 1.f;
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2)) * ck;
      // power-of-two normalisation of the head so that max |q'| < 2^14 in f16
      int ex = int((__float_as_uint(amax) >> 23) & 0xffu) - 127;
      ex = amax > 0.f ? min(max(ex, -100), 100) : 13;
      const float f = __uint_as_float(uint32_t(127 + 13 - ex) << 23);
      const float finv = __uint_as_float(uint32_t(127 - 13 + ex) << 23);
      const float fck = f * ck;  // fl(x * fck) == fl(x * ck) * f: f is a power of two
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float a = r[2 * w] * fck, b = r[2 * w + 1] * fck;
        qhi[w] = f32x2_to_f16x2(a, b);
        const float2 h = f16x2_to_f32x2(qhi[w]);
        qlo[w] = f32x2_to_f16x2(a - h.x, b - h.y);  // residual is exact in fp32
      }
      if constexpr (kMma) {
        si0 = __shfl_sync(kFull, finv, 8 * qd);   // heads 2qd and 2qd+1
        si1 = __shfl_sync(kFull, finv, 8 * qd + 4);
      }
      vscale = p.v_scale[CU.layer];
      mr0 = mr1 = thr0 = thr1 = -INFINITY;
      nb0 = nb1 = 0.f;
      lacc[0] = lacc[1] = lacc[2] = lacc[3] = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
    }

    const uint32_t Ks = ring0 + slot * kStageBytes;
    const uint32_t Vs = Ks + kStageKBytes;
    const int tok0 = (cd.st_begin + k_in_unit) * kStageTok;
    const bool edge = tok0 < cd.t_begin || tok0 + kStageTok > cd.t_end;
    if constexpr (kMma) {
    // ---- S = q' K^T for two 16-token tiles; rows (g, g+8) = tokens (2g+sw, 2g+1-sw)
    // of the tile, sw = 0 for packed K; for plain K sw = g & 1, so that lanes of
    // odd g read their second token first and a quarter-warp's 16-byte reads
    // fall in distinct banks (a relabelling of rows: nothing is moved).
    const int sw = kPackedK ? 0 : (g & 1);
    float sc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      if constexpr (kPackedK) {
        const uint32_t kp = Ks + (8 * i + g) * (2 * kHeadDim) + 32 * qd;
        const uint4 w0 = lds128(kp);
        const uint4 w1 = lds128(kp + 16);
        const uint32_t kw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(prmt(kw[2 * j], 0u, 0x3120u), a0, a1);
          e4m3x4_to_f16x2x2(prmt(kw[2 * j + 1], 0u, 0x3120u), a2, a3);
          mma_f16(sc[i], a0, a1, a2, a3, qlo[2 * j], qlo[2 * j + 1]);
          mma_f16(sc[i], a0, a1, a2, a3, qhi[2 * j], qhi[2 * j + 1]);
        }
      } else {
        // channels 16qd..16qd+15 of the two tokens; word j = channels 16qd+4j..+3
        const uint32_t kp = Ks + (16 * i + 2 * g) * kHeadDim + 16 * qd;
        const uint4 r0 = lds128(kp + sw * kHeadDim);        // row g
        const uint4 r1 = lds128(kp + (1 - sw) * kHeadDim);  // row g + 8
        const uint32_t k0[4] = {r0.x, r0.y, r0.z, r0.w};
        const uint32_t k1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(k0[j], a0, a2);
          e4m3x4_to_f16x2x2(k1[j], a1, a3);
          mma_f16(sc[i], a0, a1, a2, a3, qlo[2 * j], qlo[2 * j + 1]);
          mma_f16(sc[i], a0, a1, a2, a3, qhi[2 * j], qhi[2 * j + 1]);
        }
      }
    }
    // ---- online softmax (log2 domain); lane holds heads 2qd (c0,c2), 2qd+1 (c1,c3)
    if (edge) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t0 = tok0 + 16 * i + 2 * g + sw;      // row g
        const int t1 = tok0 + 16 * i + 2 * g + 1 - sw;  // row g + 8
        if (t0 < cd.t_begin || t0 >= cd.t_end) sc[i][0] = sc[i][1] = -INFINITY;
        if (t1 < cd.t_begin || t1 >= cd.t_end) sc[i][2] = sc[i][3] = -INFINITY;
      }
    }
    const float lm0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
    const float lm1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
    if (__any_sync(kFull, lm0 > thr0 || lm1 > thr1)) {
      // some score passed its reference by more than 2^kLazyLog2: move the
      // reference to the true running maximum and rescale what was summed
      float w0 = lm0, w1 = lm1;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        w0 = fmaxf(w0, __shfl_xor_sync(kFull, w0, off));
        w1 = fmaxf(w1, __shfl_xor_sync(kFull, w1, off));
      }
      const float n0 = fmaxf(mr0, w0), n1 = fmaxf(mr1, w1);
      const float al0 = ex2((mr0 - n0) * si0), al1 = ex2((mr1 - n1) * si1);
      mr0 = n0;
      mr1 = n1;
      nb0 = -n0 * si0;
      nb1 = -n1 * si1;
      thr0 = n0 + kLazyLog2 / si0;
      thr1 = n1 + kLazyLog2 / si1;
      lacc[0] *= al0;
      lacc[2] *= al0;
      lacc[1] *= al1;
      lacc[3] *= al1;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        o[m][0] *= al0;
        o[m][2] *= al0;
        o[m][1] *= al1;
        o[m][3] *= al1;
      }
    }
    float pr[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      pr[i][0] = ex2(fmaf(sc[i][0], si0, nb0));
      pr[i][1] = ex2(fmaf(sc[i][1], si1, nb1));
      pr[i][2] = ex2(fmaf(sc[i][2], si0, nb0));
      pr[i][3] = ex2(fmaf(sc[i][3], si1, nb1));
    }
    // ---- O += P V; rows (g, g+8) = channels (8g+2m, 8g+2m+1), k = tokens 4qd..4qd+3:
    // after the transpose b0 holds tokens (4qd, 4qd+2) and b1 (4qd+1, 4qd+3) for
    // packed K; with the plain-K row order b0 holds (4qd, 4qd+3), b1 (4qd+1, 4qd+2)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t b0 = movmatrix_trans(f32x2_to_f16x2(pr[i][0], pr[i][1]));
      const uint32_t b1 = movmatrix_trans(f32x2_to_f16x2(pr[i][2], pr[i][3]));
      // every row of the ones matrix sums the same rounded P the values see
      mma_f16(lacc, kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2, b0, b1);
      const uint32_t vp = Vs + (16 * i + 4 * qd) * kHeadDim + 8 * g;
      uint2 v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = lds64(vp + r * kHeadDim);
      if (edge) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int t = tok0 + 16 * i + 4 * qd + r;
          if (t < cd.t_begin || t >= cd.t_end) v[r] = make_uint2(0u, 0u);
        }
      }
      constexpr int r0a = 0, r0b = kPackedK ? 2 : 3;  // the tokens of b0: 4qd + r0a, 4qd + r0b
      constexpr int r1a = 1, r1b = kPackedK ? 3 : 2;  // the tokens of b1
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t sel = (m & 1) ? 0x7362u : 0x5140u;
        const uint32_t e0 = prmt(m < 2 ? v[r0a].x : v[r0a].y, m < 2 ? v[r0b].x : v[r0b].y, sel);
        const uint32_t e1 = prmt(m < 2 ? v[r1a].x : v[r1a].y, m < 2 ? v[r1b].x : v[r1b].y, sel);
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(e0, a0, a1);
        e4m3x4_to_f16x2x2(e1, a2, a3);
        mma_f16(o[m], a0, a1, a2, a3, b0, b1);
      }
    }
    }
    if constexpr (!kMma) {
      // ---- S = q' K^T with fp32 FMA; lane = token t of the stage
      const int t = lane;
      const uint32_t krow = kPackedK ? Ks + (t >> 1) * (2 * kHeadDim) : Ks + t * kHeadDim;
      const uint32_t sel = (t & 1) ? 0x7531u : 0x6420u;  // this token's byte of each pair
      float sf[kGroup];
#pragma unroll
      for (int h = 0; h < kGroup; ++h) sf[h] = 0.f;
#pragma unroll 2
      for (int c = 0; c < kHeadDim / 8; ++c) {  // 8 channels per step
        uint32_t h01, h23, h45, h67;
        if constexpr (kPackedK) {
          const uint4 w = lds128(krow + 16 * c);
          e4m3x4_to_f16x2x2(prmt(w.x, w.y, sel), h01, h23);
          e4m3x4_to_f16x2x2(prmt(w.z, w.w, sel), h45, h67);
        } else {
          const uint2 w = lds64(krow + 8 * c);
          e4m3x4_to_f16x2x2(w.x, h01, h23);
          e4m3x4_to_f16x2x2(w.y, h45, h67);
        }
        const float2 k01 = f16x2_to_f32x2(h01), k23 = f16x2_to_f32x2(h23);
        const float2 k45 = f16x2_to_f32x2(h45), k67 = f16x2_to_f32x2(h67);
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          const float4 qa = reinterpret_cast<const float4*>(ws.qf + h * kQfStride + 8 * c)[0];
          const float4 qb = reinterpret_cast<const float4*>(ws.qf + h * kQfStride + 8 * c)[1];
          sf[h] = fmaf(qa.x, k01.x, sf[h]);
          sf[h] = fmaf(qa.y, k01.y, sf[h]);
          sf[h] = fmaf(qa.z, k23.x, sf[h]);
          sf[h] = fmaf(qa.w, k23.y, sf[h]);
          sf[h] = fmaf(qb.x, k45.x, sf[h]);
          sf[h] = fmaf(qb.y, k45.y, sf[h]);
          sf[h] = fmaf(qb.z, k67.x, sf[h]);
          sf[h] = fmaf(qb.w, k67.y, sf[h]);
        }
      }
      const bool valid = !(edge && (tok0 + t < cd.t_begin || tok0 + t >= cd.t_end));
      bool over = false;
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        if (!valid) sf[h] = -INFINITY;
        over |= sf[h] > thh[h];
      }
      if (__any_sync(kFull, over)) {
        float al[kGroup];
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          float wm = sf[h];
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, off));
          const float n = fmaxf(mh[h], wm);
          al[h] = ex2(mh[h] - n);
          mh[h] = n;
          thh[h] = n + kLazyLog2;
          lsum[h] *= al[h];
        }
        float a0 = 1.f, a1 = 1.f;
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
          if (h == 2 * qd) a0 = al[h];
          if (h == 2 * qd + 1) a1 = al[h];
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          o[m][0] *= a0;
          o[m][2] *= a0;
          o[m][1] *= a1;
          o[m][3] *= a1;
        }
      }
      float pf[kGroup];
#pragma unroll
      for (int h = 0; h < kGroup; ++h) {
        pf[h] = ex2(sf[h] - mh[h]);
        lsum[h] += pf[h];
      }
      float4* prow = reinterpret_cast<float4*>(ws.pbuf + t * kGroup);
      prow[0] = make_float4(pf[0], pf[1], pf[2], pf[3]);
      prow[1] = make_float4(pf[4], pf[5], pf[6], pf[7]);
      __syncwarp();
      // ---- O += P V with fp32 FMA; lane (g, qd): heads 2qd, 2qd+1, channels 8g..8g+7
      for (int tt = 0; tt < kStageTok; ++tt) {
        if (edge && (tok0 + tt < cd.t_begin || tok0 + tt >= cd.t_end)) continue;
        const float2 pp = reinterpret_cast<const float2*>(ws.pbuf + tt * kGroup + 2 * qd)[0];
        const uint2 vv = lds64(Vs + tt * kHeadDim + 8 * g);
        uint32_t v01, v23, v45, v67;
        e4m3x4_to_f16x2x2(vv.x, v01, v23);
        e4m3x4_to_f16x2x2(vv.y, v45, v67);
        const float2 f01 = f16x2_to_f32x2(v01), f23 = f16x2_to_f32x2(v23);
        const float2 f45 = f16x2_to_f32x2(v45), f67 = f16x2_to_f32x2(v67);
        const float vf[8] = {f01.x, f01.y, f23.x, f23.y, f45.x, f45.y, f67.x, f67.y};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          o[m][0] = fmaf(pp.x, vf[2 * m], o[m][0]);
          o[m][2] = fmaf(pp.x, vf[2 * m + 1], o[m][2]);
          o[m][1] = fmaf(pp.y, vf[2 * m], o[m][1]);
          o[m][3] = fmaf(pp.y, vf[2 * m + 1], o[m][3]);
        }
      }
    }
    __syncwarp();
    ++cons;
    if (++c_slot == kStages) {
      c_slot = 0;
      c_par ^= 1u;
    }
    ++k_in_unit;
    while (prod - cons < kStages && issue_next()) {
    }

    if (k_in_unit == cd.n_st) {
      // ---- unit epilogue
      k_in_unit = 0;
      if constexpr (!kMma) {
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) lsum[h] += __shfl_xor_sync(kFull, lsum[h], off);
          if (h == 2 * qd) {
            lacc[0] = lsum[h];
            mr0 = mh[h];
          }
          if (h == 2 * qd + 1) {
            lacc[1] = lsum[h];
            mr1 = mh[h];
          }
        }
      }
      const float l0 = lacc[0], l1 = lacc[1];
      const int64_t out_row =
          ((int64_t(CU.layer) * p.Bt + CU.b) * p.Hq + CU.kvh * kGroup + 2 * qd) * kHeadDim + 8 * g;
      if (CU.ns == 1) {
        const float* snk =
            p.sinks ? p.sinks + int64_t(CU.layer) * p.Hq + CU.kvh * kGroup + 2 * qd : nullptr;
        const float i0 = out_scale(l0, mr0 * si0, snk, vscale);
        const float i1 = out_scale(l1, mr1 * si1, snk ? snk + 1 : nullptr, vscale);
        float r0[8], r1[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          r0[2 * m] = o[m][0] * i0;
          r0[2 * m + 1] = o[m][2] * i0;
          r1[2 * m] = o[m][1] * i1;
          r1[2 * m + 1] = o[m][3] * i1;
        }
        uint4 u0, u1;
        u0.x = f32x2_to_bf16x2(r0[0], r0[1]);
        u0.y = f32x2_to_bf16x2(r0[2], r0[3]);
        u0.z = f32x2_to_bf16x2(r0[4], r0[5]);
        u0.w = f32x2_to_bf16x2(r0[6], r0[7]);
        u1.x = f32x2_to_bf16x2(r1[0], r1[1]);
        u1.y = f32x2_to_bf16x2(r1[2], r1[3]);
        u1.z = f32x2_to_bf16x2(r1[4], r1[5]);
        u1.w = f32x2_to_bf16x2(r1[6], r1[7]);
        *reinterpret_cast<uint4*>(p.out + out_row) = u0;
        *reinterpret_cast<uint4*>(p.out + out_row + kHeadDim) = u1;
        if (p.out_f32) {
          float4* f0 = reinterpret_cast<float4*>(p.out_f32 + out_row);
          float4* f1 = reinterpret_cast<float4*>(p.out_f32 + out_row + kHeadDim);
          f0[0] = make_float4(r0[0], r0[1], r0[2], r0[3]);
          f0[1] = make_float4(r0[4], r0[5], r0[6], r0[7]);
          f1[0] = make_float4(r1[0], r1[1], r1[2], r1[3]);
          f1[1] = make_float4(r1[4], r1[5], r1[6], r1[7]);
        }
      } else {
        // split partial: (m, l, o) unnormalised, in log2 units, for the combine kernel
        const int j = CU.layer >> 1;
        const int64_t plane = int64_t(j) * p.Hkv + CU.kvh;
        const int64_t cap = p.cap;
        float* rec = p.partials + ((plane * cap) + p.part_base[CU.b] + CU.s) * kPartialFloats;
        if (g == 0) {
          rec[2 * qd] = mr0 * si0;  // log2 units
          rec[2 * qd + 1] = mr1 * si1;
          rec[kGroup + 2 * qd] = l0;
          rec[kGroup + 2 * qd + 1] = l1;
        }
        float4* ro0 = reinterpret_cast<float4*>(rec + 2 * kGroup + (2 * qd) * kHeadDim + 8 * g);
        float4* ro1 = reinterpret_cast<float4*>(rec + 2 * kGroup + (2 * qd + 1) * kHeadDim + 8 * g);
        ro0[0] = make_float4(o[0][0], o[0][2], o[1][0], o[1][2]);
        ro0[1] = make_float4(o[2][0], o[2][2], o[3][0], o[3][2]);
        ro1[0] = make_float4(o[0][1], o[0][3], o[1][1], o[1][3]);
        ro1[1] = make_float4(o[2][1], o[2][3], o[3][1], o[3][3]);
      }
      ++f_head;
    }
  }

#undef CU
  if (failed) {
    // A barrier wait hit its limit: record it, then wait (bounded) for this
    // warp's copies still in flight before the CTA may exit.
    if (lane == 0) set_error(GK_DEVERR_TIMEOUT);
    for (int c = cons; c < prod; ++c) {
      const uint32_t bar = bar0 + 8 * (c % kStages);
      const uint32_t parity = uint32_t(c / kStages) & 1u;
      mbar_wait_bounded(bar, parity, kWaitLimitNs);
    }
  }
}


// =========================================================================
// Split-KV combine (flash-decoding)
// =========================================================================
// One warp per (split row, plane = (layer pair j, kv head)) merges the ns
// partial records of full layer 2j + 1, row b, kv head into the output.  Lane
// (g, qd) produces heads 2qd, 2qd + 1, channels 8g .. 8g + 7.  The partials
// are read kAhead at a time (their loads in flight together) and
// folded in split order -- the same order whatever order the splits finished
// in -- with a running maximum; then the output scale (attention sink
// included) and the bf16 (+ fp32) stores.
// Two forms.  The kernel is a chain of dependent rounds of partial loads:
// when every item fits in one wave of warps, eight partials per round at two
// CTAs per SM (211 registers) finish sooner; with more items than that, four
// per round at four CTAs per SM keep more items in flight.
constexpr int kCombineThreads = 128;
constexpr int kCombineDeepAhead = 8, kCombineDeepBlocks = 2;
constexpr int kCombineAhead = 4, kCombineBlocks = 4;

template <int kAhead, int kBlocksPerSm>
__global__ void __launch_bounds__(kCombineThreads, kBlocksPerSm)
    combine_kernel(const __grid_constant__ AttnParams p) {
  // the attention grid (launched just before) must be complete: its partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, g = lane >> 2, qd = lane & 3;
  const int n_rows = p.hdr[kHdrSplitRows];
  const int planes = int(p.fd_planes.d);
  const int n_items = n_rows * planes;  // <= 8192 rows x 4096 planes
  const int warps = int(gridDim.x) * (kCombineThreads / 32);
  for (int it = int(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5); it < n_items;
       it += warps) {
    const int r = fdiv(it, p.fd_planes);
    const int plane = it - r * planes;
    const int e = p.split_rows[r];
    const int b = e & 0xffff, ns = e >> 16;
    const int j = fdiv(plane, p.fd_hkv);
    const int kvh = plane - j * p.Hkv;
    const int layer = 2 * j + 1;
    const float* base = p.partials + (int64_t(plane) * p.cap + p.part_base[b]) * kPartialFloats;
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float a0[8], a1[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) a0[c] = a1[c] = 0.f;
    for (int s0 = 0; s0 < ns; s0 += kAhead) {
      float2 ms[kAhead], ls[kAhead];
      float4 o00[kAhead], o01[kAhead], o10[kAhead], o11[kAhead];
#pragma unroll
      for (int k = 0; k < kAhead; ++k) {
        if (s0 + k < ns) {
          const float* rs = base + int64_t(s0 + k) * kPartialFloats;
          ms[k] = ldg_cg_f2(rs + 2 * qd);
          ls[k] = ldg_cg_f2(rs + kGroup + 2 * qd);
          const float* os0 = rs + 2 * kGroup + (2 * qd) * kHeadDim + 8 * g;
          o00[k] = ldg_cg_f4(os0);
          o01[k] = ldg_cg_f4(os0 + 4);
          o10[k] = ldg_cg_f4(os0 + kHeadDim);
          o11[k] = ldg_cg_f4(os0 + kHeadDim + 4);
        }
      }
#pragma unroll
      for (int k = 0; k < kAhead; ++k) {
        if (s0 + k < ns) {
          const float n0 = fmaxf(M0, ms[k].x), n1 = fmaxf(M1, ms[k].y);
          const float c0 = ex2(M0 - n0), w0 = ex2(ms[k].x - n0);
          const float c1 = ex2(M1 - n1), w1 = ex2(ms[k].y - n1);
          M0 = n0;
          M1 = n1;
          L0 = fmaf(L0, c0, ls[k].x * w0);
          L1 = fmaf(L1, c1, ls[k].y * w1);
          const float q0[8] = {o00[k].x, o00[k].y, o00[k].z, o00[k].w,
                               o01[k].x, o01[k].y, o01[k].z, o01[k].w};
          const float q1[8] = {o10[k].x, o10[k].y, o10[k].z, o10[k].w,
                               o11[k].x, o11[k].y, o11[k].z, o11[k].w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            a0[c] = fmaf(a0[c], c0, q0[c] * w0);
            a1[c] = fmaf(a1[c], c1, q1[c] * w1);
          }
        }
      }
    }
    const float* snk = p.sinks ? p.sinks + int64_t(layer) * p.Hq + kvh * kGroup + 2 * qd : nullptr;
    const float vscale = p.v_scale[layer];
    const float i0 = out_scale(L0, M0, snk, vscale);
    const float i1 = out_scale(L1, M1, snk ? snk + 1 : nullptr, vscale);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      a0[c] *= i0;
      a1[c] *= i1;
    }
    const int64_t out_row =
        ((int64_t(layer) * p.Bt + b) * p.Hq + kvh * kGroup + 2 * qd) * kHeadDim + 8 * g;
    uint4 u0, u1;
    u0.x = f32x2_to_bf16x2(a0[0], a0[1]);
    u0.y = f32x2_to_bf16x2(a0[2], a0[3]);
    u0.z = f32x2_to_bf16x2(a0[4], a0[5]);
    u0.w = f32x2_to_bf16x2(a0[6], a0[7]);
    u1.x = f32x2_to_bf16x2(a1[0], a1[1]);
    u1.y = f32x2_to_bf16x2(a1[2], a1[3]);
    u1.z = f32x2_to_bf16x2(a1[4], a1[5]);
    u1.w = f32x2_to_bf16x2(a1[6], a1[7]);
    *reinterpret_cast<uint4*>(p.out + out_row) = u0;
    *reinterpret_cast<uint4*>(p.out + out_row + kHeadDim) = u1;
    if (p.out_f32) {
      float4* f0 = reinterpret_cast<float4*>(p.out_f32 + out_row);
      float4* f1 = reinterpret_cast<float4*>(p.out_f32 + out_row + kHeadDim);
      f0[0] = make_float4(a0[0], a0[1], a0[2], a0[3]);
      f0[1] = make_float4(a0[4], a0[5], a0[6], a0[7]);
      f1[0] = make_float4(a1[0], a1[1], a1[2], a1[3]);
      f1[1] = make_float4(a1[4], a1[5], a1[6], a1[7]);
    }
  }
}

// =========================================================================
// Test hook: the bounded barrier wait running out
// =========================================================================
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none ever comes
    mbar_init_fence();
  }
  __syncwarp();
  if (!mbar_wait_bounded(b, 0, limit_ns) && threadIdx.x == 0) set_error(GK_DEVERR_TIMEOUT);
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

// =========================================================================
// Launchers
// =========================================================================
struct DeviceCache {
  int dev = -1;
  int sms = 0;
  int attn_blocks_per_sm = 0;  // of the selected path
  bool fma = false;            // GK_ATTN_PATH=fma selects the FMA comparison path
  bool attrs_set = false;
};
static DeviceCache g_cache[64];

// Attention instantiations, index = fma * 2 + plain_k.
static const void* const kAttnKernels[4] = {
    (const void*)attn_kernel<true, true>, (const void*)attn_kernel<true, false>,
    (const void*)attn_kernel<false, true>, (const void*)attn_kernel<false, false>};

static cudaError_t device_setup(DeviceCache** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceCache& c = g_cache[dev];
  if (!c.attrs_set) {
    e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const char* path = getenv("GK_ATTN_PATH");
    c.fma = path != nullptr && strcmp(path, "fma") == 0;
    // every instantiation of the selected path is launched with the smallest
    // occupancy among them, so that all fit the same persistent grid
    c.attn_blocks_per_sm = 1 << 30;
    for (int k = 0; k < 4; ++k) {
      const bool mma = (k & 2) == 0;
      const size_t smem = mma ? attn_smem<true>() : attn_smem<false>();
      e = cudaFuncSetAttribute(kAttnKernels[k], cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(smem));
      if (e != cudaSuccess) return e;
      if (mma == c.fma) continue;
      int blocks = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kAttnKernels[k], kWarps * 32,
                                                        smem);
      if (e != cudaSuccess) return e;
      if (blocks < c.attn_blocks_per_sm) c.attn_blocks_per_sm = blocks;
    }
    e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(2 * kMaxBatch * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(2 * kMaxBatch * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    if (c.attn_blocks_per_sm < 1) c.attn_blocks_per_sm = 1;
    c.dev = dev;
    c.attrs_set = true;
  }
  *out = &c;
  return cudaSuccess;
}

int attention_resident_warps() {
  DeviceCache* c = nullptr;
  if (device_setup(&c) != cudaSuccess) return 0;
  return c->sms * c->attn_blocks_per_sm * kWarps;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t st) {
  const int64_t warps = int64_t(p.NL) * p.Bt;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  kv_append_kernel<<<unsigned(blocks), threads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const float* x, float scale, uint8_t* codes, int64_t n,
                            cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  DeviceCache* c = nullptr;
  cudaError_t e = device_setup(&c);
  if (e != cudaSuccess) return e;
  const int threads = 256;
  int64_t blocks = (n / 2 + threads) / threads;
  blocks = blocks < int64_t(c->sms) * 8 ? blocks : int64_t(c->sms) * 8;
  quantize_kernel<<<unsigned(blocks), threads, 0, st>>>(x, scale, codes, n);
  return cudaGetLastError();
}

cudaError_t launch_attention(const PlanParams& plan, const AttnParams& p, cudaStream_t st,
                             const AppendParams* app) {
  DeviceCache* c = nullptr;
  cudaError_t e = device_setup(&c);
  if (e != cudaSuccess) return e;
  PlanParams pp = plan;
  pp.n_warps = c->sms * c->attn_blocks_per_sm * kWarps;
  // Programmatic dependent launches: the planner may overlap the kernel before
  // it (it reads no KV and waits for that kernel before exiting); the
  // attention CTAs start while the planner runs and wait for it
  // (griddepcontrol.wait) before reading its plan.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3(1);
  pcfg.blockDim = dim3(kPlanThreads);
  pcfg.dynamicSmemBytes = size_t(2) * p.Bt * sizeof(int32_t);
  pcfg.stream = st;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  if (app) {
    // gk_decode_step appends in CTAs beside the planner's: one warp
    // per (layer, row) pair
    PlanAppendParams pa;
    pa.plan = pp;
    pa.app = *app;
    pcfg.gridDim = dim3(unsigned(1 + (int64_t(app->NL) * app->Bt * 32 + kPlanThreads - 1) /
                                         kPlanThreads));
    e = cudaLaunchKernelEx(&pcfg, plan_append_kernel, pa);
  } else {
    e = cudaLaunchKernelEx(&pcfg, plan_kernel, pp);
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(c->sms * c->attn_blocks_per_sm));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = c->fma ? attn_smem<false>() : attn_smem<true>();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int k = (c->fma ? 2 : 0) + (p.k_packed ? 0 : 1);
  void* args[] = {const_cast<AttnParams*>(&p)};
  e = cudaLaunchKernelExC(&cfg, kAttnKernels[k], args);
  if (e != cudaSuccess || p.cap == 0) return e;  // no partial records: nothing to combine
  // the deep form when even batch x planes items (every row split) fit in
  // one wave of its warps
  const bool deep = int64_t(p.Bt) * int64_t(p.fd_planes.d) <=
                    int64_t(c->sms) * kCombineDeepBlocks * (kCombineThreads / 32);
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(unsigned(c->sms * (deep ? kCombineDeepBlocks : kCombineBlocks)));
  ccfg.blockDim = dim3(kCombineThreads);
  ccfg.stream = st;
  ccfg.attrs = attr;
  ccfg.numAttrs = 1;
  return deep ? cudaLaunchKernelEx(&ccfg, combine_kernel<kCombineDeepAhead, kCombineDeepBlocks>, p)
              : cudaLaunchKernelEx(&ccfg, combine_kernel<kCombineAhead, kCombineBlocks>, p);
}

cudaError_t read_device_error(cudaStream_t st, uint32_t* bits, bool clear) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(bits, g_dev_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gk
