/*
 * gk.h -- C ABI of the GB300 (sm_103a) stack-wide paged-FP8 decode-attention library.
 *
 * One decode step of GPT-OSS-style attention over a whole layer stack, as the
 * "GPT-OSS-120B giga-kernel decode" page describes it:
 *   - section "Kernel contract": even layers are sliding-window (window 128),
 *     odd layers are full attention; the block table, the KV write index and
 *     the position are chosen by i % 2, and the KV buffer by i / 2; the
 *     attention-control tensors (RoPE cos/sin, a full and a trimmed
 *     sliding-window block table, an active mask, absolute and window-frame
 *     positions, two KV-update indices) are shared by all layers;
 *   - section "KV-cache layout (per-buffer, HMA-preserving)": one base-0 group
 *     buffer [2, num_blocks, kv, block, d] per layer pair, K half then V half;
 *     K is read through the packed FP8 view [.., block/2, d, 2] (or unpacked,
 *     like V), V is never packed;
 *   - section "Kernel contract": the cache is passed either as per-group K and
 *     V buffers or as stacked K_cache / V_cache, exactly one of the two forms
 *     (gk_kv_cache below).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless a parameter says "host".
 *   - The caller owns every buffer.  The library allocates nothing, keeps no
 *     state between calls other than a per-device error word (see
 *     gk_read_device_error), cached device properties and the fixed scratch
 *     array of gk_decode_attn_stack_static, and does not retain pointers after
 *     a call returns.
 *   - `stream` is a cudaStream_t passed as void*.  Calls are asynchronous and
 *     stream-ordered: a call returns after validating its arguments and
 *     enqueueing its kernels.  NULL means the legacy default stream.
 *   - Calls may be captured into a CUDA graph and replayed (the step's
 *     launches are chained by programmatic dependent launch, which capture
 *     keeps).  The first call on a device sets kernel attributes and caches
 *     device properties: make it before any capture.
 *   - Programmatic dependent launch at the start of an attention call: its
 *     first kernel (the planner) is launched as a programmatic dependent of
 *     whatever kernel precedes it in the stream and reads `active`, `pos` and
 *     `pos_w` as soon as it runs; everything else (q, the cache, the tables,
 *     the scales) is read only after that preceding kernel has completed.  A
 *     preceding kernel can let the planner start early only by opening
 *     dependent launch itself (griddepcontrol.launch_dependents, or
 *     cudaTriggerProgrammaticLaunchCompletion); kernels that never do so,
 *     which is the common case, are always complete first.  So a kernel that
 *     writes a call's `active`, `pos` or `pos_w` must not open dependent
 *     launch before those writes.  (gk_kv_append opens it early and writes
 *     none of them.)
 *   - Errors: every entry point returns a gk_status and never aborts, traps or
 *     prints.  Argument checks run on the host before anything is enqueued; a
 *     failed check enqueues nothing.  Launch failures map to GK_ERR_CUDA.
 *     Out-of-range data found on the device (a block id >= num_blocks, an
 *     update slot outside the buffer, a position beyond its table row) makes
 *     the kernel skip that access and set a bit in the device error word.
 *
 * Layouts (row-major, innermost last; Hkv = num_kv_heads, G = Hq / Hkv,
 * B = block_size, D = head_dim, NL = num_layers, Bt = batch):
 *   q, out            bf16  [NL, Bt, Hq, D]      q head h uses kv head h / G
 *   k_new, v_new      bf16  [NL, Bt, Hkv, D]
 *   cos, sin          fp32  [Bt, D/2]            rotate-half pairs (e, e + D/2)
 *   k_scale, v_scale  fp32  [NL]                 code = E4M3(x / scale), value = code * scale
 *   bt_full           int32 [Bt, max_blocks_full] physical block ids
 *   bt_swa            int32 [Bt, max_blocks_swa]  trimmed rows: first entry = block of the window start
 *   pos, pos_w        int32 [Bt]                  absolute / window-frame position of the new token
 *   upd_full, upd_swa int32 [Bt]                  flat slot = block * B + offset
 *   active            uint8 [Bt]                  0 = row skipped (no write, zero output)
 *   sinks             fp32  [NL, Hq] or NULL      optional attention-sink logits (see
 *                                                 gk_decode_attn_stack)
 *   kv                the cache (gk_kv_cache): group buffer j's K and V halves, each
 *                     num_blocks * Hkv * B * D bytes (one FP8 byte per element):
 *                     K byte (pb, h, t, e) = ((pb*Hkv + h)*(B/2) + t/2)*(2D) + 2e + (t & 1)
 *                                            (GK_K_PACKED, the view [.., B/2, D, 2])
 *                                          = ((pb*Hkv + h)*B + t)*D + e   (GK_K_PLAIN)
 *                     V byte (pb, h, t, e) = ((pb*Hkv + h)*B + t)*D + e
 * Supported shapes: D == 64, G == 8, B == 16 or a multiple of 32 up to 1024,
 * NL even and <= 128, Bt <= 8192.  Other shapes return GK_ERR_UNSUPPORTED.
 */
#ifndef GK_H
#define GK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GK_OK = 0,
    GK_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, inconsistent shape */
    GK_ERR_UNSUPPORTED = 2,   /* valid shape outside what this version implements */
    GK_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
    GK_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    GK_ERR_DEVICE_BOUNDS = 5, /* gk_read_device_error found a device-side error bit */
    GK_ERR_BUDGET = 6         /* gk_kv_budget: the KV budget is below the minimum */
} gk_status;

/* Device error-word bits (gk_read_device_error). */
#define GK_DEVERR_SLOT 0x1u     /* an update slot lies outside its group buffer: write skipped */
#define GK_DEVERR_BLOCK 0x2u    /* a block-table entry is outside [0, num_blocks): read skipped */
#define GK_DEVERR_POS 0x4u      /* a position is negative or beyond its table row */
#define GK_DEVERR_TIMEOUT 0x8u  /* a shared-memory barrier wait hit its iteration limit */
#define GK_DEVERR_PLAN 0x10u    /* the work plan did not fit the workspace */
#define GK_DEVERR_INGEST 0x20u  /* an ingest descriptor names a region or block out of range: copy skipped */

/* K layouts.  The page infers packed-ness from the K tensor's rank
 * (k.dim() == v.dim() + 1); across this ABI it is stated. */
#define GK_K_PACKED 0 /* K through the packed view [.., B/2, D, 2]: tokens 2p, 2p+1 interleaved */
#define GK_K_PLAIN 1  /* K laid out like V: [.., B, D] */

/*
 * gk_kv_cache -- the KV cache in one of the page's two forms ("GPT-OSS-120B
 * giga-kernel decode", section "Kernel contract": the kernel takes per-group
 * buffers or the stacked K_cache / V_cache and asserts that exactly one form
 * is present).  Set the pointers of exactly one form and leave the other form's
 * NULL; anything else is GK_ERR_INVALID_ARG.
 *   per-group: k_bufs[j], v_bufs[j] (HOST arrays of NL/2 DEVICE pointers) are
 *              the K and V halves of group buffer j, each 16-byte aligned;
 *   stacked:   k_cache, v_cache (DEVICE pointers, 16-byte aligned) hold the
 *              NL/2 halves back to back, [NL/2, num_blocks, Hkv, B, D] bytes:
 *              group j's K half starts at k_cache + j * num_blocks*Hkv*B*D.
 * Offsets are 64-bit throughout, so a stacked cache may exceed 4 GiB.
 * The library reads the pointer arrays during the call only.
 */
typedef struct {
    void *const *k_bufs;
    void *const *v_bufs;
    void *k_cache;
    void *v_cache;
    int32_t k_layout; /* GK_K_PACKED or GK_K_PLAIN */
} gk_kv_cache;

typedef struct {
    int32_t num_layers;      /* NL, even: layer pairs (2j, 2j+1) share group buffer j */
    int32_t batch;           /* Bt */
    int32_t num_q_heads;     /* Hq */
    int32_t num_kv_heads;    /* Hkv */
    int32_t head_dim;        /* D */
    int32_t block_size;      /* B, tokens per KV block */
    int32_t num_blocks;      /* blocks per group buffer (one global scalar) */
    int32_t window;          /* sliding window W of the even layers, in positions */
    int32_t max_blocks_full; /* columns of bt_full */
    int32_t max_blocks_swa;  /* columns of bt_swa; >= ceil((W + B - 1) / B) */
} gk_shape;

/*
 * gk_kv_append -- write the new token's K and V into the group buffers.
 * ("GPT-OSS-120B giga-kernel decode", sections "Kernel contract" (two
 * KV-update indices) and "KV-cache layout" (packed K, plain V).)
 *
 * For every layer i, active row b and kv head h:
 *   slot = (i even) ? upd_swa[b] : upd_full[b];  pb = slot / B;  t = slot % B
 *   k' = RoPE(k_new[i,b,h,:], cos[b], sin[b]) in IEEE fp32, no fused multiply-add:
 *        k'_e = k_e*c_e - k_{e+D/2}*s_e,  k'_{e+D/2} = k_{e+D/2}*c_e + k_e*s_e
 *   K_{i/2}[(pb,h,t,e)] = E4M3(k'_e / k_scale[i])   (fp32 division, RNE; kv->k_layout)
 *   V_{i/2}[(pb,h,t,e)] = E4M3(v_new[i,b,h,e] / v_scale[i])
 * E4M3 = round to nearest, ties to even mantissa, saturating to +-448; NaN -> 0x7F.
 * Inactive rows write nothing.  No other byte of any buffer changes.
 * Returns GK_ERR_INVALID_ARG for null pointers, inconsistent shapes, k_new,
 * v_new, cos or sin not 16-byte aligned, or a kv that does not hold exactly
 * one form.
 */
gk_status gk_kv_append(const gk_shape *shape, const void *k_new, const void *v_new,
                       const float *cos, const float *sin, const float *k_scale,
                       const float *v_scale, const int32_t *upd_full, const int32_t *upd_swa,
                       const uint8_t *active, const gk_kv_cache *kv, void *stream);

/*
 * gk_attn_workspace_bytes -- recommended workspace size for gk_decode_attn_stack.
 * host_positions is reserved (may be NULL; not read).  Any workspace of at
 * least gk_attn_workspace_min_bytes() works: the planner fits its split-KV
 * partials into whatever capacity it is given (less capacity -> fewer, longer
 * splits).  Returns 0 for an invalid or unsupported shape.
 */
size_t gk_attn_workspace_bytes(const gk_shape *shape, const int32_t *host_positions);
size_t gk_attn_workspace_min_bytes(const gk_shape *shape);

/*
 * gk_decode_attn_stack -- GQA decode attention for all layers of one step.
 * ("GPT-OSS-120B giga-kernel decode", section "Kernel contract"; the
 * split-KV combine is the flash-decoding log-sum-exp merge.)
 *
 * For every layer i, row b, q head h (kv head kvh = h / G):
 *   i odd  (full):   keys t in [0, pos[b]] through row b of bt_full
 *   i even (window): keys t in [max(0, pos_w[b] - W + 1), pos_w[b]] through row b of bt_swa
 *   q' = RoPE(q[i,b,h,:], cos[b], sin[b]);  k_t = decode(K_{i/2}) * k_scale[i];
 *   v_t = decode(V_{i/2}) * v_scale[i];  s_t = q'.k_t / sqrt(D)
 *   out[i,b,h,:] = bf16_rne( sum_t softmax(s)_t v_t );  out_f32 (optional) gets the fp32 value.
 * Attention sinks (GPT-OSS; not on the pages): when sinks is not NULL, the
 * per-layer, per-head logit sinks[i*Hq + h] (natural-log units, like s_t)
 * joins the softmax denominator and carries no value:
 *   out = sum_t e^(s_t) v_t / (sum_t e^(s_t) + e^(sinks[i*Hq + h])).
 * Inactive rows get zeros.  The cache is read, never written: run gk_kv_append
 * first on the same stream when the new token must be attended to.
 * workspace: device memory, 256-byte aligned, ws_bytes >= gk_attn_workspace_min_bytes;
 * it is overwritten by every call (do not share one workspace between calls
 * that may overlap on the device).  Calls issued one after another on one
 * stream are ordered: a call runs a planner, the attention grid and, when
 * rows are split across warps, a combine grid, chained by programmatic
 * dependent launches, and the next call's planner starts only once this
 * call no longer reads the workspace.
 * Returns GK_ERR_WORKSPACE for a missing/small/misaligned workspace,
 * GK_ERR_INVALID_ARG for null or non-16-byte-aligned tensors (sinks: 4-byte)
 * or a kv that does not hold exactly one form.
 */
gk_status gk_decode_attn_stack(const gk_shape *shape, const void *q, const gk_kv_cache *kv,
                               const float *k_scale, const float *v_scale,
                               const float *cos, const float *sin, const int32_t *bt_full,
                               const int32_t *bt_swa, const int32_t *pos, const int32_t *pos_w,
                               const uint8_t *active, const float *sinks, void *out, float *out_f32,
                               void *workspace, size_t ws_bytes, void *stream);

/*
 * gk_decode_step -- the whole decode step in two launches instead of three:
 * gk_kv_append followed by gk_decode_attn_stack, with the same arguments and
 * results (KV bytes identical to gk_kv_append's, outputs to
 * gk_decode_attn_stack's).  ("GPT-OSS-120B giga-kernel decode", section
 * "Kernel contract": one program consumes the new token's K/V, both update
 * indices and the attention-control tensors per step.)
 * The append runs in CTAs beside the planner's, in the planner's launch; the
 * attention launch starts while that grid runs and reads the plan and the
 * cache only once the whole grid, append included, is complete.  The append
 * starts once the work queued before the call is complete.  Inactive rows
 * write nothing and output zeros.  Errors: those of gk_kv_append and
 * gk_decode_attn_stack.
 */
gk_status gk_decode_step(const gk_shape *shape, const void *q, const void *k_new,
                         const void *v_new, const float *cos, const float *sin,
                         const float *k_scale, const float *v_scale, const int32_t *upd_full,
                         const int32_t *upd_swa, const int32_t *bt_full, const int32_t *bt_swa,
                         const int32_t *pos, const int32_t *pos_w, const uint8_t *active,
                         const float *sinks, const gk_kv_cache *kv, void *out, float *out_f32,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * gk_decode_attn_stack_static -- gk_decode_attn_stack without a caller
 * workspace.  (No counterpart on the pages: an addition of this library.)
 *
 * For callers that cannot allocate device memory: a host framework that
 * budgets every device byte before the first step, a plugin or foreign-language
 * boundary with no device allocator, or a step that must not risk the
 * synchronisation and failure modes of cudaMalloc.  The library holds a
 * GK_STATIC_SCRATCH_BYTES device array of its own on every GPU that loads it,
 * until the process exits; this call allocates nothing and uses that array as
 * the workspace.  Arguments and results are those of gk_decode_attn_stack
 * (the caller still passes inputs and outputs).
 *   - Returns GK_ERR_WORKSPACE when the shape needs more than
 *     GK_STATIC_SCRATCH_BYTES of workspace (gk_attn_workspace_min_bytes); no
 *     shape the library accepts does (the largest needs under 1 MiB).  An
 *     array smaller than the recommended workspace only means fewer split-KV
 *     chunks.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress, with the caller's device current; no work is
 *     enqueued), so the address stays right after cudaDeviceReset or in a
 *     context other than the primary one.  The first call in a context may
 *     also load the library's device code there: make one call on each device
 *     before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; each call re-initialises what it needs.  Calls that may overlap
 *     on the GPU (different streams without ordering between them) race on the
 *     array and give wrong results: order them.
 */
#define GK_STATIC_SCRATCH_BYTES (16u << 20)
gk_status gk_decode_attn_stack_static(const gk_shape *shape, const void *q,
                                      const gk_kv_cache *kv, const float *k_scale,
                                      const float *v_scale, const float *cos, const float *sin,
                                      const int32_t *bt_full, const int32_t *bt_swa,
                                      const int32_t *pos, const int32_t *pos_w,
                                      const uint8_t *active, const float *sinks, void *out,
                                      float *out_f32,
                                      void *stream);

/*
 * gk_e4m3_quantize -- codes[i] = E4M3(x[i] / scale) with the same fp32
 * division and encoder as gk_kv_append (for bulk KV ingest and checks).
 * x, codes: device arrays of n elements.
 */
gk_status gk_e4m3_quantize(const float *x, float scale, uint8_t *codes, int64_t n, void *stream);

/*
 * gk_read_device_error -- synchronise `stream`, return the current device's
 * error word (GK_DEVERR_* bits) in *bits, and clear it if `clear` != 0.
 * Returns GK_ERR_DEVICE_BOUNDS when any bit was set, GK_OK otherwise.
 */
gk_status gk_read_device_error(void *stream, uint32_t *bits, int clear);

/*
 * gk_kv_budget -- size the KV pool (host only; no GPU call).
 * ("determine_available_memory design", sections "Heuristic formula" and
 * "Minimum KV guard"; "GPT-OSS-120B giga-kernel decode", section "KV budget".)
 *
 *   total_budget = floor(total_bytes * gpu_memory_utilization)
 *   kv_budget    = max(total_budget - used_bytes, 0)
 *   cap          = floor(total_budget * cap_fraction)      (cap_fraction 0.30 by default on
 *                                                            the page; 1.0 = no cap)
 *   available    = max(min(kv_budget, cap), 0)
 * *available_bytes receives `available`.  If shape is not NULL, *num_blocks
 * receives floor(available / bytes_per_block) with bytes_per_block =
 * (num_layers/2) * 2 * num_kv_heads * block_size * head_dim (one byte per FP8
 * element, K and V halves of every group buffer); shape->num_blocks and the
 * table sizes are not read.  Returns GK_ERR_BUDGET when available is below
 * min_budget_gib GiB (the page's minimum-KV guard, 1.0 by default) or yields
 * fewer than 2 blocks (one usable block plus the padding block); both outputs
 * are still written.  GK_ERR_INVALID_ARG for gmu or cap_fraction outside
 * (0, 1], negative min_budget_gib, or null outputs.
 */
gk_status gk_kv_budget(uint64_t total_bytes, uint64_t used_bytes, double gpu_memory_utilization,
                       double cap_fraction, double min_budget_gib, const gk_shape *shape,
                       uint64_t *available_bytes, int64_t *num_blocks);

/*
 * Disaggregated-inference KV landing ("GPT-OSS-120B giga-kernel decode",
 * section "DI wiring (NIXL)").  A prefill engine's KV blocks land on the group
 * buffer block the decode kernel reads: each group buffer's K half and V half
 * is one region of num_blocks blocks of block_len = kv * block * d bytes (one
 * layer-pair block), and block b of a region is base + b * block_len.  The
 * transport itself is not part of this library: gk_kv_ingest is the local
 * landing copy that stands in for it.
 */
typedef struct {
    void *base;         /* device address of block 0 */
    uint64_t length;    /* bytes: num_blocks * block_len */
    uint64_t block_len; /* bytes of one block: num_kv_heads * block_size * head_dim */
} gk_kv_region;

/*
 * gk_kv_regions -- the region list of a per-layer KV binding (host only).
 * Layers are taken in order 0..NL-1, each adding its K half and then its V
 * half as a region unless a region with the same base address is already
 * listed: buffers shared by paired layers are de-duplicated by base address,
 * which for the page's layout gives 2 * NL/2 regions K_0, V_0, K_1, V_1, ...
 * layer_k, layer_v: HOST arrays of NL device addresses (16-byte aligned), the
 * K and V halves layer i is bound to.  out: HOST array of `capacity` regions.
 * *count receives the number of distinct regions even when it exceeds
 * capacity (then GK_ERR_INVALID_ARG and only `capacity` are written).
 */
gk_status gk_kv_regions(const gk_shape *shape, void *const *layer_k, void *const *layer_v,
                        gk_kv_region *out, int32_t capacity, int32_t *count);

/*
 * gk_kv_ingest -- land n transferred blocks: for d in [0, n), copy block_len
 * bytes from src + d * block_len to regions[dst_region[d]].base +
 * dst_block[d] * block_len.
 *   regions: HOST array of n_regions (<= 128) regions sharing one block_len
 *            (a multiple of 16); dst_region, dst_block: DEVICE int32 [n];
 *   src:     n * block_len bytes, 16-byte aligned, in device memory or in host
 *            memory the device can address (pinned, mapped); plain pageable
 *            host memory is refused with GK_ERR_INVALID_ARG.
 * Descriptors must name distinct destination blocks (the copies run
 * concurrently).  A descriptor whose region or block is out of range is
 * skipped on the device and sets GK_DEVERR_INGEST.  n == 0 enqueues nothing.
 */
gk_status gk_kv_ingest(const gk_kv_region *regions, int32_t n_regions, const int32_t *dst_region,
                       const int32_t *dst_block, int64_t n, const void *src, void *stream);

/*
 * gk_di_blocks -- which of a prompt's blocks the decode engine needs
 * (host only; "DI wiring (NIXL)", the sliding-window truncation fix: both
 * engines operate at N - 1).  For a prompt of N >= 1 tokens whose last token
 * the decode engine recomputes at position N - 1, the transferred keys are
 * positions 0 .. N-2:
 *   full layers:   row blocks [0, *full_count),  full_count = ceil((N - 1) / B);
 *   window layers: row blocks [*swa_first, *swa_first + *swa_count) (absolute
 *                  block numbers), the blocks of keys max(0, N - W) .. N - 2,
 *                  i.e. the window of position N - 1 without the new token;
 *                  swa_first = max(0, N - W) / B.
 * Computing the window for length N instead (keys from N - W + 1) drops block
 * swa_first exactly when N >= W and N % B == B - 1 (for B dividing W): the
 * block the page's fix keeps.  GK_ERR_INVALID_ARG for N < 1, B < 1, W < 1 or
 * null outputs.
 */
gk_status gk_di_blocks(int64_t num_tokens, int32_t block_size, int32_t window,
                       int64_t *full_count, int64_t *swa_first, int64_t *swa_count);

/* Human-readable name of a status code (static string). */
const char *gk_status_str(gk_status status);

/* Library ABI version (3: the cache is passed as a gk_kv_cache; optional sinks). */
int32_t gk_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GK_H */
