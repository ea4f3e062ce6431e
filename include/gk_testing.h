/*
 * gk_testing.h -- test hooks of the GB300 decode-attention library.  Not part
 * of the decode path; no counterpart on the pages.
 */
#ifndef GK_TESTING_H
#define GK_TESTING_H

#include "gk.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gk_selftest_wait_timeout -- exercise the bounded shared-memory barrier wait
 * that every pipeline stage of the attention kernel uses: one warp waits on a
 * barrier phase that nothing completes, gives up after limit_ns nanoseconds of
 * device wall time (1 us .. 1 s), sets GK_DEVERR_TIMEOUT and returns.  Nothing
 * faults or hangs; the context stays usable.  Synchronises `stream` and
 * returns the error word in *bits (cleared afterwards), with
 * GK_ERR_DEVICE_BOUNDS when a bit is set.
 */
gk_status gk_selftest_wait_timeout(uint64_t limit_ns, void *stream, uint32_t *bits);

/*
 * gk_selftest_decode_attn_split -- gk_decode_attn_stack with the split-KV
 * chunk length fixed by the caller instead of chosen by the planner, so that
 * tests can put a given number of flash-decoding partials on a row (up to the
 * cap of 64 per (layer, row, kv head)) and check their combine.  Arguments
 * are those of gk_decode_attn_stack plus split_tokens: a power of two from 512
 * to 512 << 21 (GK_ERR_INVALID_ARG otherwise).  Every full-layer row with
 * L > split_tokens keys is cut into ceil(L / split_tokens) chunks; the length
 * is still raised where a row would need more than 64 chunks or the workspace
 * cannot hold the partial records (the length used is header word 4 of the
 * workspace), and no chunk is cut into last-wave pieces.
 */
gk_status gk_selftest_decode_attn_split(const gk_shape *shape, const void *q,
                                        const gk_kv_cache *kv, const float *k_scale,
                                        const float *v_scale, const float *cos, const float *sin,
                                        const int32_t *bt_full, const int32_t *bt_swa,
                                        const int32_t *pos, const int32_t *pos_w,
                                        const uint8_t *active, const float *sinks, void *out,
                                        float *out_f32, void *workspace, size_t ws_bytes,
                                        int32_t split_tokens, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GK_TESTING_H */
