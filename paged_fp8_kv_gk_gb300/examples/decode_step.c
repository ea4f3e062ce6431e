/*
 * decode_step.c -- one decode step through the C ABI alone (include/gk.h), no
 * Python: the program reads a step's inputs from raw little-endian files in a
 * directory, uploads them, runs gk_kv_append and gk_decode_attn_stack (or the
 * gk_decode_step) on CUDA device 0, checks the device error word
 * and writes the output and the group buffers back.
 *
 *   usage: decode_step <dir> [split|fused]
 *     split (default): gk_kv_append, then gk_decode_attn_stack
 *     fused:           gk_decode_step (append and attention in one launch)
 *   inputs  (in <dir>): shape.bin (gk_shape, 10 x int32), q.bin, k_new.bin,
 *     v_new.bin (bf16), cos.bin, sin.bin, k_scale.bin, v_scale.bin (fp32),
 *     bt_full.bin, bt_swa.bin, pos.bin, pos_w.bin, upd_full.bin, upd_swa.bin
 *     (int32), active.bin (uint8), cache_<j>.bin (group buffer j: K half then
 *     V half, uint8) for j < num_layers / 2; optional sinks.bin (fp32
 *     [num_layers, num_q_heads] attention-sink logits)
 *   outputs (in <dir>): out.bin (bf16 [NL, Bt, Hq, D]), cache_out_<j>.bin
 *
 * Build (see the package's build step for libgk.so):
 *   cc -O2 -I<repo>/include decode_step.c -o decode_step \
 *      -L<repo>/paged_fp8_kv_gk_gb300/_build -lgk -L<cuda>/lib64 -lcudart
 * Exit status: 0 on success, 1 on a usage or I/O error, 2 on a library or CUDA error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gk.h"

static void *read_file(const char *dir, const char *name, size_t *size) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  long n = ftell(f);
  fseek(f, 0, SEEK_SET);
  void *buf = malloc(n > 0 ? (size_t)n : 1);
  if (buf && n > 0 && fread(buf, 1, (size_t)n, f) != (size_t)n) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  if (size) *size = (size_t)n;
  return buf;
}

static int write_file(const char *dir, const char *name, const void *data, size_t size) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return -1;
  size_t w = fwrite(data, 1, size, f);
  fclose(f);
  return w == size ? 0 : -1;
}

/* Read a file into fresh device memory. */
static void *upload(const char *dir, const char *name, size_t *size) {
  size_t n = 0;
  void *h = read_file(dir, name, &n);
  if (!h) return NULL;
  void *d = NULL;
  if (cudaMalloc(&d, n > 0 ? n : 16) != cudaSuccess ||
      cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) {
    free(h);
    return NULL;
  }
  free(h);
  if (size) *size = n;
  return d;
}

int main(int argc, char **argv) {
  int fused = 0;
  if (argc == 3 && strcmp(argv[2], "fused") == 0)
    fused = 1;
  else if (!(argc == 2 || (argc == 3 && strcmp(argv[2], "split") == 0))) {
    fprintf(stderr, "usage: %s <dir> [split|fused]\n", argv[0]);
    return 1;
  }
  const char *dir = argv[1];
  size_t n = 0;
  gk_shape *sh = (gk_shape *)read_file(dir, "shape.bin", &n);
  if (!sh || n != sizeof(gk_shape)) {
    fprintf(stderr, "shape.bin missing or of the wrong size\n");
    return 1;
  }
  const char *names[] = {"q.bin", "k_new.bin", "v_new.bin", "cos.bin", "sin.bin",
                         "k_scale.bin", "v_scale.bin", "bt_full.bin", "bt_swa.bin", "pos.bin",
                         "pos_w.bin", "upd_full.bin", "upd_swa.bin", "active.bin"};
  void *d[14];
  for (int k = 0; k < 14; ++k) {
    d[k] = upload(dir, names[k], NULL);
    if (!d[k]) {
      fprintf(stderr, "cannot read or upload %s\n", names[k]);
      return 1;
    }
  }
  size_t sinks_bytes = 0;
  const float *sinks = NULL;  /* optional */
  {
    char path[4096];
    snprintf(path, sizeof(path), "%s/sinks.bin", dir);
    FILE *f = fopen(path, "rb");
    if (f) {
      fclose(f);
      sinks = (const float *)upload(dir, "sinks.bin", &sinks_bytes);
      if (!sinks ||
          sinks_bytes != (size_t)sh->num_layers * sh->num_q_heads * sizeof(float)) {
        fprintf(stderr, "sinks.bin unreadable or of the wrong size\n");
        return 1;
      }
    }
  }
  const int groups = sh->num_layers / 2;
  const size_t half = (size_t)sh->num_blocks * sh->num_kv_heads * sh->block_size * sh->head_dim;
  void **kb = (void **)calloc((size_t)groups, sizeof(void *));
  void **vb = (void **)calloc((size_t)groups, sizeof(void *));
  void **bufs = (void **)calloc((size_t)groups, sizeof(void *));
  for (int j = 0; j < groups; ++j) {
    char name[64];
    snprintf(name, sizeof(name), "cache_%d.bin", j);
    size_t got = 0;
    bufs[j] = upload(dir, name, &got);
    if (!bufs[j] || got != 2 * half) {
      fprintf(stderr, "%s missing or of the wrong size\n", name);
      return 1;
    }
    kb[j] = bufs[j];                    /* K half, then V half of group buffer j */
    vb[j] = (uint8_t *)bufs[j] + half;
  }
  gk_kv_cache kv;
  memset(&kv, 0, sizeof(kv));
  kv.k_bufs = kb;
  kv.v_bufs = vb;
  kv.k_layout = GK_K_PACKED;

  const size_t out_bytes =
      (size_t)sh->num_layers * sh->batch * sh->num_q_heads * sh->head_dim * 2;
  void *out = NULL, *ws = NULL;
  const size_t ws_bytes = gk_attn_workspace_bytes(sh, NULL);
  if (ws_bytes == 0 || cudaMalloc(&out, out_bytes) != cudaSuccess ||
      cudaMalloc(&ws, ws_bytes) != cudaSuccess) {
    fprintf(stderr, "unsupported shape or allocation failure\n");
    return 2;
  }

  gk_status st;
  if (fused) {
    st = gk_decode_step(sh, d[0], d[1], d[2], (const float *)d[3], (const float *)d[4],
                        (const float *)d[5], (const float *)d[6], (const int32_t *)d[11],
                        (const int32_t *)d[12], (const int32_t *)d[7], (const int32_t *)d[8],
                        (const int32_t *)d[9], (const int32_t *)d[10], (const uint8_t *)d[13],
                        sinks, &kv, out, NULL, ws, ws_bytes, NULL);
  } else {
    st = gk_kv_append(sh, d[1], d[2], (const float *)d[3], (const float *)d[4],
                      (const float *)d[5], (const float *)d[6], (const int32_t *)d[11],
                      (const int32_t *)d[12], (const uint8_t *)d[13], &kv, NULL);
    if (st == GK_OK)
      st = gk_decode_attn_stack(sh, d[0], &kv, (const float *)d[5], (const float *)d[6],
                                (const float *)d[3], (const float *)d[4], (const int32_t *)d[7],
                                (const int32_t *)d[8], (const int32_t *)d[9],
                                (const int32_t *)d[10], (const uint8_t *)d[13], sinks, out,
                                NULL, ws, ws_bytes, NULL);
  }
  uint32_t bits = 0;
  if (st == GK_OK) st = gk_read_device_error(NULL, &bits, 1);
  if (st != GK_OK) {
    fprintf(stderr, "library call failed: %s (device error bits 0x%x)\n", gk_status_str(st),
            bits);
    return 2;
  }

  void *h = malloc(out_bytes > 2 * half ? out_bytes : 2 * half);
  if (!h || cudaMemcpy(h, out, out_bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
      write_file(dir, "out.bin", h, out_bytes) != 0) {
    fprintf(stderr, "cannot write out.bin\n");
    return 2;
  }
  for (int j = 0; j < groups; ++j) {
    char name[64];
    snprintf(name, sizeof(name), "cache_out_%d.bin", j);
    if (cudaMemcpy(h, bufs[j], 2 * half, cudaMemcpyDeviceToHost) != cudaSuccess ||
        write_file(dir, name, h, 2 * half) != 0) {
      fprintf(stderr, "cannot write %s\n", name);
      return 2;
    }
  }
  printf("decode_step ok (%s%s): abi %d, %d layers x %d rows\n", fused ? "fused" : "split",
         sinks ? ", sinks" : "", gk_abi_version(), sh->num_layers, sh->batch);
  return 0;
}
