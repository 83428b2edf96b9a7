/*
 * A plain C99 client of the FLCE C ABI: no C++, no torch, only flce.h and the
 * CUDA runtime's C API for device memory. It shows that the boundary is usable
 * from any language that can call C, and it is driven by tests/test_c_client.py.
 *
 *   flce_client host N H V
 *       host-side entry points only (no GPU needed): prints the default
 *       parameters, the workspace sizes of the three modes, the status strings
 *       and the code returned for a call without buffers.
 *   flce_client gpu IN OUT
 *       reads one problem from IN, allocates its device buffers with
 *       cudaMalloc, runs flce_forward_backward on the legacy default stream and
 *       writes the results to OUT.
 *   flce_client vp IN OUT S
 *       the same problem with W split by vocabulary rows into S shards, run
 *       one after another: every shard's flce_vp_forward into one [S][4][N]
 *       partials buffer, then every shard's flce_vp_backward, adding into one
 *       fp32 grad_h and into its own rows of grad_W. OUT as for gpu, except
 *       that grad_h is fp32 (float grad_h[N*H]).
 *   flce_client vps IN OUT S
 *       as vp, with FLCE_FLAG_VP_STORED: every shard keeps its logits between
 *       its two calls, in a workspace of its own.
 *
 * IN (little endian): int64 N, H, V, chunk_rows; float softcap, out_mult;
 *   uint16 h[N*H] (bf16 bits), uint16 W[V*H], int64 labels[N], float gW0[V*H].
 * OUT: float loss, token_accuracy; int32 return code, device status;
 *   int64 predicted[N]; uint16 grad_h[N*H]; float grad_W[V*H].
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "flce.h"

static int host_mode(int64_t n, int64_t h, int64_t v) {
  flce_params p;
  flce_default_params(&p);
  printf("default softcap=%g out_mult=%g ignore_index=%lld reduction=%d grad_scale=%g chunk_rows=%lld\n",
         (double)p.softcap, (double)p.out_mult, (long long)p.ignore_index, p.reduction, (double)p.grad_scale,
         (long long)p.chunk_rows);
  p.n_rows = n;
  p.hidden = h;
  p.vocab = v;
  printf("workspace ce_only=%zu forward=%zu forward_backward=%zu\n",
         flce_workspace_size(&p, FLCE_MODE_CE_ONLY, 0, 0), flce_workspace_size(&p, FLCE_MODE_FORWARD, 0, 0),
         flce_workspace_size(&p, FLCE_MODE_FORWARD_BACKWARD, 1, 1));
  {
    flce_params bad = p;
    bad.hidden = 12; /* not a multiple of 8 */
    printf("workspace bad_hidden=%zu\n", flce_workspace_size(&bad, FLCE_MODE_FORWARD_BACKWARD, 1, 1));
  }
  {
    const int codes[] = {FLCE_OK, FLCE_ERR_ARG, FLCE_ERR_ALIGN, FLCE_ERR_WORKSPACE, FLCE_ERR_UNSUPPORTED,
                         FLCE_ERR_CUDA, FLCE_ERR_LABEL, FLCE_ERR_TIMEOUT};
    size_t i;
    for (i = 0; i < sizeof(codes) / sizeof(codes[0]); ++i) printf("status %d %s\n", codes[i], flce_status_string(codes[i]));
  }
  printf("no_buffers %d\n", flce_forward_backward(&p, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL));
  printf("kernel0 %s\n", flce_kernel_name(0));
  return 0;
}

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }
static int write_all(FILE* f, const void* src, size_t bytes) { return fwrite(src, 1, bytes, f) == bytes; }

#define CK(x)                                                        \
  do {                                                               \
    if ((x) != cudaSuccess) {                                        \
      fprintf(stderr, "CUDA call failed at line %d: %s\n", __LINE__, #x); \
      return 2;                                                      \
    }                                                                \
  } while (0)

static int gpu_mode(const char* in_path, const char* out_path) {
  int64_t hdr[4];
  float fl[2];
  FILE* f = fopen(in_path, "rb");
  if (!f || !read_all(f, hdr, sizeof hdr) || !read_all(f, fl, sizeof fl)) return 3;
  {
    const int64_t n = hdr[0], h = hdr[1], v = hdr[2];
    const size_t nh = (size_t)(n * h), vh = (size_t)(v * h);
    uint16_t* h_h = malloc(nh * 2);
    uint16_t* w_h = malloc(vh * 2);
    int64_t* y_h = malloc((size_t)n * 8);
    float* gw_h = malloc(vh * 4);
    int64_t* pred_h = malloc((size_t)n * 8);
    uint16_t* gh_h = malloc(nh * 2);
    void *h_d, *w_d, *y_d, *gw_d, *pred_d, *gh_d, *ws_d, *sc_d;
    float sc[2];
    int32_t status = -1;
    int rc;
    size_t ws_bytes;
    flce_params p;
    if (!h_h || !w_h || !y_h || !gw_h || !pred_h || !gh_h) return 4;
    if (!read_all(f, h_h, nh * 2) || !read_all(f, w_h, vh * 2) || !read_all(f, y_h, (size_t)n * 8) ||
        !read_all(f, gw_h, vh * 4))
      return 3;
    fclose(f);

    flce_default_params(&p);
    p.n_rows = n;
    p.hidden = h;
    p.vocab = v;
    p.chunk_rows = hdr[3];
    p.softcap = fl[0];
    p.out_mult = fl[1];
    ws_bytes = flce_workspace_size(&p, FLCE_MODE_FORWARD_BACKWARD, 1, 1);
    if (ws_bytes == 0) return 5;

    CK(cudaMalloc(&h_d, nh * 2));
    CK(cudaMalloc(&w_d, vh * 2));
    CK(cudaMalloc(&y_d, (size_t)n * 8));
    CK(cudaMalloc(&gw_d, vh * 4));
    CK(cudaMalloc(&pred_d, (size_t)n * 8));
    CK(cudaMalloc(&gh_d, nh * 2));
    CK(cudaMalloc(&ws_d, ws_bytes));
    CK(cudaMalloc(&sc_d, 2 * sizeof(float)));
    CK(cudaMemcpy(h_d, h_h, nh * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(w_d, w_h, vh * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(y_d, y_h, (size_t)n * 8, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(gw_d, gw_h, vh * 4, cudaMemcpyHostToDevice));

    rc = flce_forward_backward(&p, h_d, w_d, (const int64_t*)y_d, (float*)sc_d, (float*)sc_d + 1,
                               (int64_t*)pred_d, gh_d, (float*)gw_d, ws_d, ws_bytes, NULL);
    if (rc == FLCE_OK) rc = flce_get_status(ws_d, NULL, &status);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(sc, sc_d, sizeof sc, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(pred_h, pred_d, (size_t)n * 8, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gh_h, gh_d, nh * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gw_h, gw_d, vh * 4, cudaMemcpyDeviceToHost));

    f = fopen(out_path, "wb");
    if (!f) return 6;
    {
      const int32_t codes[2] = {rc, status};
      if (!write_all(f, sc, sizeof sc) || !write_all(f, codes, sizeof codes) ||
          !write_all(f, pred_h, (size_t)n * 8) || !write_all(f, gh_h, nh * 2) || !write_all(f, gw_h, vh * 4))
        return 6;
    }
    fclose(f);
    cudaFree(h_d);
    cudaFree(w_d);
    cudaFree(y_d);
    cudaFree(gw_d);
    cudaFree(pred_d);
    cudaFree(gh_d);
    cudaFree(ws_d);
    cudaFree(sc_d);
    free(h_h);
    free(w_h);
    free(y_h);
    free(gw_h);
    free(pred_h);
    free(gh_h);
    printf("rc %d status %d loss %.9g\n", rc, (int)status, (double)sc[0]);
    return rc == FLCE_OK && status == 0 ? 0 : 1;
  }
}

static int vp_mode(const char* in_path, const char* out_path, int S, int stored) {
  int64_t hdr[4];
  float fl[2];
  FILE* f = fopen(in_path, "rb");
  if (S < 1 || S > 64) return 7;
  if (!f || !read_all(f, hdr, sizeof hdr) || !read_all(f, fl, sizeof fl)) return 3;
  {
    const int64_t n = hdr[0], h = hdr[1], v = hdr[2];
    const size_t nh = (size_t)(n * h), vh = (size_t)(v * h);
    uint16_t* h_h = malloc(nh * 2);
    uint16_t* w_h = malloc(vh * 2);
    int64_t* y_h = malloc((size_t)n * 8);
    float* gw_h = malloc(vh * 4);
    int64_t* pred_h = malloc((size_t)n * 8);
    float* gh_h = malloc(nh * 4);
    int64_t offsets[65];
    void *h_d, *w_d, *y_d, *gw_d, *pred_d, *gh_d, *ws_d, *sc_d, *part_d;
    void* ws_k[64];        /* the workspace of each shard's calls */
    size_t wsb_k[64];
    float sc[2];
    int32_t status = -1;
    int rc = FLCE_OK;
    size_t ws_bytes = 0;
    int k;
    flce_params p;
    if (!h_h || !w_h || !y_h || !gw_h || !pred_h || !gh_h) return 4;
    if (!read_all(f, h_h, nh * 2) || !read_all(f, w_h, vh * 2) || !read_all(f, y_h, (size_t)n * 8) ||
        !read_all(f, gw_h, vh * 4))
      return 3;
    fclose(f);
    for (k = 0; k <= S; ++k) offsets[k] = (int64_t)k * v / S;

    flce_default_params(&p);
    p.n_rows = n;
    p.hidden = h;
    p.chunk_rows = hdr[3];
    p.softcap = fl[0];
    p.out_mult = fl[1];
    if (stored) p.flags |= FLCE_FLAG_VP_STORED;
    for (k = 0; k < S; ++k) { /* one workspace as large as any shard's call needs, or one per shard */
      size_t a, b;
      p.vocab = offsets[k + 1] - offsets[k];
      a = flce_vp_workspace_size(&p, 0, 0, 0);
      b = flce_vp_workspace_size(&p, 1, 1, 1);
      if (a == 0 || b == 0) return 5;
      wsb_k[k] = a > b ? a : b;
      if (wsb_k[k] > ws_bytes) ws_bytes = wsb_k[k];
    }

    CK(cudaMalloc(&h_d, nh * 2));
    CK(cudaMalloc(&w_d, vh * 2));
    CK(cudaMalloc(&y_d, (size_t)n * 8));
    CK(cudaMalloc(&gw_d, vh * 4));
    CK(cudaMalloc(&pred_d, (size_t)n * 8));
    CK(cudaMalloc(&gh_d, nh * 4));
    CK(cudaMalloc(&ws_d, ws_bytes));
    for (k = 0; k < S; ++k) {
      if (stored) {
        CK(cudaMalloc(&ws_k[k], wsb_k[k]));
      } else {
        ws_k[k] = ws_d;
        wsb_k[k] = ws_bytes;
      }
    }
    CK(cudaMalloc(&sc_d, 2 * sizeof(float)));
    CK(cudaMalloc(&part_d, (size_t)S * 4 * (size_t)n * sizeof(float)));
    CK(cudaMemcpy(h_d, h_h, nh * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(w_d, w_h, vh * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(y_d, y_h, (size_t)n * 8, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(gw_d, gw_h, vh * 4, cudaMemcpyHostToDevice));
    CK(cudaMemset(gh_d, 0, nh * 4));

    for (k = 0; k < S && rc == FLCE_OK; ++k) {
      p.vocab = offsets[k + 1] - offsets[k];
      rc = flce_vp_forward(&p, offsets[k], v, h_d, (const uint16_t*)w_d + offsets[k] * h, (const int64_t*)y_d,
                           (float*)part_d + (size_t)k * 4 * (size_t)n, ws_k[k], wsb_k[k], NULL);
    }
    for (k = 0; k < S && rc == FLCE_OK; ++k) {
      p.vocab = offsets[k + 1] - offsets[k];
      rc = flce_vp_backward(&p, offsets[k], v, S, offsets, (const float*)part_d, h_d,
                            (const uint16_t*)w_d + offsets[k] * h, (const int64_t*)y_d, (float*)sc_d,
                            (float*)sc_d + 1, (int64_t*)pred_d, NULL, (float*)gh_d, (float*)gw_d + offsets[k] * h,
                            ws_k[k], wsb_k[k], NULL);
    }
    for (k = 0; k < S && rc == FLCE_OK; ++k) { /* every shard's status word (one shared word without stored) */
      int32_t st = 0;
      rc = flce_get_status(ws_k[k], NULL, &st);
      status = (k == 0 ? 0 : status) | st;
    }
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(sc, sc_d, sizeof sc, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(pred_h, pred_d, (size_t)n * 8, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gh_h, gh_d, nh * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gw_h, gw_d, vh * 4, cudaMemcpyDeviceToHost));

    f = fopen(out_path, "wb");
    if (!f) return 6;
    {
      const int32_t codes[2] = {rc, status};
      if (!write_all(f, sc, sizeof sc) || !write_all(f, codes, sizeof codes) ||
          !write_all(f, pred_h, (size_t)n * 8) || !write_all(f, gh_h, nh * 4) || !write_all(f, gw_h, vh * 4))
        return 6;
    }
    fclose(f);
    cudaFree(h_d);
    cudaFree(w_d);
    cudaFree(y_d);
    cudaFree(gw_d);
    cudaFree(pred_d);
    cudaFree(gh_d);
    cudaFree(ws_d);
    if (stored)
      for (k = 0; k < S; ++k) cudaFree(ws_k[k]);
    cudaFree(sc_d);
    cudaFree(part_d);
    free(h_h);
    free(w_h);
    free(y_h);
    free(gw_h);
    free(pred_h);
    free(gh_h);
    printf("rc %d status %d loss %.9g\n", rc, (int)status, (double)sc[0]);
    return rc == FLCE_OK && status == 0 ? 0 : 1;
  }
}

int main(int argc, char** argv) {
  if (argc == 5 && strcmp(argv[1], "host") == 0)
    return host_mode(strtoll(argv[2], NULL, 10), strtoll(argv[3], NULL, 10), strtoll(argv[4], NULL, 10));
  if (argc == 4 && strcmp(argv[1], "gpu") == 0) return gpu_mode(argv[2], argv[3]);
  if (argc == 5 && strcmp(argv[1], "vp") == 0) return vp_mode(argv[2], argv[3], atoi(argv[4]), 0);
  if (argc == 5 && strcmp(argv[1], "vps") == 0) return vp_mode(argv[2], argv[3], atoi(argv[4]), 1);
  fprintf(stderr, "usage: flce_client host N H V | flce_client gpu IN OUT | flce_client vp|vps IN OUT S\n");
  return 64;
}
