/* A plain C99 consumer of the library's C ABI (include/flint_moe.h): no Python, no C++.
 *
 * Without arguments it runs the host-side checks that need no GPU: workspace sizing, the
 * refusal of other shapes, status strings and argument errors; it prints "host checks ok".
 *
 * Built with -DWITH_CUDA and given a directory and token counts, it runs the layer as a C
 * program would: it reads the bf16 weights and inputs from raw files in that directory
 * (w_router.bin, w_gate.bin, w_up.bin, w_down.bin, ws_gate.bin, ws_up.bin, ws_down.bin and
 * x_<T>.bin, written by the test), copies them to the device with the CUDA runtime, and for
 * each T creates a handle, calls flint_moe_forward (device buffers) and flint_moe_forward_host
 * (host buffers), polls the device status and writes y_<T>.bin, yh_<T>.bin (bf16), idx_<T>.bin
 * (int32 [T][6]) and gw_<T>.bin (fp32 [T][6]) for the test to check against the oracle.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "flint_moe.h"

#define H 2048
#define E 256
#define K 6
#define I 512
#define IS 1024

static int failures = 0;

#define CHECK(cond, what)                          \
  do {                                             \
    if (!(cond)) {                                 \
      fprintf(stderr, "FAILED: %s\n", (what));     \
      ++failures;                                  \
    }                                              \
  } while (0)

static flint_moe_config config(int max_tokens) {
  flint_moe_config c;
  c.hidden = H;
  c.n_experts = E;
  c.top_k = K;
  c.expert_inter = I;
  c.shared_inter = IS;
  c.max_tokens = max_tokens;
  c.flags = 0u;
  c.rms_eps = 1e-6f;
  return c;
}

static void host_checks(void) {
  flint_moe_config c = config(16);
  size_t bytes = 0, bytes256 = 0;
  flint_moe_t h = NULL;
  flint_moe_weights w;
  int code;
  CHECK(flint_moe_workspace_bytes(&c, &bytes) == FLINT_MOE_OK && bytes > 0 && bytes % 256 == 0,
        "workspace bytes for 16 tokens");
  c.max_tokens = 256;
  CHECK(flint_moe_workspace_bytes(&c, &bytes256) == FLINT_MOE_OK && bytes256 > bytes, "workspace grows with T");
  c.hidden = 4096;
  CHECK(flint_moe_workspace_bytes(&c, &bytes) == FLINT_MOE_ERR_UNSUPPORTED, "another hidden size is refused");
  c = config(16);
  c.top_k = 8;
  CHECK(flint_moe_workspace_bytes(&c, &bytes) == FLINT_MOE_ERR_UNSUPPORTED, "another top-k is refused");
  c = config(0);
  CHECK(flint_moe_workspace_bytes(&c, &bytes) == FLINT_MOE_ERR_INVALID_ARG, "max_tokens 0 is invalid");
  c = config(16);
  CHECK(flint_moe_workspace_bytes(&c, NULL) == FLINT_MOE_ERR_INVALID_ARG, "NULL output is invalid");
  for (code = 0; code <= 6; ++code) {
    const char* s = flint_moe_status_string((flint_moe_status)code);
    CHECK(s != NULL && strcmp(s, "unknown status") != 0, "status string");
  }
  CHECK(strcmp(flint_moe_status_string((flint_moe_status)99), "unknown status") == 0, "unknown status string");
  memset(&w, 0, sizeof w);
  CHECK(flint_moe_create(&c, &w, NULL, 0, &h) != FLINT_MOE_OK && h == NULL, "create without weights fails");
  CHECK(flint_moe_create(&c, NULL, NULL, 0, &h) != FLINT_MOE_OK, "create with NULL weights fails");
  CHECK(flint_moe_destroy(NULL) == FLINT_MOE_ERR_INVALID_ARG, "destroy(NULL)");
  CHECK(flint_moe_forward(NULL, NULL, 1, NULL, NULL, NULL, NULL) == FLINT_MOE_ERR_INVALID_ARG, "forward(NULL)");
}

#ifdef WITH_CUDA
#include <cuda_runtime_api.h>

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  FILE* f;
  void* p = malloc(bytes);
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "rb");
  if (!p || !f || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %s\n", path);
    exit(2);
  }
  fclose(f);
  return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  FILE* f;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "wb");
  if (!f || fwrite(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(2);
  }
  fclose(f);
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "device copy failed\n");
    exit(2);
  }
  return d;
}

/* The seven weight matrices, read once and copied to the device. */
static void load_weights(const char* dir, void* dw[7]) {
  static const char* names[7] = {"w_router.bin", "w_gate.bin", "w_up.bin", "w_down.bin",
                                 "ws_gate.bin", "ws_up.bin", "ws_down.bin"};
  const size_t sizes[7] = {(size_t)H * E * 2, (size_t)E * H * I * 2, (size_t)E * H * I * 2, (size_t)E * I * H * 2,
                           (size_t)H * IS * 2, (size_t)H * IS * 2, (size_t)IS * H * 2};
  int i;
  for (i = 0; i < 7; ++i) {
    void* p = read_file(dir, names[i], sizes[i]);
    dw[i] = to_device(p, sizes[i]);
    free(p);
  }
}

static void run(const char* dir, void* const dw[7], int T) {
  char name[64];
  flint_moe_config c = config(T);
  flint_moe_weights w;
  flint_moe_t h = NULL;
  size_t ws_bytes = 0;
  void *ws = NULL, *dx = NULL, *dy = NULL, *didx = NULL, *dgw = NULL, *x, *y, *yh;
  int32_t* idx;
  float* gw;
  const size_t xb = (size_t)T * H * 2;
  w.w_router = dw[0];
  w.router_bias = NULL;
  w.w_gate = dw[1];
  w.w_up = dw[2];
  w.w_down = dw[3];
  w.ws_gate = dw[4];
  w.ws_up = dw[5];
  w.ws_down = dw[6];
  snprintf(name, sizeof name, "x_%d.bin", T);
  x = read_file(dir, name, xb);
  y = malloc(xb);
  yh = malloc(xb);
  idx = (int32_t*)malloc((size_t)T * K * 4);
  gw = (float*)malloc((size_t)T * K * 4);
  CHECK(flint_moe_workspace_bytes(&c, &ws_bytes) == FLINT_MOE_OK, "workspace bytes");
  CHECK(cudaMalloc(&ws, ws_bytes) == cudaSuccess, "workspace allocation");
  CHECK(flint_moe_create(&c, &w, ws, ws_bytes, &h) == FLINT_MOE_OK, "create");
  dx = to_device(x, xb);
  CHECK(cudaMalloc(&dy, xb) == cudaSuccess && cudaMalloc(&didx, (size_t)T * K * 4) == cudaSuccess &&
            cudaMalloc(&dgw, (size_t)T * K * 4) == cudaSuccess,
        "output allocation");
  CHECK(flint_moe_forward(h, dx, T, dy, (int32_t*)didx, (float*)dgw, NULL) == FLINT_MOE_OK, "forward");
  CHECK(flint_moe_forward_host(h, x, T, yh, NULL) == FLINT_MOE_OK, "forward_host");
  CHECK(flint_moe_poll_device_status(h, NULL) == FLINT_MOE_OK, "device status");
  CHECK(cudaMemcpy(y, dy, xb, cudaMemcpyDeviceToHost) == cudaSuccess, "read y");
  CHECK(cudaMemcpy(idx, didx, (size_t)T * K * 4, cudaMemcpyDeviceToHost) == cudaSuccess, "read idx");
  CHECK(cudaMemcpy(gw, dgw, (size_t)T * K * 4, cudaMemcpyDeviceToHost) == cudaSuccess, "read gates");
  snprintf(name, sizeof name, "y_%d.bin", T);
  write_file(dir, name, y, xb);
  snprintf(name, sizeof name, "yh_%d.bin", T);
  write_file(dir, name, yh, xb);
  snprintf(name, sizeof name, "idx_%d.bin", T);
  write_file(dir, name, idx, (size_t)T * K * 4);
  snprintf(name, sizeof name, "gw_%d.bin", T);
  write_file(dir, name, gw, (size_t)T * K * 4);
  CHECK(flint_moe_destroy(h) == FLINT_MOE_OK, "destroy");
  cudaFree(ws);
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(didx);
  cudaFree(dgw);
  free(x);
  free(y);
  free(yh);
  free(idx);
  free(gw);
}
#endif

int main(int argc, char** argv) {
  host_checks();
  if (argc > 2) {
#ifdef WITH_CUDA
    void* dw[7];
    int a;
    load_weights(argv[1], dw);
    for (a = 2; a < argc; ++a) run(argv[1], dw, atoi(argv[a]));
    for (a = 0; a < 7; ++a) cudaFree(dw[a]);
#else
    (void)argv;
    fprintf(stderr, "built without WITH_CUDA\n");
    return 2;
#endif
  }
  if (failures) return 1;
  printf(argc > 2 ? "host checks and forwards ok\n" : "host checks ok\n");
  return 0;
}
