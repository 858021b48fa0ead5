/* A C99 program that runs one Muon step through libmuonbank.so with device
 * memory from the CUDA runtime, and checks what C alone can check exactly:
 *   - a slot whose gradient is zero only decays: its new fp32 weight is the
 *     fp32 product of the old one and (1 - lr*wd), split back into bf16 and
 *     mantissa halves, bit for bit (the update of v = 0 adds nothing);
 *   - the step is deterministic: two runs from the same state give the same bytes.
 * Numerical parity of the live slots is the oracle tests' job.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "muonbank.h"

#define B 3
#define R 256
#define C 384
#define E ((size_t)B * R * C)

static int failures = 0;

#define CHECK(cond)                                                             \
  do {                                                                          \
    if (!(cond)) {                                                              \
      fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
      ++failures;                                                               \
    }                                                                           \
  } while (0)

static uint32_t lcg(uint32_t* s) { return *s = *s * 1664525u + 1013904223u; }

static uint16_t bf16_of(float f) {   /* round to nearest even; inputs are finite */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

struct state {
  uint16_t w[E], mant[E], g[E];
  float mom[E];
};

/* failures of this program itself, apart from the library's statuses */
#define NO_WORKSPACE_SIZE 1000
#define NO_DEVICE_MEMORY 1001

static int run(const struct state* in, struct state* out, float lr, float wd, float mu) {
  void *w, *g, *mant, *mom, *ws;
  size_t ws_bytes = 0;
  const mb_shape shape = {B, R, C};
  int st;
  if (mb_workspace_bytes(shape, 0, &ws_bytes) != MB_OK) return NO_WORKSPACE_SIZE;
  if (cudaMalloc(&w, E * 2) || cudaMalloc(&g, E * 2) || cudaMalloc(&mant, E * 2) || cudaMalloc(&mom, E * 4) ||
      cudaMalloc(&ws, ws_bytes)) {
    fprintf(stderr, "cudaMalloc: %s\n", cudaGetErrorString(cudaGetLastError()));
    return NO_DEVICE_MEMORY;
  }
  cudaMemcpy(w, in->w, E * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(g, in->g, E * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(mant, in->mant, E * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(mom, in->mom, E * 4, cudaMemcpyHostToDevice);
  st = muon_bank_step(w, g, (float*)mom, (uint16_t*)mant, shape, lr, wd, mu, 5, ws, ws_bytes, NULL);
  if (st == MB_OK) st = mb_sync_status(NULL);
  cudaMemcpy(out->w, w, E * 2, cudaMemcpyDeviceToHost);
  cudaMemcpy(out->mant, mant, E * 2, cudaMemcpyDeviceToHost);
  cudaMemcpy(out->mom, mom, E * 4, cudaMemcpyDeviceToHost);
  cudaFree(w);
  cudaFree(g);
  cudaFree(mant);
  cudaFree(mom);
  cudaFree(ws);
  return st;
}

int main(void) {
  static struct state in, out1, out2;
  const float lr = 0.02f, wd = 0.01f, mu = 0.95f;
  const float decay = (float)fma(-(double)lr, (double)wd, 1.0);
  uint32_t s = 12345u;
  size_t i, dead0 = (size_t)R * C, dead1 = 2 * (size_t)R * C;   /* slot 1 has a zero gradient */
  int st;

  for (i = 0; i < E; ++i) {
    const float wv = ((float)(lcg(&s) >> 8) / 16777216.0f - 0.5f) * 0.1f;
    const float gv = ((float)(lcg(&s) >> 8) / 16777216.0f - 0.5f) * 2e-3f;
    in.w[i] = bf16_of(wv);
    in.mant[i] = (uint16_t)(lcg(&s) >> 16);
    in.g[i] = (i >= dead0 && i < dead1) ? 0 : bf16_of(gv);
    in.mom[i] = 0.f;
  }
  st = run(&in, &out1, lr, wd, mu);
  if (st != MB_OK) {
    fprintf(stderr, "status %d: %s (%s)\n", st, st < 0 ? mb_status_string(st) : "see above", mb_last_cuda_error());
    return 1;
  }
  CHECK(run(&in, &out2, lr, wd, mu) == MB_OK);
  CHECK(memcmp(out1.w, out2.w, sizeof out1.w) == 0);
  CHECK(memcmp(out1.mant, out2.mant, sizeof out1.mant) == 0);
  CHECK(memcmp(out1.mom, out2.mom, sizeof out1.mom) == 0);

  for (i = dead0; i < dead1; ++i) {
    const uint32_t w32 = ((uint32_t)in.w[i] << 16) | in.mant[i];
    float wf, r;
    uint32_t r32;
    memcpy(&wf, &w32, 4);
    r = wf * decay;
    memcpy(&r32, &r, 4);
    if (out1.w[i] != (uint16_t)(r32 >> 16) || out1.mant[i] != (uint16_t)(r32 & 0xFFFFu) || out1.mom[i] != 0.f) {
      fprintf(stderr, "decay-only slot differs at %zu\n", i - dead0);
      ++failures;
      break;
    }
  }
  /* the live slots moved */
  CHECK(memcmp(out1.w, in.w, (size_t)R * C * 2) != 0);

  if (failures) fprintf(stderr, "%d check(s) failed\n", failures);
  else printf("step consumer ok\n");
  return failures ? 1 : 0;
}
