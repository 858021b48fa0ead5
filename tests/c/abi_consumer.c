/* A C99 caller of libmuonbank.so that sees nothing but include/muonbank.h.
 *
 * It calls the entry points that need no device (workspace sizes, argument
 * checks, status strings): every argument error must come back as its status
 * before the library touches a device or dereferences a pointer, so the
 * pointers here are aligned addresses that are never read.  Exits non-zero
 * after printing each mismatch.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "muonbank.h"

static int failures = 0;

#define CHECK(cond)                                                    \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
      ++failures;                                                      \
    }                                                                  \
  } while (0)

int main(void) {
  const mb_shape attn = {40, 768, 768}, mlp = {24, 3072, 768}, empty = {0, 768, 768};
  void* const dev = (void*)(uintptr_t)0x10000;   /* 256-byte aligned, never dereferenced */
  void* const odd = (void*)(uintptr_t)0x10002;
  float* const devf = (float*)dev;
  uint16_t* const devu = (uint16_t*)dev;
  size_t ws = 0, ws_nm = 0, ws_mlp = 0, ws_two = 0;
  mb_bank_desc banks[MB_MAX_BANKS + 1];
  int i;

  CHECK((mb_version() >> 16) == 1);
  CHECK(strcmp(mb_status_string(MB_OK), "ok") == 0);
  CHECK(strcmp(mb_status_string(12345), "unknown status") == 0);
  CHECK(mb_last_cuda_error() != NULL);

  /* workspace sizes: four bf16 copies of the bank at least, 1 KiB granules, more with NorMuon */
  CHECK(mb_workspace_bytes(attn, 0, &ws) == MB_OK);
  CHECK(ws >= (size_t)4 * 40 * 768 * 768 * 2 && ws % 1024 == 0);
  CHECK(mb_workspace_bytes(attn, 1, &ws_nm) == MB_OK && ws_nm > ws);
  CHECK(mb_workspace_bytes(mlp, 0, &ws_mlp) == MB_OK);
  CHECK(mb_workspace_bytes(empty, 0, &ws) == MB_ERR_SHAPE);
  CHECK(mb_workspace_bytes(attn, 0, NULL) == MB_ERR_NULL);

  /* a multi-bank call lays the banks' workspaces one after another */
  for (i = 0; i <= MB_MAX_BANKS; ++i) {
    memset(&banks[i], 0, sizeof banks[i]);
    banks[i].bank = dev;
    banks[i].grad = dev;
    banks[i].momentum = devf;
    banks[i].mantissa = devu;
    banks[i].shape = (i & 1) ? mlp : attn;
  }
  CHECK(mb_workspace_bytes(attn, 0, &ws) == MB_OK);
  CHECK(mb_multi_workspace_bytes(banks, 2, 0, &ws_two) == MB_OK && ws_two == ws + ws_mlp);
  CHECK(mb_multi_workspace_bytes(banks, MB_MAX_BANKS + 1, 0, &ws_two) == MB_ERR_TOO_MANY);

  /* argument errors of a step, each before anything is enqueued */
  CHECK(muon_bank_step(NULL, dev, devf, devu, attn, 0.02f, 0.01f, 0.95f, 5, dev, ws, NULL) == MB_ERR_NULL);
  CHECK(muon_bank_step(odd, dev, devf, devu, attn, 0.02f, 0.01f, 0.95f, 5, dev, ws, NULL) == MB_ERR_ALIGN);
  CHECK(muon_bank_step(dev, dev, devf, devu, empty, 0.02f, 0.01f, 0.95f, 5, dev, ws, NULL) == MB_ERR_SHAPE);
  CHECK(muon_bank_step(dev, dev, devf, devu, attn, 0.02f, 0.01f, 0.95f, 17, dev, ws, NULL) == MB_ERR_NS_STEPS);
  CHECK(muon_bank_step(dev, dev, devf, devu, attn, NAN, 0.01f, 0.95f, 5, dev, ws, NULL) == MB_ERR_ARG);
  CHECK(muon_bank_step(dev, dev, devf, devu, attn, 0.02f, 0.01f, 1.5f, 5, dev, ws, NULL) == MB_ERR_ARG);
  CHECK(muon_bank_step(dev, dev, devf, devu, attn, 0.02f, 0.01f, 0.95f, 5, dev, 16, NULL) == MB_ERR_WORKSPACE);
  CHECK(muon_bank_step(dev, dev, devf, devu, attn, 0.02f, 0.01f, 0.95f, 5, NULL, ws, NULL) == MB_ERR_WORKSPACE);
  CHECK(normuon_bank_step(dev, dev, devf, devu, NULL, attn, 0.02f, 0.01f, 0.95f, 0.95f, 5, dev, ws_nm, NULL) ==
        MB_ERR_NULL);
  CHECK(muon_multi_step(banks, 0, 0.02f, 0.01f, 0.95f, 0, 0.95f, 5, dev, ws_two, NULL) == MB_ERR_ARG);
  CHECK(muon_multi_step(banks, MB_MAX_BANKS + 1, 0.02f, 0.01f, 0.95f, 0, 0.95f, 5, dev, ws_two, NULL) ==
        MB_ERR_TOO_MANY);
  CHECK(muon_multi_step_dev(banks, 2, NULL, 0, 5, dev, ws_two, NULL) == MB_ERR_NULL);
  CHECK(mb_newton_schulz(dev, dev, attn, -1, dev, ws, NULL) == MB_ERR_NS_STEPS);
  CHECK(mb_newton_schulz_noalloc(dev, dev, mlp, 5, NULL) == MB_ERR_SCRATCH_LIMIT);
  CHECK(mb_timing_end(0, NULL, NULL, NULL) == MB_ERR_ARG);   /* no timing session open */

  if (failures) fprintf(stderr, "%d check(s) failed\n", failures);
  else printf("abi consumer ok\n");
  return failures ? 1 : 0;
}
