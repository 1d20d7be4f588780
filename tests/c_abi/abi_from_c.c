/*
 * The library's boundary used from plain C (no C++, no torch): compiled with
 * gcc -std=c11 against include/moe.h and linked to libmoe_gb300.so.  Every
 * call here is answered on the host: constants, defaults, sizes and argument
 * checks that return before any device work.  Prints "ok" and exits 0 when
 * every check holds.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int failures = 0;

#define CHECK(cond)                                                    \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
      ++failures;                                                      \
    }                                                                  \
  } while (0)

int main(void) {
  CHECK(moe_abi_version() == 102);

  moe_config_t cfg;
  memset(&cfg, 0x5A, sizeof cfg);
  moe_config_default(&cfg);
  CHECK(cfg.score == MOE_SCORE_SOFTMAX);
  CHECK(cfg.renormalize == 1);
  CHECK(cfg.route_scale == 1.0f);
  CHECK(cfg.n_group == 1 && cfg.topk_group == 1 && cfg.group_topn == 0);
  CHECK(cfg.logit_bias == NULL && cfg.F_shared == 0 && cfg.ws_gate == NULL && cfg.w_shared_gate == NULL);
  CHECK(cfg.activation == MOE_ACT_SILU);

  CHECK(strcmp(moe_status_string(MOE_OK), "MOE_OK") == 0);
  CHECK(strstr(moe_status_string(MOE_ERR_WORKSPACE), "WORKSPACE") != NULL);

  /* Workspace of the Mixtral-shaped layer at T=4096: at least the grouped
   * token copies, the SwiGLU activations and the fp16 expert outputs. */
  const size_t Tk = (size_t)4096 * 2;
  const size_t ws = moe_workspace_bytes(&cfg, 4096, 4096, 14336, 8, 2);
  CHECK(ws >= Tk * 4096 * 2 + Tk * 14336 * 2 + Tk * 4096 * 2);
  CHECK(moe_workspace_bytes(NULL, 4096, 4096, 14336, 8, 2) == ws); /* NULL = the default config */
  CHECK(moe_workspace_bytes(&cfg, 4096, 4000, 14336, 8, 2) == 0);   /* H not a multiple of 128 */
  CHECK(moe_route_scratch_bytes(&cfg, 4096, 4096, 8) == 0); /* partial logits reduced on chip */

  /* Arguments are checked before any launch (the pointers are never used). */
  void* const dev = (void*)(uintptr_t)0x1000;
  void* const misaligned = (void*)(uintptr_t)0x1008;
  void* const y = (void*)(uintptr_t)0x6000;
  CHECK(moe_forward(dev, dev, dev, dev, dev, 4, 512, 1024, 8, 9, dev, NULL) == MOE_ERR_UNSUPPORTED); /* k > E */
  CHECK(moe_forward(dev, dev, dev, dev, dev, 4, 512, 1024, 300, 2, dev, NULL) == MOE_ERR_UNSUPPORTED); /* E > 256 */
  CHECK(moe_forward(misaligned, dev, dev, dev, dev, 4, 512, 1024, 8, 2, dev, NULL) == MOE_ERR_INVALID_VALUE);
  CHECK(moe_forward(dev, dev, dev, dev, dev, 0, 512, 1024, 8, 2, dev, NULL) == MOE_OK); /* T = 0: no-op */
  CHECK(moe_expert_ffn_ex(dev, NULL, 16, 512, 1024, 8, dev, dev, dev, MOE_ACT_GELU, dev, y, NULL) ==
        MOE_ERR_INVALID_VALUE); /* offsets NULL needs E = 1 */
  CHECK(moe_expert_ffn_ex(dev, (const int32_t*)dev, 16, 512, 1024, 8, dev, dev, dev, 7, dev, y, NULL) ==
        MOE_ERR_INVALID_VALUE); /* unknown activation */
  cfg.n_group = 8;
  cfg.topk_group = 9; /* keeps more groups than exist */
  cfg.group_topn = 2;
  CHECK(moe_forward_ex(&cfg, dev, dev, dev, dev, dev, 4, 512, 1024, 256, 8, dev, dev, (size_t)1 << 30, NULL) ==
        MOE_ERR_INVALID_VALUE);

  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("ok\n");
  return 0;
}
