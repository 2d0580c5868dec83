/* Plain C99 user of the C ABI: configuration checks, workspace sizes, status
 * strings and argument errors, none of which needs a GPU.  Exit code 0 on
 * success, the number of the failed check otherwise. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

static moe_cfg_t v3_prefill(void) {
  moe_cfg_t c;
  memset(&c, 0, sizeof(c));
  c.T = 8192;
  c.d = 7168;
  c.E = 256;
  c.K = 8;
  c.S = 1;
  c.I = 2048;
  c.act_dtype = MOE_BF16;
  c.wgt_dtype = MOE_BF16;
  c.score_func = MOE_SCORE_SIGMOID;
  c.normalize = 1;
  c.add_residual = 1;
  c.gamma = 1e-3f;
  return c;
}

int main(void) {
  moe_cfg_t c = v3_prefill();
  if (moe_check_cfg(&c) != MOE_OK) return 1;
  size_t fwd = moe_workspace_size(&c, MOE_WS_FORWARD);
  /* xp [T*K, d], act [R, I], y [R, d] in bf16, R = T*K + S*T */
  const size_t R = 8192u * 8u + 8192u;
  if (fwd < 2u * (8192u * 8u * 7168u + R * 2048u + R * 7168u)) return 2;
  /* behind the RMSNorm: + normalised tokens, weighted centroids, inv_rms */
  if (moe_workspace_size(&c, MOE_WS_FORWARD_PRENORM) !=
      fwd + 8192u * 7168u * 2u + 256u * 7168u * 2u + 8192u * 4u)
    return 3;
  c.K = 0;
  if (moe_check_cfg(&c) != MOE_ERR_INVALID_ARG) return 4;
  if (moe_workspace_size(&c, MOE_WS_FORWARD) != 0) return 5;
  c = v3_prefill();
  c.wgt_dtype = MOE_E4M3;
  if (moe_check_cfg(&c) != MOE_OK) return 6;
  if (moe_workspace_size(&c, MOE_WS_FORWARD_W8A16) == 0) return 7;
  /* null pointers are argument errors, returned before any launch */
  c = v3_prefill();
  if (moe_route(&c, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) != MOE_ERR_INVALID_ARG) return 8;
  if (moe_selftest_wait_timeout(0, NULL) != MOE_ERR_INVALID_ARG) return 9;
  if (strlen(moe_status_string(MOE_ERR_DEVICE_TIMEOUT)) == 0) return 10;
  if (strstr(moe_version(), "sm_103a") == NULL) return 11;
  /* training: the state and gradient structs are plain C; missing ones and
   * non-bf16 layers are refused before any launch */
  {
    moe_train_state_t st;
    moe_grads_t gr;
    memset(&st, 0, sizeof(st));
    memset(&gr, 0, sizeof(gr));
    if (moe_workspace_size(&c, MOE_WS_BACKWARD) == 0) return 12;
    if (moe_workspace_size(&c, MOE_WS_FORWARD_TRAIN) == 0) return 13;
    if (moe_backward(&c, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, &gr, NULL, 0, NULL) !=
        MOE_ERR_INVALID_ARG)
      return 14;
    if (moe_forward_train(&c, NULL, NULL, NULL, NULL, NULL, NULL, NULL, &st, NULL, NULL, 0,
                          NULL) != MOE_ERR_INVALID_ARG)
      return 15;
    c.wgt_dtype = MOE_E4M3;
    if (moe_backward(&c, NULL, NULL, NULL, NULL, NULL, NULL, NULL, &st, &gr, NULL, 0, NULL) !=
        MOE_ERR_UNSUPPORTED)
      return 16;
    c = v3_prefill();
  }
  printf("abi ok: forward workspace %zu bytes\n", fwd);
  return 0;
}
