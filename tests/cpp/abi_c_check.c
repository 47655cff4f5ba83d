/* The boundary is a C ABI: this C99 translation unit includes the header, takes the address
 * of every entry point and calls the ones that need no GPU. */
#include <stdio.h>
#include <string.h>

#include "../../include/longstraw.h"

typedef void (*any_fn)(void);

int main(void) {
  any_fn fns[] = {
      (any_fn)ls_prefix_prepare, (any_fn)ls_prefix_destroy, (any_fn)ls_replay_fwd,
      (any_fn)ls_replay_bwd_workspace_bytes, (any_fn)ls_replay_bwd, (any_fn)ls_replay_fwd_packed,
      (any_fn)ls_replay_bwd_packed_workspace_bytes, (any_fn)ls_replay_bwd_packed,
      (any_fn)ls_block_replay_fwd, (any_fn)ls_block_replay_bwd, (any_fn)ls_grpo_loss_workspace_bytes,
      (any_fn)ls_grpo_loss, (any_fn)ls_token_logp, (any_fn)ls_grpo_loss_noalloc,
      (any_fn)ls_grpo_loss_noalloc_max_rows, (any_fn)ls_replay_fwd_prompt_only,
      (any_fn)ls_replay_bwd_prompt_only, (any_fn)ls_attn_merge, (any_fn)ls_sum_bf16,
      (any_fn)ls_prefix_grad_finalize, (any_fn)ls_prefix_grad_finalize_rows,
      (any_fn)ls_get_device_status, (any_fn)ls_timing_enable, (any_fn)ls_timing_read,
      (any_fn)ls_debug_wait_timeout, (any_fn)ls_status_string, (any_fn)ls_last_error,
      (any_fn)ls_version};
  size_t i;
  for (i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i)
    if (fns[i] == NULL) return 1;
  if (ls_version() == NULL || strlen(ls_version()) == 0) return 2;
  if (strcmp(ls_status_string(LS_OK), ls_status_string(LS_ERR_CUDA)) == 0) return 3;
  if (ls_prefix_destroy(NULL) != LS_OK) return 4;
  if (ls_replay_fwd(NULL, 4, NULL, NULL, NULL, NULL, NULL, NULL) != LS_ERR_NOT_PREPARED) return 5;
  if (ls_grpo_loss_noalloc_max_rows() < 1) return 6;
  printf("OK %s\n", ls_version());
  return 0;
}
