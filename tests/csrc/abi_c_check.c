/* abi_c_check.c -- compiled as C99 against include/gdn.h and linked with libgdn.so: the header
 * is plain C and every host-side entry point resolves with C linkage.  Runs without a GPU: it
 * calls only functions that answer from host checks. */
#include <stdio.h>
#include <string.h>

#include "gdn.h"

int main(void) {
  gdn_dims d;
  memset(&d, 0, sizeof(d));
  d.num_k_heads = 16;
  d.num_v_heads = 48;
  d.head_k_dim = 128;
  d.head_v_dim = 128;
  d.conv_kernel = 4;
  d.l2_eps = 1e-6f;
  d.norm_eps = 1e-6f;
  const size_t slot = gdn_state_slot_bytes(&d, GDN_BF16);
  const size_t want = (size_t)48 * 128 * 128 * 4 + (size_t)3 * 10240 * 2;
  if (slot != want) {
    printf("slot bytes %zu != %zu\n", slot, want);
    return 1;
  }
  if (gdn_prefill_workspace_bytes(&d, 1, 4096) == 0) return 2;
  /* host checks fail before anything touches the GPU */
  gdn_weights w;
  memset(&w, 0, sizeof(w));
  w.act = GDN_BF16;
  gdn_pool p;
  memset(&p, 0, sizeof(p));
  if (gdn_decode_step(&d, &w, &p, 0, 1, 0, 0, 0, 0, 0, 0) != GDN_ERR_INVALID_ARG) return 3;
  if (gdn_decode_multi(&d, &w, &p, 0, 1, 0, 0, 0, 0, 0, 0, 0) != GDN_ERR_INVALID_ARG) return 4;
  gdn_decode_graphs* g = (gdn_decode_graphs*)&p;
  if (gdn_decode_graphs_create(&d, &w, &p, 0, 0, &g) != GDN_ERR_INVALID_ARG || g != 0) return 5;
  if (gdn_decode_graphs_launch(0, 1, 0) != GDN_ERR_INVALID_ARG) return 6;
  gdn_decode_graphs_destroy(0);
  if (!gdn_status_string(GDN_ERR_TOO_LARGE)) return 7;
  gdn_proj_route r;
  memset(&r, 0, sizeof(r));
  if (gdn_linear_bf16(0, 0, 1, 64, 64, &r, 0, 0, 0) != GDN_ERR_INVALID_ARG) return 8;
  if (gdn_in_proj(&d, &p, &p, 1, 100, &p, &p, &p, &p, 0, 0) != GDN_ERR_UNSUPPORTED_SHAPE) return 9;
  if (gdn_out_proj(&d, 0, 0, 0, 64, 0, 0, 0) != GDN_ERR_INVALID_ARG) return 10;
  printf("ok %s\n", gdn_status_string(GDN_OK));
  return 0;
}
