/* A plain C consumer of the C ABI (no C++, no torch): size queries, status strings and
 * argument checks, none of which launch a kernel. Built and run by test_c_consumer.py. */
#include <stdio.h>
#include <string.h>

#include "psk.h"

int main(void) {
  psk_layout L;
  memset(&L, 0, sizeof L);
  L.batch = 64;
  L.num_q_heads = 32;
  L.num_kv_heads = 8;
  L.head_dim = 128;
  L.v_head_dim = 128;
  L.page_size = 16;
  L.num_blocks = 150000;
  L.max_pages = 4096;
  L.dtype = PSK_BF16;
  L.latent = 0;
  size_t sel = psk_score_select_workspace_size(&L, 205);
  size_t dec = psk_sparse_decode_workspace_size(&L, 205);
  size_t den = psk_dense_decode_workspace_size(&L);
  size_t app = psk_append_workspace_size(&L);
  if (sel == 0 || dec == 0 || den == 0 || app == 0) return 1;
  /* a missing argument is refused before any launch */
  int rc = psk_page_score_select(&L, NULL, NULL, NULL, NULL, NULL, 205, 1.0f, NULL, NULL, NULL, 0, NULL);
  if (rc != PSK_ERR_INVALID_ARG) return 2;
  psk_select_params prm;
  memset(&prm, 0, sizeof prm);
  prm.mode = PSK_BUDGET_FRACTION;
  prm.budget_fraction = 0.05;
  prm.sink_pages = 1;
  prm.window_pages = 1;
  rc = psk_page_score(&L, NULL, NULL, NULL, NULL, &prm, 205, 1.0f, NULL, NULL, 0, NULL);
  if (rc != PSK_ERR_INVALID_ARG) return 3;
  L.head_dim = 96; /* not built */
  if (psk_score_select_workspace_size(&L, 205) != 0) return 4;
  printf("version %d; %s; sizes %zu %zu %zu %zu\n", psk_version(), psk_status_string(PSK_ERR_UNSUPPORTED), sel,
         dec, den, app);
  return 0;
}
