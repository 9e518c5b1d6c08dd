/* A plain C99 caller of the library's host-side entry points (no GPU needed): packing of the
 * three layouts, workspace sizes and an argument error.  Prints one "key value..." line per
 * result; tests/test_abi_c.py compiles it with gcc, runs it and compares the lines with the
 * Python binding's results. */
#include <stdio.h>
#include <stdlib.h>

#include "pg_grouped_attn.h"
#include "pg_layer.h"

static void print_layout(const char* name, const pg_layout* L, const int32_t* pos) {
  printf("%s_tokens %lld\n", name, (long long)L->total_tokens);
  printf("%s_pairs %lld\n", name, (long long)L->pairs);
  printf("%s_depth %lld\n", name, (long long)L->max_depth);
  printf("%s_pad_rows %lld\n", name, (long long)L->n_pad_rows);
  printf("%s_pos", name);
  for (int64_t t = 0; t < L->total_tokens; ++t) printf(" %d", (int)pos[t]);
  printf("\n");
}

static int packed(void) {
  const int32_t prefix_lens[2] = {5, 0};
  const int32_t group_sizes[2] = {3, 2};
  const int32_t suffix_lens[5] = {2, 0, 3, 4, 1};
  int64_t T = 0, bytes = 0;
  if (pg_pack_size(2, prefix_lens, group_sizes, suffix_lens, &T, &bytes) != PG_OK) return 1;
  int32_t* pos = malloc(sizeof(int32_t) * (size_t)T);
  void* tab = malloc((size_t)bytes);
  pg_layout L;
  if (!pos || !tab) return 1;
  if (pg_pack_host(2, prefix_lens, group_sizes, suffix_lens, pos, tab, bytes, &L) != PG_OK)
    return 1;
  print_layout("packed", &L, pos);
  /* workspace of the backward, plain and with q / k arriving rotated */
  pg_opts plain = {0.0f, 1e4f, 0u, 0u};
  pg_opts pre = {0.0f, 1e4f, PG_FLAG_PRE_ROTATED, 0u};
  size_t w0 = 0, w1 = 0;
  if (pg_workspace_size(&L, PG_BF16, 4, 2, 128, &plain, 1, &w0) != PG_OK) return 1;
  if (pg_workspace_size(&L, PG_BF16, 4, 2, 128, &pre, 1, &w1) != PG_OK) return 1;
  printf("ws_plain %zu\nws_pre %zu\n", w0, w1);
  /* an argument error is reported on the host, before any launch */
  pg_status st = pg_grouped_attn_fwd(&L, PG_BF16, 3, 2, 128, pos, pos, pos, pos, NULL, &plain,
                                     NULL, 0, NULL);
  printf("bad_heads %d %s\n", (int)st, pg_status_string(st));
  free(pos);
  free(tab);
  return 0;
}

static int tree(void) {
  const int32_t parent[5] = {-1, 0, 1, 1, 0};
  const int32_t seg_lens[5] = {2, 1, 2, 1, 1};
  int64_t T = 0, bytes = 0;
  if (pg_pack_tree_size(5, parent, seg_lens, &T, &bytes) != PG_OK) return 1;
  int32_t* pos = malloc(sizeof(int32_t) * (size_t)T);
  void* tab = malloc((size_t)bytes);
  pg_layout L;
  if (!pos || !tab) return 1;
  if (pg_pack_tree_host(5, parent, seg_lens, pos, tab, bytes, &L) != PG_OK) return 1;
  print_layout("tree", &L, pos);
  free(pos);
  free(tab);
  return 0;
}

static int padded(void) {
  const int32_t response_lens[6] = {4, 0, 2, 1, 4, 3};
  int64_t T = 0, bytes = 0;
  if (pg_pack_padded_size(2, 5, 3, 4, response_lens, &T, &bytes) != PG_OK) return 1;
  int32_t* pos = malloc(sizeof(int32_t) * (size_t)T);
  void* tab = malloc((size_t)bytes);
  pg_layout L;
  if (!pos || !tab) return 1;
  if (pg_pack_padded_host(2, 5, 3, 4, response_lens, pos, tab, bytes, &L) != PG_OK) return 1;
  print_layout("padded", &L, pos);
  free(pos);
  free(tab);
  return 0;
}

int main(void) {
  if (packed() || tree() || padded()) {
    fprintf(stderr, "failed: %s\n", pg_last_error_message());
    return 1;
  }
  return 0;
}
