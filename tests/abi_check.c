/*
 * Built by the host ABI test as plain C99 against include/skv.h and linked
 * with libskv.so: the header must compile as C, the struct layout the C
 * compiler gives skv_cache is printed for comparison with the Python
 * binding, and the calls that answer without a GPU are checked.
 */
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include "skv.h"

#define FIELD(f) printf("%s %zu\n", #f, offsetof(skv_cache, f))

static int expect(const char* what, long long got, long long want) {
  if (got == want) return 0;
  printf("FAIL %s: %lld, want %lld\n", what, got, want);
  return 1;
}

int main(void) {
  int fails = 0;
  skv_cache c;
  printf("size %zu\n", sizeof(skv_cache));
  FIELD(n_cache);
  FIELD(n_view);
  FIELD(n_frame);
  FIELD(frame_len);
  FIELD(prefix_len);
  FIELD(tail_cap);
  FIELD(n_kv_head);
  FIELD(head_dim);
  FIELD(row_cap);
  FIELD(rope_len);
  FIELD(k);
  FIELD(vt);
  FIELD(head);
  FIELD(sync);
  FIELD(rope);
  FIELD(status);
  FIELD(wait_ns);
  FIELD(rope_mode);
  FIELD(reserved);

  fails += expect("version", skv_version(), SKV_VERSION);
  fails += expect("row_cap", skv_row_cap(256, 4, 4, 180, 128), 3328);
  fails += expect("row_cap of a bad geometry", skv_row_cap(0, 0, 1, 1, 0), -1);
  fails += expect("status string", skv_status_string(SKV_ERR_INVALID) != NULL, 1);
  fails += expect("null descriptor", kv_stream_insert(NULL, NULL, NULL, NULL), SKV_ERR_INVALID);

  memset(&c, 0, sizeof c);
  c.n_cache = 2;
  c.n_view = 4;
  c.n_frame = 4;
  c.frame_len = 180;
  c.prefix_len = 256;
  c.tail_cap = 128;
  c.n_kv_head = 8;
  c.head_dim = 96; /* not a supported head size */
  c.row_cap = 3328;
  c.rope_len = 3264;
  fails += expect("head_dim 96", kv_stream_insert(&c, NULL, NULL, NULL), SKV_ERR_INVALID);
  c.head_dim = 128;
  c.n_cache = 0; /* an empty set of caches touches nothing, device or memory */
  fails += expect("empty cache set", kv_stream_insert(&c, NULL, NULL, NULL), SKV_OK);
  fails += expect("empty cache set, prefill",
                  stream_attn_prefill(&c, 32, NULL, NULL, NULL, 1.0f, NULL), SKV_OK);
  printf("fails %d\n", fails);
  return fails != 0;
}
