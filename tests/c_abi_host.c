/*
 * Host-only use of the library's C ABI from plain C (C99): everything here
 * runs without a GPU -- status strings, workspace sizes, argument validation
 * that fails before any launch, and the radix tree.  Prints "ok" and exits 0
 * when every check holds; otherwise prints the failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "sgl_attn.h"

static int failures = 0;
#define CHECK(cond)                                             \
  do {                                                          \
    if (!(cond)) {                                              \
      printf("FAILED: %s (line %d)\n", #cond, __LINE__);        \
      ++failures;                                               \
    }                                                           \
  } while (0)

int main(void) {
  /* fake device pointers: aligned, never dereferenced (every call below
   * fails validation or sizes something on the host) */
  void* dev = (void*)(uintptr_t)0x100000;
  sgl_attn_dims d = {16, 8, 128, 1024, 0.0f};

  CHECK(sgl_version() != NULL && strlen(sgl_version()) > 0);
  CHECK(strlen(sgl_status_string(SGL_ERR_WORKSPACE)) > 0);

  /* workspace sizes */
  CHECK(sgl_extend_workspace_bytes(4, 100, &d) >= 16);
  CHECK(sgl_decode_workspace_bytes(4, 4096, &d) > sgl_decode_workspace_bytes(4, 64, &d));
  CHECK(sgl_cascade_decode_workspace_bytes(4, 4096, 2, &d) > sgl_decode_workspace_bytes(4, 4096, &d));

  /* validation before any launch */
  CHECK(sgl_store_kv(dev, dev, dev, -1, dev, dev, &d, NULL) == SGL_ERR_INVALID_ARG);
  CHECK(sgl_store_kv(NULL, NULL, NULL, 0, NULL, NULL, &d, NULL) == SGL_OK);
  CHECK(sgl_decode_attention(dev, dev, dev, dev, 4, 64, dev, dev, 2, 64, dev, NULL, 0, &d, NULL) ==
        SGL_ERR_WORKSPACE);
  {
    sgl_attn_dims bad = d;
    bad.head_dim = 96;
    CHECK(sgl_store_kv(dev, dev, dev, 4, dev, dev, &bad, NULL) == SGL_ERR_UNSUPPORTED);
  }
  CHECK(sgl_store_kv_fp8(dev, dev, dev, 4, dev, dev, 0.0f, 1.0f, &d, NULL) == SGL_ERR_INVALID_ARG);

  /* radix tree: two prompts sharing a 3-token prefix */
  {
    sgl_radix_tree* t = sgl_radix_create();
    const int32_t a[5] = {7, 8, 9, 1, 2};
    const int32_t b[4] = {7, 8, 9, 5};
    const int32_t sa[5] = {100, 101, 102, 103, 104};
    const int32_t sb[4] = {100, 101, 102, 200};
    int32_t slots[8];
    int64_t na = 0, nb = 0, nodes[2];
    int32_t start[4], len[4], depth[4], off[5], mem[8], n_members = 0, ng;
    int32_t freed[16];
    CHECK(t != NULL);
    CHECK(sgl_radix_insert(t, a, sa, 5) == 0);
    CHECK(sgl_radix_insert(t, b, sb, 4) == 3);           /* the shared prefix was cached */
    CHECK(sgl_radix_match_prefix(t, b, 4, slots, 8, &nb) == 4);
    CHECK(slots[0] == 100 && slots[2] == 102 && slots[3] == 200);
    CHECK(sgl_radix_match_prefix(t, a, 5, slots, 8, &na) == 5);
    nodes[0] = na;
    nodes[1] = nb;
    ng = sgl_radix_groups(t, nodes, 2, start, len, depth, off, mem, 4, 8, &n_members);
    CHECK(ng == 1 && start[0] == 0 && len[0] == 3 && depth[0] == 0 && n_members == 2);
    CHECK(off[0] == 0 && off[1] == 2 && mem[0] == 0 && mem[1] == 1);
    CHECK(sgl_radix_inc_lock_ref(t, na) == SGL_OK);
    CHECK(sgl_radix_protected_tokens(t) == 5 && sgl_radix_evictable_tokens(t) == 1);
    CHECK(sgl_radix_evict(t, 16, freed, 16) == 1 && freed[0] == 200); /* only b's own leaf */
    CHECK(sgl_radix_dec_lock_ref(t, na) == SGL_OK);
    CHECK(sgl_radix_dec_lock_ref(t, na) == SGL_ERR_INVALID_ARG);     /* unbalanced */
    CHECK(sgl_radix_evict(t, 16, freed, 16) == 5);
    CHECK(sgl_radix_evictable_tokens(t) == 0);
    sgl_radix_destroy(t);
  }

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
