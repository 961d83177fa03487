/* A plain C caller of libpagedkv.so: it includes only include/pagedkv.h and
 * uses no Python or torch.  It exercises the calls that need no device (the
 * block allocator, the split-size queries, status strings and the argument
 * checks that return before any device work) and exits 0 when every check
 * holds; otherwise it prints the first failing check and exits 1.
 *
 * The allocator checks follow "Only 20.4% of your KV cache held actual
 * tokens", sections "The page table, relocated into attention" (blocks fill
 * left to right; a new block only when the last is full) and "The part
 * everyone forgets: pages enable sharing, not just packing" (forks share
 * blocks by reference count; a write into a shared, partly filled block
 * copies it first). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pagedkv.h"

#define CHECK(cond)                                                        \
  do {                                                                     \
    if (!(cond)) {                                                         \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      return 1;                                                            \
    }                                                                      \
  } while (0)

int main(void) {
  CHECK(pkv_version() >= 1);
  CHECK(strcmp(pkv_status_string(PKV_OK), "ok") == 0);
  CHECK(strcmp(pkv_status_string(PKV_ERR_OUT_OF_BLOCKS), "out of blocks") == 0);

  /* 16 blocks of 4 slots; a 7-token prompt takes two blocks (the second holds
   * 3 tokens). */
  pkv_allocator* a = NULL;
  CHECK(pkv_alloc_create(16, 4, &a) == PKV_OK && a != NULL);
  CHECK(pkv_alloc_add_seq(a, 1, 7) == PKV_OK);
  int num_tokens = 0, num_blocks = 0;
  CHECK(pkv_alloc_seq_info(a, 1, &num_tokens, &num_blocks) == PKV_OK);
  CHECK(num_tokens == 7 && num_blocks == 2);

  /* A fork shares both blocks. */
  CHECK(pkv_alloc_fork(a, 1, 2) == PKV_OK);
  int64_t ids[2] = {1, 2};
  int32_t table[2][4];
  CHECK(pkv_alloc_block_table(a, ids, 2, &table[0][0], 4) == PKV_OK);
  CHECK(table[0][0] == table[1][0] && table[0][1] == table[1][1]);
  CHECK(table[0][2] == -1 && table[1][3] == -1);
  int refcount = 0;
  CHECK(pkv_alloc_refcount(a, table[0][1], &refcount) == PKV_OK && refcount == 2);

  /* Each sequence's next token lands at offset 3 of the shared last block:
   * the first writer copies that block, the last writer keeps it. */
  int64_t slots[2], pairs[4];
  int num_pairs = -1;
  CHECK(pkv_alloc_append_slots(a, ids, 2, slots, pairs, &num_pairs) == PKV_OK);
  CHECK(num_pairs == 1);
  CHECK(pairs[0] == table[0][1] && pairs[1] != table[0][1]);
  CHECK(slots[0] == pairs[1] * 4 + 3);
  CHECK(slots[1] == (int64_t)table[0][1] * 4 + 3);

  pkv_alloc_stats_t st;
  CHECK(pkv_alloc_stats(a, &st) == PKV_OK);
  CHECK(st.num_seqs == 2 && st.cow_copies == 1);
  CHECK(st.used_blocks == 3 && st.shared_blocks == 1 && st.free_blocks == 13);
  CHECK(st.logical_tokens == 16);

  /* Everything comes back once every sequence is freed. */
  CHECK(pkv_alloc_free_seq(a, 1) == PKV_OK && pkv_alloc_free_seq(a, 2) == PKV_OK);
  CHECK(pkv_alloc_stats(a, &st) == PKV_OK && st.free_blocks == 16 && st.used_blocks == 0);

  /* Errors leave the state unchanged. */
  CHECK(pkv_alloc_free_seq(a, 1) == PKV_ERR_UNKNOWN_SEQ);
  CHECK(pkv_alloc_add_seq(a, 3, 100) == PKV_ERR_OUT_OF_BLOCKS); /* 25 blocks > 16 */
  CHECK(pkv_alloc_stats(a, &st) == PKV_OK && st.free_blocks == 16 && st.num_seqs == 0);
  pkv_alloc_destroy(a);

  /* Split-size queries need no device. */
  const int part = pkv_decode_partition_size(64, 40, 40, 128, 2048);
  CHECK(part > 0 && part % 32 == 0);
  CHECK(pkv_decode_workspace_size(64, 40, 40, 128, 2048, 2048) == 0);
  CHECK(pkv_decode_workspace_size(2, 8, 8, 128, 4096, 1024) == (size_t)2 * 8 * 4 * (128 + 2) * 4);

  /* Argument checks return before any device work. */
  CHECK(pkv_kv_append(NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 16, 4, PKV_F16, NULL) == PKV_OK);
  CHECK(pkv_block_copy(NULL, NULL, NULL, 2, 4, 4090, NULL) == PKV_ERR_INVALID_ARG);

  printf("c abi ok\n");
  return 0;
}
