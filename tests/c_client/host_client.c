/* A plain C client of libpagedkv's host page-table calls (no GPU needed).
 * It runs a fixed scenario and prints what the calls report, one fact per
 * line; tests/test_c_client.py runs the same scenario through the oracle's
 * page table and compares the lines.
 *
 * Scenario (8 pages of 4 rows, free list NULL: page 0 first):
 *   new 0, append 10 rows to 0; new 1, append 5 rows to 1;
 *   fork 0 -> 2; append 1 row to 2 (its shared tail page is copied);
 *   trim 0 to keep_from = 6 (its first page goes); append 1 row to 0. */
#include <stdio.h>

#include "pagedkv.h"

#define CHECK(call)                                          \
  do {                                                       \
    int rc_ = (call);                                        \
    if (rc_ != KVP_OK) {                                     \
      printf("error %d at %s\n", rc_, #call);                \
      return 1;                                              \
    }                                                        \
  } while (0)

static int append(kvp_host* h, int rid, int count) {
  int32_t rids[16], slots[16], twr[16], twc[16], twv[16], cs[16], cd[16];
  int n_tw = 0, n_cow = 0;
  for (int i = 0; i < count; ++i) rids[i] = rid;
  CHECK(kvp_host_append(h, rids, count, slots, twr, twc, twv, 16, &n_tw, cs, cd, &n_cow));
  printf("append %d:", rid);
  for (int i = 0; i < count; ++i) printf(" %d", slots[i]);
  printf("\n");
  for (int i = 0; i < n_cow; ++i) printf("cow %d %d\n", cs[i], cd[i]);
  return 0;
}

static int dump(kvp_host* h, int rid) {
  int32_t row[16];
  int n = 0, len = 0, dropped = 0;
  CHECK(kvp_host_block_row(h, rid, row, 16, &n));
  CHECK(kvp_host_length(h, rid, &len, &dropped));
  printf("row %d len %d:", rid, len);
  for (int i = 0; i < n; ++i) printf(" %d", row[i]);
  printf("\n");
  return 0;
}

int main(void) {
  kvp_host* h = NULL;
  int32_t twr[16], twc[16], twv[16], buf[16];
  int n_tw = 0, n = 0, used = 0;
  CHECK(kvp_host_create(8, 4, 4, NULL, &h));
  CHECK(kvp_host_new(h, 0));
  if (append(h, 0, 10)) return 1;
  CHECK(kvp_host_new(h, 1));
  if (append(h, 1, 5)) return 1;
  CHECK(kvp_host_fork(h, 0, 2, twr, twc, twv, 16, &n_tw));  /* creates request 2 */
  if (append(h, 2, 1)) return 1;
  CHECK(kvp_host_trim(h, 0, 6, twr, twc, twv, 16, &n_tw));
  printf("trim 0: %d released\n", n_tw);
  if (append(h, 0, 1)) return 1;
  for (int r = 0; r < 3; ++r)
    if (dump(h, r)) return 1;
  CHECK(kvp_host_free_list(h, buf, 16, &n));
  printf("free:");
  for (int i = 0; i < n; ++i) printf(" %d", buf[i]);
  printf("\n");
  CHECK(kvp_host_refcounts(h, buf, 8));
  printf("ref:");
  for (int i = 0; i < 8; ++i) printf(" %d", buf[i]);
  printf("\n");
  CHECK(kvp_host_used(h, &used));
  printf("used %d\n", used);
  CHECK(kvp_host_destroy(h));
  return 0;
}
