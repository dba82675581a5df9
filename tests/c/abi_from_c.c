/* Uses libtide from plain C through include/tide.h only: plan creation for
 * the tiny group (three parameters [8,64], [4,64], [12,64] over N = 4), the
 * geometry and level-2 queries, an error status, and destruction.  No call
 * reaches a GPU.  Prints "ok" and returns 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "tide.h"

#define CHECK(cond)                                                \
  do {                                                             \
    if (!(cond)) {                                                 \
      printf("failed: %s (line %d): %s\n", #cond, __LINE__,        \
             tide_last_error());                                   \
      return 1;                                                    \
    }                                                              \
  } while (0)

int main(void) {
  const int32_t ndim[3] = {2, 2, 2};
  const int64_t dims[6] = {8, 64, 4, 64, 12, 64};
  tide_group_desc d;
  tide_plan* plan = NULL;
  int64_t rows, rp, kp, op;
  int32_t order[2];

  memset(&d, 0, sizeof d);
  d.P = 3;
  d.ndim = ndim;
  d.dims = dims;
  d.N = 4;
  d.M = 1;
  d.L = 4;
  CHECK(tide_plan_create(&d, &plan) == TIDE_OK && plan != NULL);
  /* pieces of 2, 1 and 3 rows of 64: S = 384 elements per rank */
  CHECK(tide_plan_shard_elems(plan) == 384);
  CHECK(tide_plan_param_geometry(plan, 2, &rows, &rp, &kp, &op) == TIDE_OK);
  CHECK(rows == 12 && rp == 3 && kp == 64 && op == 192);
  CHECK(tide_plan_level2_order(plan, 0, 3, order) == TIDE_OK && order[0] == 0);
  CHECK(tide_plan_num_items(plan, 0) > 0 && tide_plan_num_items(plan, 1) > 0);
  CHECK(tide_plan_set_option(plan, 99, 0) == TIDE_ERR_INVALID_ARG);
  CHECK(strlen(tide_last_error()) > 0);
  CHECK(tide_rd_rounds(5) == 3 && tide_rd_send_count(5, 2) == 1);
  tide_plan_destroy(plan);

  d.M = 3; /* N != M * L */
  CHECK(tide_plan_create(&d, &plan) == TIDE_ERR_INVALID_ARG);
  CHECK(strcmp(tide_status_string(TIDE_ERR_INVALID_ARG), "invalid argument") == 0);
  tide_plan_destroy(NULL);
  printf("ok\n");
  return 0;
}
