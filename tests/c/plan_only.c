/* A C99 caller of the library's planner (no GPU needed): plans three tensors
 * into 4 ranks and prints the layout the planner chose, one value per line. */
#include <stdint.h>
#include <stdio.h>

#include "dpsync.h"

int main(void) {
  const int64_t sizes[3] = {1000, 70000, 12};
  const uint8_t decay[3] = {1, 1, 0};
  dp_plan* plan = NULL;
  if (dp_plan_buckets(sizes, decay, 3, 64 * 1024, 4, &plan) != DP_OK) {
    fprintf(stderr, "plan: %s\n", dp_last_error());
    return 1;
  }
  dp_plan_info_t info;
  if (dp_plan_info(plan, &info) != DP_OK) return 2;
  printf("%lld\n%lld\n%d\n", (long long)info.n_params, (long long)info.padded_len, info.n_buckets);
  for (int32_t t = 0; t < 3; ++t) {
    int32_t b = -1;
    int64_t off = -1;
    if (dp_plan_tensor(plan, t, &b, &off) != DP_OK) return 3;
    printf("%d %lld\n", b, (long long)off);
  }
  /* the layout fingerprint, and the cross-process check against a second rank's */
  uint64_t fp = 0;
  if (dp_plan_fingerprint(plan, &fp) != DP_OK) return 4;
  printf("%016llx\n", (unsigned long long)fp);
  uint64_t ranks[2] = {fp, fp};
  const int same = dp_plan_check_match(plan, ranks, 2);
  ranks[1] = fp ^ 1u;
  const int differ = dp_plan_check_match(plan, ranks, 2);
  printf("%d %d\n", same == DP_OK, differ == DP_EPLAN);
  /* a refused call leaves a message and no plan */
  dp_plan* bad = NULL;
  const int rc = dp_plan_buckets(sizes, decay, 3, 64 * 1024, 0, &bad);
  printf("%d %d\n", rc == DP_EINVAL, bad == NULL);
  /* the workspace's result fields: the header's offsets, then the library's */
  int64_t offs[4] = {-1, -1, -1, -1};
  if (dp_workspace_result_offsets(offs) != DP_OK) return 5;
  printf("%d %d %d %d\n", DP_WS_NORM2_OFFSET, DP_WS_NORM_OFFSET, DP_WS_COEF_OFFSET,
         DP_WS_STATUS_OFFSET);
  printf("%lld %lld %lld %lld\n", (long long)offs[0], (long long)offs[1], (long long)offs[2],
         (long long)offs[3]);
  dp_plan_free(plan);
  return 0;
}
