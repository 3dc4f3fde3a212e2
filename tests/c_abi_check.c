/* Plain-C user of the libzero ABI: plans the tiny workload and prints the
 * map, so that a test can check the header compiles as C99 and the library
 * links and answers without a GPU. */
#include <stdio.h>

#include "zero.h"

int main(void) {
  const int64_t numels[3] = {4096, 3000, 2904};
  zero_plan_t* plan = NULL;
  zero_plan_info_t info;
  zero_mem_t mem;
  zero_seg_t segs[8];
  int64_t send = 0, recv = 0, n = 0;
  int r, s = zero_plan(numels, 3, 4, 16, NULL, &plan);
  if (s != ZERO_OK) {
    printf("error %s\n", zero_strerror(s));
    return 1;
  }
  zero_plan_info(plan, &info);
  printf("psi %lld psi_pad %lld shard %lld\n", (long long)info.psi, (long long)info.psi_pad,
         (long long)info.shard_total);
  for (r = 0; r < info.n_ranks; ++r) {
    int i;
    zero_plan_segments(plan, r, segs, 8, &n);
    printf("rank %d:", r);
    for (i = 0; i < n; ++i)
      printf(" (%lld %lld %lld %lld)", (long long)segs[i].tensor, (long long)segs[i].tensor_off,
             (long long)segs[i].flat_off, (long long)segs[i].len);
    printf("\n");
  }
  zero_plan_memory(plan, 2, &mem);
  zero_plan_volume(plan, &send, &recv);
  printf("stage2 %lld %lld volume %lld %lld\n", (long long)mem.values, (long long)mem.bytes,
         (long long)send, (long long)recv);
  s = zero_plan(numels, 3, 0, 16, NULL, &plan);
  printf("bad %d %s\n", s, zero_strerror(s));
  zero_plan_destroy(plan);
  return 0;
}
