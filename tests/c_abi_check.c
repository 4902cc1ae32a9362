/* A plain C caller of the library, compiled and run by tests/test_c_abi.py: the header must
 * compile as C, the library must link, and the calls that need no GPU must behave as the
 * header states.  Prints "ok" and exits 0 on success; prints the failed check otherwise. */
#include <stdio.h>
#include <string.h>

#include "moe_gb300.h"

#define CHECK(cond)                                        \
  do {                                                     \
    if (!(cond)) {                                         \
      printf("failed: %s (line %d)\n", #cond, __LINE__);   \
      return 1;                                            \
    }                                                      \
  } while (0)

int main(void) {
  moe_config_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.T_max = 1024;
  cfg.H = 512;
  cfg.I = 256;
  cfg.E = 16;
  cfg.top_k = 4;
  cfg.schedule = MOE_SCHED_AUTO;
  size_t bytes = 0;
  CHECK(moe_workspace_bytes(&cfg, &bytes) == MOE_OK);
  CHECK(bytes > (size_t)cfg.T_max * cfg.top_k * (size_t)(2 * cfg.I + 2 * cfg.H));

  moe_config_t bad = cfg;
  bad.H = 500; /* not a multiple of 64 */
  CHECK(moe_workspace_bytes(&bad, &bytes) == MOE_ERR_UNSUPPORTED);
  bad = cfg;
  bad.top_k = 0;
  CHECK(moe_workspace_bytes(&bad, &bytes) == MOE_ERR_INVALID_ARG);
  CHECK(moe_workspace_bytes(NULL, &bytes) == MOE_ERR_INVALID_ARG);

  CHECK(moe_status_string(MOE_OK) != NULL && strlen(moe_status_string(MOE_OK)) > 0);
  CHECK(moe_status_string(MOE_ERR_TIMEOUT) != NULL);
  CHECK(moe_host_wait(NULL, NULL) == MOE_ERR_INVALID_ARG);   /* rejected before any CUDA call */

  /* host evaluation of the tile schedule: 3 experts with 300, 0 and 40 rows */
  int32_t counts[3] = {300, 0, 40};
  int64_t n[2] = {0, 0};
  CHECK(moe_schedule_host(counts, 3, cfg.H, cfg.I, 74, MOE_SCHED_WAVE_SERIAL, 0, 1, NULL, 0, n) == MOE_OK);
  /* units: ceil(300/256) + ceil(40/256) = 3; Linear-1 tiles = 3 * I/128, all tiles = 3 * (I/128 + H/256) */
  CHECK(n[0] == 3 * (cfg.I / 128));
  CHECK(n[1] == 3 * (cfg.I / 128 + cfg.H / 256));
  int32_t tiles[4 * 64];
  CHECK(moe_schedule_host(counts, 3, cfg.H, cfg.I, 74, MOE_SCHED_WAVE_SERIAL, 0, 1, tiles, 64, n) == MOE_OK);
  for (int64_t i = 0; i < n[1]; ++i) {
    const int phase = tiles[4 * i] & 1, expert = tiles[4 * i + 1];
    CHECK(expert == 0 || expert == 2);                  /* the expert without rows has no tile */
    CHECK(phase == (i >= n[0]));                        /* every Linear-1 tile before the Linear-2 tiles */
  }
  printf("ok\n");
  return 0;
}
