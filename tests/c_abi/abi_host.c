/* Host-only checks of the C ABI from plain C99 (no device is touched): the
 * headers compile as C, the library links, and the planning calls and error
 * statuses behave as include/muon.h states.  Exit status 0 = all passed. */
#include <stdio.h>
#include <string.h>

#include "muon.h"
#include "muon_testing.h"

static int failures = 0;
#define CHECK(cond, what)                                          \
  do {                                                             \
    if (!(cond)) {                                                 \
      fprintf(stderr, "FAIL %s:%d: %s\n", __FILE__, __LINE__, what); \
      ++failures;                                                  \
    }                                                              \
  } while (0)

static muon_shape_t shape2(int64_t r, int64_t c) {
  muon_shape_t s;
  memset(&s, 0, sizeof s);
  s.ndim = 2;
  s.dims[0] = r;
  s.dims[1] = c;
  return s;
}

static muon_shape_t shape3(int64_t e, int64_t r, int64_t c) {
  muon_shape_t s = shape2(r, c);
  s.ndim = 3;
  s.dims[0] = e;
  s.dims[1] = r;
  s.dims[2] = c;
  return s;
}

int main(void) {
  muon_plan_options o;
  CHECK(muon_default_options(&o) == MUON_OK, "default options");
  CHECK(o.mode == MUON_MODE_BF16 && o.eps > 0.f && o.column_shards == 0 && o.flags == 0u,
        "default option values");
  CHECK(muon_default_options(NULL) == MUON_ERR_INVALID_ARG, "NULL options pointer");
  CHECK(muon_version() != NULL && strlen(muon_version()) > 0, "version string");
  CHECK(muon_status_string(MUON_ERR_INVALID_ARG) != NULL, "status string");

  /* 74 x [24, 10240]: one group of 74 members */
  muon_shape_t c2[74];
  for (int i = 0; i < 74; ++i) c2[i] = shape2(24, 10240);
  int32_t ng = 0;
  int64_t nm = 0;
  size_t ws = 0;
  muon_group_info_t g[4];
  int32_t mp[80], me[80];
  CHECK(muon_plan_describe(c2, 74, NULL, g, 4, &ng, mp, me, 80, &nm, &ws) == MUON_OK, "describe c2");
  CHECK(ng == 1 && nm == 74 && g[0].batch == 74 && g[0].rows == 24 && g[0].cols == 10240, "c2 groups");
  CHECK(g[0].path == MUON_PATH_SKINNY && g[0].transposed == 0 && ws > 0, "c2 path and workspace");
  CHECK(mp[73] == 73 && me[73] == 0, "c2 member order");

  /* orientation merge: [r, c] and [c, r] share a group with the flag */
  muon_shape_t mix[4] = {shape2(4096, 16384), shape2(16384, 4096), shape3(2, 4096, 16384), shape2(64, 64)};
  CHECK(muon_plan_describe(mix, 4, NULL, g, 4, &ng, NULL, NULL, 0, &nm, NULL) == MUON_OK, "describe mix");
  CHECK(ng == 3 && nm == 5, "separate orientations");
  o.flags = MUON_FLAG_MERGE_TRANSPOSED;
  CHECK(muon_plan_describe(mix, 4, &o, g, 4, &ng, NULL, NULL, 0, &nm, NULL) == MUON_OK, "describe merged");
  CHECK(ng == 2 && g[0].batch == 4 && g[0].transposed == 2, "merged orientations");

  /* ownership planner: 74 equal members over 8 replicas, 9 or 10 each */
  int32_t owner[74];
  double rank_cost[8];
  CHECK(muon_plan_assign(c2, 74, NULL, 5, 8, owner, 74, NULL, rank_cost) == MUON_OK, "assign");
  int count[8] = {0};
  for (int i = 0; i < 74; ++i) {
    CHECK(owner[i] >= 0 && owner[i] < 8, "owner in range");
    if (owner[i] >= 0 && owner[i] < 8) ++count[owner[i]];
  }
  for (int r = 0; r < 8; ++r) CHECK(count[r] == 9 || count[r] == 10, "even spread");

  /* errors are statuses, with a message */
  muon_shape_t bad = shape2(0, 4);
  CHECK(muon_plan_describe(&bad, 1, NULL, NULL, 0, &ng, NULL, NULL, 0, NULL, NULL) == MUON_ERR_INVALID_ARG,
        "empty dim");
  CHECK(muon_last_error() != NULL && strlen(muon_last_error()) > 0, "error message");
  CHECK(muon_plan_describe(NULL, 1, NULL, NULL, 0, &ng, NULL, NULL, 0, NULL, NULL) == MUON_ERR_INVALID_ARG,
        "NULL shapes");
  muon_default_options(&o);
  o.column_shards = 3;
  CHECK(muon_plan_describe(c2, 1, &o, NULL, 0, &ng, NULL, NULL, 0, NULL, NULL) == MUON_ERR_INVALID_ARG,
        "bad column_shards");
  muon_default_options(&o);
  o.flags = 1u << 20;
  CHECK(muon_plan_describe(c2, 1, &o, NULL, 0, &ng, NULL, NULL, 0, NULL, NULL) == MUON_ERR_INVALID_ARG,
        "unknown flag bits");
  CHECK(muon_step(NULL, NULL, NULL, NULL, 0.9f, 0.02f, 0.1f, 5, 3.4445f, -4.775f, 2.0315f, NULL) ==
            MUON_ERR_INVALID_ARG,
        "NULL plan");
  float rows[3] = {3.4445f, -4.775f, 2.0315f};
  CHECK(muon_step_schedule(NULL, NULL, NULL, NULL, 0.9f, 0.02f, 0.1f, 5, rows, 1, NULL) == MUON_ERR_INVALID_ARG,
        "NULL plan (schedule)");
  CHECK(muon_plan_num_groups(NULL) == 0, "groups of a NULL plan");

  /* the GEMMs' tile walks (host only): m = 300 with 128 x 128 tiles is the
   * upper triangle of a 3 x 3 tile grid, row by row, for the Gram; the
   * update of a 300 x 400 output sweeps 3 tile rows together */
  int32_t tm[16], tn[16];
  CHECK(muon_testing_tile_walk(0, 300, 0, 128, tm, tn, 16) == 6, "sym tile count");
  CHECK(tm[0] == 0 && tn[0] == 0 && tm[2] == 0 && tn[2] == 2 && tm[3] == 1 && tn[3] == 1 &&
            tm[5] == 2 && tn[5] == 2,
        "sym tile order");
  CHECK(muon_testing_tile_walk(2, 300, 400, 128, tm, tn, 16) == 12, "update tile count");
  CHECK(tm[0] == 0 && tn[0] == 0 && tm[1] == 1 && tn[1] == 0 && tm[3] == 0 && tn[3] == 1,
        "update tile order");
  CHECK(muon_testing_tile_walk(0, 300, 0, 96, NULL, NULL, 0) == -1, "tile walk: bad width");
  CHECK(muon_testing_tile_walk(3, 300, 300, 128, NULL, NULL, 0) == -1, "tile walk: bad op");

  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("c abi host checks passed\n");
  return 0;
}
