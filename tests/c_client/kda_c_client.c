/*
 * A plain C99 client of libkda: it compiles against include/kda.h alone and
 * links every function the header declares, so a declaration without an
 * exported definition (or with a different C name) fails the link.  Without
 * a GPU it runs the calls that need none: the version and status strings,
 * the dispatch policy queries, and the host-side contract checks, which
 * must reject a malformed call with a status and a message before any CUDA
 * work.  Exit status 0 when every check holds.
 */
#include <stdio.h>
#include <string.h>

#include "kda.h"

static int failures = 0;

static void expect(int ok, const char* what) {
  if (!ok) {
    fprintf(stderr, "FAILED: %s\n", what);
    ++failures;
  }
}

typedef void (*any_fn)(void);

int main(void) {
  /* Every entry point of the header, taken by address. */
  const any_fn fns[] = {
      (any_fn)kda_recurrent_decode,   (any_fn)kda_packed_decode,      (any_fn)kda_fused_decode,
      (any_fn)kda_spec_decode,        (any_fn)kda_spec_verify_decode, (any_fn)kda_packed_fused_decode,
      (any_fn)kda_plan_split,         (any_fn)kda_set_split_override, (any_fn)kda_plan_schedule,
      (any_fn)kda_set_schedule_override, (any_fn)kda_device_error,    (any_fn)kda_selftest_wait_timeout,
      (any_fn)kda_status_string,      (any_fn)kda_last_error_message, (any_fn)kda_version};
  size_t i;
  for (i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i) expect(fns[i] != NULL, "declared function resolves");

  expect(kda_version() != NULL && strlen(kda_version()) > 0, "version string");
  expect(strcmp(kda_status_string(KDA_OK), "KDA_OK") == 0, "status string of KDA_OK");
  expect(strcmp(kda_status_string(KDA_ERR_INVALID_ARG), "KDA_ERR_INVALID_ARG") == 0,
         "status string of KDA_ERR_INVALID_ARG");

  /* Dispatch policy: valid queries give a split and a schedule, invalid ones 0. */
  expect(kda_plan_split(KDA_OP_RECURRENT, 16384, KDA_F32, 1, 152) > 0, "split of a valid query");
  expect(kda_plan_schedule(KDA_OP_RECURRENT, 16384, KDA_F32, 1, 152) > 0, "schedule of a valid query");
  expect(kda_plan_split(9, 1, KDA_F32, 1, 152) == 0, "split of an unknown operation");
  expect(kda_plan_split(KDA_OP_RECURRENT, 1, 7, 1, 152) == 0, "split of an unknown dtype");
  expect(kda_set_split_override(3) == KDA_ERR_INVALID_ARG, "override with a split that has no kernel");
  expect(kda_set_split_override(0) == KDA_OK, "override cleared");

  /* Contract checks before any CUDA work: null descriptors, then rank 0. */
  {
    kda_tensor t;
    const kda_tensor* p = &t;
    kda_status s = kda_recurrent_decode(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 0.f,
                                        0.088388f, NULL);
    expect(s == KDA_ERR_INVALID_ARG, "null descriptors rejected");
    expect(strlen(kda_last_error_message()) > 0, "message for null descriptors");
    memset(&t, 0, sizeof(t));
    s = kda_recurrent_decode(p, p, p, p, p, p, p, p, p, p, 0, 0.f, 0.088388f, NULL);
    expect(s == KDA_ERR_INVALID_ARG, "rank-0 descriptors rejected");
    expect(strstr(kda_last_error_message(), "ndim") != NULL, "message names the rank");
    s = kda_packed_decode(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
    expect(s == KDA_ERR_INVALID_ARG, "packed: null descriptors rejected");
  }

  if (failures == 0) printf("kda C client: all checks passed\n");
  return failures == 0 ? 0 : 1;
}
