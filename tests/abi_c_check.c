/*
 * A plain C99 caller of the library's C ABI (include/savgb.h), for the
 * CPU test suite: the header compiles as C, the library links from C, and
 * the host-only calls behave as the header states.  No call here touches a
 * GPU: every one returns before any launch (host logic or argument
 * validation).  Prints "ok" and exits 0, or names the first failed check.
 *
 * Shifted time grid values: with sigma_i = 1 - i/S and
 * sigma' = s*sigma / (1 + (s-1)*sigma), dt_i = sigma'_i - sigma'_(i+1); at
 * s = 3, S = 30 that gives dt_0 = 1 - 87/88 = 1/88 and dt_29 = 3/32 exactly.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "savgb.h"

static int failures = 0;

#define CHECK(cond)                                                  \
  do {                                                               \
    if (!(cond)) {                                                   \
      fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
      ++failures;                                                    \
    }                                                                \
  } while (0)

int main(void) {
  int i, fits = -1;
  int64_t bytes = -1;
  double dt[30], sum = 0.0;
  const int codes[] = {SAVGB_OK, SAVGB_ERR_INVALID_ARG, SAVGB_ERR_UNSUPPORTED, SAVGB_ERR_ALIGNMENT,
                       SAVGB_ERR_OOM, SAVGB_ERR_CUDA, SAVGB_ERR_TIMEOUT, SAVGB_ERR_STATE};
  chunk_stream_config_t cfg;
  chunk_stream_t* s = NULL;
  kv_segment_t seg;
  float x = 0.f;

  CHECK(savgb_version() > 0);
  for (i = 0; i < (int)(sizeof codes / sizeof codes[0]); ++i) {
    const char* name = savgb_status_string(codes[i]);
    CHECK(name != NULL && name[0] != '\0');
  }

  /* flow_time_grid: shift 3 over 30 steps (values in the comment above) */
  CHECK(flow_time_grid(30, 3.0, dt) == SAVGB_OK);
  for (i = 0; i < 30; ++i) {
    CHECK(dt[i] > 0.0);
    sum += dt[i];
  }
  CHECK(fabs(sum - 1.0) < 1e-12);
  CHECK(fabs(dt[0] - 1.0 / 88.0) < 1e-14);
  CHECK(fabs(dt[29] - 3.0 / 32.0) < 1e-14);
  /* uniform grid: shift 1 */
  CHECK(flow_time_grid(4, 1.0, dt) == SAVGB_OK);
  for (i = 0; i < 4; ++i) CHECK(dt[i] == 0.25);
  /* invalid arguments: status and a thread-local message */
  CHECK(flow_time_grid(0, 1.0, dt) == SAVGB_ERR_INVALID_ARG);
  CHECK(strlen(savgb_last_error()) > 0);
  CHECK(flow_time_grid(4, -1.0, dt) == SAVGB_ERR_INVALID_ARG);
  CHECK(flow_time_grid(4, 1.0, NULL) == SAVGB_ERR_INVALID_ARG);

  /* shape queries of the fused-RoPE attention */
  CHECK(chunk_attention_qrope_fits(128, 8, 30, 52, &fits) == SAVGB_OK && fits == 1);
  CHECK(chunk_attention_qrope_fits(96, 2, 4, 4, &fits) == SAVGB_OK && fits == 0); /* head_dim not 64/128 */
  CHECK(chunk_attention_qrope_fits(128, 0, 4, 4, &fits) == SAVGB_ERR_INVALID_ARG);
  CHECK(chunk_attention_qrope_fits(128, 1, 1, 1, NULL) == SAVGB_ERR_INVALID_ARG);
  CHECK(chunk_attention_qrope_table_bytes(128, 8, 30, 52, &bytes) == SAVGB_OK && bytes > 0);
  CHECK(chunk_attention_qrope_table_bytes(96, 8, 30, 52, &bytes) == SAVGB_ERR_UNSUPPORTED);

  /* argument validation before any launch */
  CHECK(rope3d_apply(NULL, NULL, 1, 16, 2, 64, 1, 4, 4, 0, 10000.0, NULL) == SAVGB_ERR_INVALID_ARG);
  seg.k = NULL;
  seg.v = NULL;
  seg.n_tokens = 4;
  CHECK(chunk_attention(NULL, 1, 16, 2, 64, &seg, 1, 0.f, NULL, NULL, NULL) == SAVGB_ERR_INVALID_ARG);
  CHECK(out_proj_euler_step(NULL, NULL, NULL, &x, 16, 128, 128, 0.1f, NULL, NULL) == SAVGB_ERR_INVALID_ARG);
  CHECK(chunk_stream_create(NULL, NULL, &s) == SAVGB_ERR_INVALID_ARG && s == NULL);
  memset(&cfg, 0, sizeof cfg);
  cfg.B = 1;
  cfg.H = 2;
  cfg.D = 96; /* head_dim must be 64 or 128 */
  cfg.F = 2;
  cfg.grid_h = 4;
  cfg.grid_w = 4;
  cfg.ref_frames = 1;
  cfg.ref_t = -1;
  cfg.rope_base = 10000.0;
  CHECK(chunk_stream_create(&cfg, NULL, &s) != SAVGB_OK && s == NULL);
  CHECK(chunk_stream_step(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0.1f, 0) == SAVGB_ERR_INVALID_ARG);
  CHECK(chunk_stream_sync(NULL) == SAVGB_ERR_INVALID_ARG);

  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("ok\n");
  return 0;
}
