/*
 * specverify_testing.h - entry points of libspecverify.so that exist for
 * tests only.  They are not part of the verify-step interface of
 * specverify.h and no production caller needs them.
 */
#ifndef SPECVERIFY_TESTING_H_
#define SPECVERIFY_TESTING_H_

#include "specverify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------
 * sv_test_mla_verify_decode_wait_limit
 *
 * The verify attention of mla_verify_decode_gated (kv_fp8 == 0: kv_pages is
 * the bf16 pool, kv_scale ignored) or of mla_verify_decode_kv8 (kv_fp8 != 0:
 * kv_pages holds E4M3 codes, kv_scale their scale), with every bounded wait
 * of the attention kernel limited to wait_ns nanoseconds of %globaltimer
 * instead of the usual two seconds; with wait_ns == 0 a wait gives up unless
 * the phase it waits for has already completed (a non-blocking test: a poll
 * of the usual wait may suspend the thread until the phase completes, and
 * %globaltimer advances in steps, so a limit of a few nanoseconds is not
 * reliably seen to pass).  The waits that drain
 * outstanding copies and MMAs before a CTA exits keep their usual limit.
 *
 * It lets a test make a wait run out on purpose, to check the guard that
 * turns a stalled pipeline into a reported error rather than a hang or a
 * silently wrong result: the kernel sets SV_DEV_TIMEOUT in *status, gives up
 * its remaining work, drains what it started, frees its TMEM and returns.
 * The outputs of that call are undefined; the device and the library stay
 * usable, and the next call with the usual limit is exact again.
 *
 * wait_ns above two seconds (2e9) returns SV_ERR_SHAPE: the entry point can
 * only shorten the waits, never make them unbounded.  Every other argument,
 * layout, error
 * and ownership rule is that of mla_verify_decode_gated /
 * mla_verify_decode_kv8 in specverify.h.
 * ---------------------------------------------------------------------- */
sv_status sv_test_mla_verify_decode_wait_limit(const void* q_latent, const void* kv_pages, int kv_fp8,
                                               float kv_scale, int num_pages, int page_size,
                                               const int32_t* block_table, int R, int q_per_req,
                                               int max_pages_per_req, const int32_t* kv_bounds,
                                               const void* gate, int gate_dim, int H, float softmax_scale,
                                               int num_splits, int form, void* workspace,
                                               size_t workspace_bytes, void* out, float* lse,
                                               int32_t* status, sv_stream_t stream, uint64_t wait_ns);

/* ------------------------------------------------------------------------
 * sv_test_mla_wuv_project_wait_limit
 *
 * mla_wuv_project with every bounded wait of its kernel limited to wait_ns
 * nanoseconds (0: a wait gives up unless its phase has already completed),
 * as sv_test_mla_verify_decode_wait_limit above.  When a wait gives up the
 * kernel sets SV_DEV_TIMEOUT in *status, writes no output row, waits for the
 * copies and MMAs it started, frees its TMEM and returns.  wait_ns above 2e9
 * returns SV_ERR_SHAPE; everything else as mla_wuv_project in specverify.h.
 * ---------------------------------------------------------------------- */
sv_status sv_test_mla_wuv_project_wait_limit(const void* x, const void* w_uv, int T, int H, int v_dim,
                                             void* out_v, int32_t* status, sv_stream_t stream,
                                             uint64_t wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_TESTING_H_ */
