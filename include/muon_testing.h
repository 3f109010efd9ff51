/*
 * muon_testing.h -- test hooks of the Muon library (not needed by users).
 *
 * They run one building block of the TENSOR path on caller buffers so a test
 * can compare it with an independent matrix product.  Unlike muon_step they
 * may allocate (a few bytes of device scalars) and they synchronise `stream`.
 */
#ifndef MUON_GB300_TESTING_H
#define MUON_GB300_TESTING_H

#include "muon.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One batched tcgen05 product of a Newton-Schulz step («关于分布式Muon的想法整合
 * 及讨论» §2: the Gram matrix and the products that follow it), on contiguous
 * row-major device buffers of 16-bit elements (ns_dtype: muon_ns_dtype_t):
 *   op 0 (Gram):   out[B][m][m] = y y^T / alpha^2,   y   [B][m][n]
 *   op 1 (poly):   out[B][m][m] = pa I + pb a + pc a a,  a [B][m][m] (symmetric)
 *   op 2 (update): out[B][m][n] = q y,               q   [B][m][m], y [B][m][n]
 * Needs m % 8 == 0 and n % 8 == 0 (16-byte rows).  INVALID_ARG otherwise;
 * CUDA on a failed launch; TIMEOUT if the kernel gave up a bounded wait. */
MUON_API muon_status_t muon_testing_tc_gemm(int32_t op, int32_t ns_dtype, int32_t B, int64_t m,
                                            int64_t n, const void* y, const void* a,
                                            const void* q, void* out, float alpha, float pa,
                                            float pb, float pc, void* stream);

/* The 128-row x bn-column tiles one batch item of the one-CTA form of a
 * tcgen05 product (op as in muon_testing_tc_gemm; groups with
 * min(rows, cols) < 256) computes, in launch order.  op 0 / 1: the Gram and
 * polynomial outputs are symmetric m x m (n is ignored), so only tiles that
 * reach the upper triangle run; each writes its elements with col >= row in
 * place and mirrors those with col > row.  op 2: every tile of the m x n
 * update, in groups of 8 tile rows that sweep the tile columns together.
 * For t = 0 .. count-1, tm[t] and tn[t] receive tile t's row and column;
 * entries past cap are not written.  Returns count, or -1 for another op,
 * m (or, for op 2, n) outside [1, 2^20], bn other than 128 or 256, cap < 0,
 * or a NULL array with cap > 0.  Host only: no device. */
MUON_API int32_t muon_testing_tile_walk(int32_t op, int64_t m, int64_t n, int32_t bn,
                                        int32_t* tm, int32_t* tn, int32_t cap);

/* The same walk for the CTA-pair form of the products (a cluster of two CTAs
 * per 256 x 256 tile, tcgen05.mma.cta_group::2), which groups with
 * min(rows, cols) >= 256 use: tm[t] / tn[t] count 256-row / 256-column
 * tiles.  The products are those of muon_testing_tc_gemm («关于分布式Muon的
 * 想法整合及讨论» §2).  Same return values and errors as
 * muon_testing_tile_walk.  Host only. */
MUON_API int32_t muon_testing_tile_walk_pair(int32_t op, int64_t m, int64_t n, int32_t* tm,
                                             int32_t* tn, int32_t cap);

/* 1 when a group of min dim m runs its products in the CTA-pair form, else 0.
 * Host only. */
MUON_API int32_t muon_testing_tc_pair_form(int64_t m);

/* Number of skinny-path clusters (one per member of min dim m, 1..64) that the
 * current device can hold at once for the given operand type; -1 on error. */
MUON_API int32_t muon_testing_skinny_max_clusters(int32_t ns_dtype, int64_t m);

/* Failure detection without a GPU fault: one kernel waits on an mbarrier with
 * the bounded wait every wait of this library uses, for at most limit_cycles
 * SM cycles (1 .. 2^33).  arrive != 0: a second thread completes the barrier
 * and the call returns OK.  arrive == 0: nothing completes it, the wait gives
 * up, the kernel records the timeout in an error word and ends normally, and
 * the call returns TIMEOUT; the context stays usable.  INVALID_ARG for a
 * limit out of range; CUDA or OOM on a runtime failure.  Synchronises
 * `stream`. */
MUON_API muon_status_t muon_testing_wait_probe(int32_t arrive, int64_t limit_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_TESTING_H */
