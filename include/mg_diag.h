/*
 * mg_diag.h -- device measurements that bound the attention path's time per call from
 * below, exported by the same library as mg_attn.h (libmgattn.so).
 *
 * They are not part of the computation. They measure two ceilings that the roofline of
 * the exp-normalised GQA graph (4 B M N d flops at the tensor peak, the Q+K+V+O bytes at
 * the HBM bandwidth) does not contain:
 *
 *   - the launch floor: how often a kernel with the fused kernel's launch shape can be
 *     launched back to back when it does nothing but that kernel's prologue and teardown
 *     (tensor-memory allocation, the programmatic-dependent-launch handshake, the cluster
 *     barrier); no call of mg_attn_run can take less on the same stream;
 *   - the exponential rate: E = exp(A) of the graph (Mirage documentation,
 *     tutorials/group-query-attention, "Define GQA Computation Graph") needs B M N
 *     exponentials; this measures how many the instruction sequence of the fused kernel's
 *     softmax warps delivers per SM clock.
 *
 * Both calls are synchronous: they run on a stream of their own, wait for it and return
 * the figure. Status codes are those of mg_attn.h; the detail of a failure is in
 * mg_diag_last_error(). No call prints, aborts or exits the process.
 */
#ifndef MG_DIAG_H_
#define MG_DIAG_H_

#include <stdint.h>

#include "mg_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Average time per launch, in microseconds, of `launches` back-to-back launches (replayed
 * from one CUDA graph, after a warm-up replay) of a no-work kernel on the current device with
 *   ctas        grid size (1 .. 65535; a multiple of `cluster`)
 *   cluster     thread-block cluster size (1 = none, else 2 .. 16); every CTA passes one
 *               cluster barrier when > 1
 *   smem_bytes  dynamic shared memory per CTA; at least 120 KB (so that no two CTAs share an
 *               SM: each holds all 512 tensor-memory columns, as the fused kernel does) and
 *               at most the device's opt-in limit
 *   pdl         nonzero: programmatic dependent launch, as mg_attn_run uses by default
 *   launches    1 .. 100000
 * Each CTA has as many threads as the fused kernel. Errors: MG_ERR_INVALID_ARG (a NULL
 * output or a value out of range), MG_ERR_CONFIG (the cluster cannot be scheduled),
 * MG_ERR_CUDA. */
mg_status mg_diag_launch_floor(int32_t ctas, int32_t cluster, int32_t smem_bytes, int32_t pdl, int32_t launches,
                               float *us_per_launch);

/* Exponentials per SM clock and per SM nanosecond of the fused kernel's exponential: one
 * two-wide fp32 multiply by log2(e), then ex2.approx on the MUFU unit, for pairs of fp32
 * values; poly != 0 measures the fused kernel's alternative on the FMA pipe (a degree-5
 * polynomial of 2^f after a Cody-Waite split) instead. One CTA of 512 threads per SM, each
 * thread running `iters` rounds of eight independent pairs (1 .. 1000000); the figure is the
 * median over the CTAs of (exponentials / elapsed SM clocks), and of (exponentials /
 * elapsed global-timer ns). Errors: MG_ERR_INVALID_ARG, MG_ERR_CUDA. */
mg_status mg_diag_exp_rate(int32_t iters, int32_t poly, double *exp_per_clk_per_sm, double *exp_per_ns_per_sm);

/* Detail of the last failure of an mg_diag call on the calling thread; "" if none. */
const char *mg_diag_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MG_DIAG_H_ */
