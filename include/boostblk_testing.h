/*
 * boostblk_testing.h -- test hook into the GEMM engine of libboostblk.
 *
 * Not needed to run a block: it exposes one launch of the engine that
 * bn_block_forward / bn_block_backward use internally, so each fused epilogue
 * and each operand layout can be checked on its own. Every GEMM of the block
 * ("BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank
 * Large Language Models", project page, "Move the chunk boundary to the
 * bottleneck" and "Three supporting changes") is one such launch.
 *
 * Per problem: acc[i, j] = sum_k Aop[i, k] Bop[j, k], i < M, j < N, k < K.
 * An operand is stored row-major either as [MN, K] (mn_major = 0, rows of K
 * elements) or as [K, MN] (mn_major = 1); `ld` is its row stride in elements.
 * Epilogues (bn_gemm_epi):
 *   STORE      out0 = acc * rowv[i] * colv[j]   (rowv fp32, colv element type; optional)
 *   SIGMA      out0 = z = acc, out1 = sigma(z)
 *   NORM       Online RMSNorm over S equal shards of K: rowv = per-row, per-shard
 *              sums of squares [M, S] fp32; z = sum_s (rms_s / rms_g)(P_s / rms_s),
 *              rms_s = sqrt(ss_s/(K/S) + eps), rms_g = sqrt(sum_s ss_s / K + eps);
 *              out0 = z, out1 = sigma(z) (out1 optional)
 *   RESID      out0 = in0 + acc
 *   SWIGLU     G from (a, b), U from (a2, b2): out0 = G, out1 = U (optional), out2 = SiLU(G) U
 *   DSIGMA     out0 = acc * sigma'(in0) * rowv[i]
 *   DSWIGLU    out0 = acc * in1 * SiLU'(in0) * rowv[i], out1 = acc * SiLU(in0) * rowv[i]
 *   CHAIN      acc over (a, b) then (a2, b2) summed, then as STORE
 * All outputs/inputs use leading dimension ldo / ldi.
 */
#ifndef BOOSTBLK_TESTING_H
#define BOOSTBLK_TESTING_H

#include "boostattn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BN_GEMM_STORE = 0, BN_GEMM_SIGMA = 1, BN_GEMM_NORM = 2, BN_GEMM_RESID = 3,
  BN_GEMM_SWIGLU = 4, BN_GEMM_DSIGMA = 5, BN_GEMM_DSWIGLU = 6, BN_GEMM_CHAIN = 7
} bn_gemm_epi;

typedef struct {
  int64_t M, N, K;
  const void* a; const void* a2; int64_t lda; int32_t a_mn_major;
  const void* b; const void* b2; int64_t ldb; int32_t b_mn_major;
  void* out0; void* out1; void* out2; int64_t ldo;
  const void* in0; const void* in1; int64_t ldi;
  const float* rowv; const void* colv;
} bn_gemm_problem;

/* Launch 1..16 problems of one epilogue in one engine launch. dtype: bn_dtype.
 * allow_split lets the tensor-core engine cut the STORE tiles left over after
 * whole rounds of CTA groups into K ranges (fp32 partial tiles in `scratch`
 * after its 256-byte status word, summed in a fixed order by a second kernel).
 * Pointers are device pointers, 16-byte aligned. Asynchronous on `stream`. */
bn_status bn_testing_gemm(int32_t dtype, int32_t epi, int32_t sigma, int32_t S, float eps,
                          int32_t allow_split, int32_t nprob, const bn_gemm_problem* probs,
                          void* scratch, size_t scratch_bytes, bn_stream_t stream);

/* Failure-detection check: one bf16 STORE problem (M <= 256), launched as a
 * chained consumer of an upstream launch that never comes. Its operand
 * producer waits for `counters` (two device ints, zero, that nothing
 * increments) to count the upstream CTAs; after the engine's wait limit (1 s)
 * it records a timeout in the status word at the start of `scratch`, every
 * role of the kernel unwinds, TMEM is freed and the kernel returns. out0 is
 * then not written. Returns BN_OK if the launch was made;
 * bn_get_device_status(scratch) then reports BN_ERR_TIMEOUT. */
bn_status bn_testing_gemm_unfed(const bn_gemm_problem* prob, int* counters, void* scratch,
                                size_t scratch_bytes, bn_stream_t stream);

/* Failure-detection check of the attention core (boostattn.h): the forward,
 * launched with its first stationary (query) tile never loaded. The MMA
 * thread's wait for it gives up after the kernels' wait limit (1 s), every role
 * unwinds, TMEM is freed and the kernel returns; the status word at the start
 * of `scratch` then reads BN_ERR_TIMEOUT (bn_get_device_status). Argument rules
 * as for bn_attn_forward. */
bn_status bn_testing_attn_forward_unfed(const bn_attn_desc* desc, const void* q, const void* k,
                                        const void* v, void* o, float* lse, void* scratch,
                                        bn_stream_t stream);

/* Failure-detection check of bn_weight_grad_noalloc (boostblk.h): the same
 * launch on the library's fixed array, for M <= 256 and with no K split, made a
 * chained consumer of an upstream launch that never comes (`counters`: two
 * device ints, zero, that nothing increments). Its wait gives up after 1 s,
 * every role unwinds and the kernel returns with dW not written;
 * bn_weight_grad_noalloc_status() then reports BN_ERR_TIMEOUT. */
bn_status bn_testing_weight_grad_noalloc_unfed(int64_t M, int64_t N, int64_t T, const void* A,
                                               int64_t lda, const void* B, int64_t ldb, void* dW,
                                               int64_t ldw, int* counters, bn_stream_t stream);

/* One launch of the block's RMSNorm backward (bf16; the kernel the block's
 * backward runs for these rows), then its dw column sums:
 *   dx[t, j] = dres[t, j] + dn[t, j] w[j] - x[t, j] rstd[t]^2 sum_k(dn w x)[t, k] / d
 *   dw[j]    = sum_t dn[t, j] x[t, j]
 * where dn is the gradient of the normalised input already multiplied by the
 * row's rstd. All tensors [rows, d] row-major (d a multiple of 8), w [d];
 * `part` is fp32 scratch of part_elems >= 2 x SMs x d. With `unfed` != 0 (d at
 * most 5120) the first row of the kernel's first warp is never loaded: that
 * warp's bounded wait gives up after 1 s, the kernel records a timeout in the
 * status word at the start of `scratch` (bn_get_device_status reports
 * BN_ERR_TIMEOUT), waits (bounded) for its other copies in flight and returns;
 * dx and dw are then not meaningful. Returns BN_OK if the launches were made. */
bn_status bn_testing_norm_bwd(int64_t rows, int64_t d, const void* dn, const void* x,
                              const void* w, const float* rstd, const void* dres, void* dx,
                              void* dw, float* part, int64_t part_elems, int32_t unfed,
                              void* scratch, bn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BOOSTBLK_TESTING_H */
