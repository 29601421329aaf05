/*
 * boostattn.h -- C ABI of the attention core of the GB300 low-rank bottleneck
 * block library (the step between the block's grouped Q/K/V up-projection and
 * its O projection).
 *
 * The project page of BOOST ("Move the chunk boundary to the bottleneck", the
 * decoder-block figure) places the attention core between the Q/K/V and the O
 * projections of the LLaMA block, and its paper summary page cites
 * FlashAttention for it; neither gives a formula. This library computes exact
 * multi-head softmax attention, causal or not, with the FlashAttention
 * recomputation scheme (the backward recomputes the probabilities from the
 * saved row log-sum-exp instead of storing them):
 *
 *   s[i, j] = (q_i . k_j) / sqrt(d_head)      per sequence and head
 *   visible(i, j) = j <= i (causal) or always
 *   lse[i] = log sum_{visible j} exp(s[i, j]),  p[i, j] = exp(s[i, j] - lse[i])
 *   o_i = sum_j p[i, j] v_j
 * and for the upstream gradient do, with D_i = do_i . o_i:
 *   dv_j = sum_i p[i, j] do_i,   ds[i, j] = p[i, j] (do_i . v_j - D_i)
 *   dq_i = sum_j ds[i, j] k_j / sqrt(d_head),  dk_j = sum_i ds[i, j] q_i / sqrt(d_head)
 *
 * Layout. q, k, v, o, dout, dq, dk, dv are bf16 [B * L, H * d_head] row-major:
 * sequence b holds token rows b L .. b L + L - 1 and head h the columns
 * h d_head .. h d_head + d_head - 1 -- the layout of the block's Q, K and V
 * outputs with d = H d_head. lse is fp32 [B * H, Lp] with Lp = L rounded up to
 * a multiple of 128 (bn_attn_lse_stride); entries L .. Lp - 1 of a row are
 * written by the forward and carry no meaning.
 *
 * Conventions are those of boostblk.h: device pointers owned by the caller,
 * 16-byte aligned; no device memory allocated; argument errors returned before
 * any launch; launches asynchronous on `stream`; a kernel that gives up on an
 * internal wait records a timeout in the status word at the start of
 * `scratch` (bn_get_device_status reads and clears it); gradients are
 * overwritten. bf16 operands multiply on the tcgen05 tensor cores with fp32
 * accumulation; the softmax runs in fp32 and p is rounded to bf16 before it
 * multiplies v (forward) or do (backward), as FlashAttention does.
 */
#ifndef BOOSTATTN_H
#define BOOSTATTN_H

#include "boostblk.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int64_t B;       /* sequences, >= 1 */
  int64_t L;       /* tokens per sequence, >= 1 */
  int64_t H;       /* heads, >= 1 */
  int64_t d_head;  /* head width: 128 is the one this build implements */
  int32_t causal;  /* 1: key j is visible to query i iff j <= i; 0: every key */
} bn_attn_desc;

/* Row stride of lse and of the backward's row terms: L rounded up to 128. */
int64_t bn_attn_lse_stride(int64_t L);

/* Bytes of lse ([B H, Lp] fp32) and of the scratch buffer: the status word
 * (256 bytes) and the backward's two row terms, [B H, Lp] fp32 each. The
 * forward needs only the status word; the backward the whole buffer. */
bn_status bn_attn_workspace_size(const bn_attn_desc* desc, size_t* lse_bytes,
                                 size_t* scratch_bytes);

/* o = attention(q, k, v) and the row log-sum-exp lse (natural logarithm). */
bn_status bn_attn_forward(const bn_attn_desc* desc, const void* q, const void* k, const void* v,
                          void* o, float* lse, void* scratch, bn_stream_t stream);

/* dq, dk, dv from the forward's inputs, its outputs o and lse, and the
 * upstream gradient dout. Three launches: the row terms D = rowsum(dout * o),
 * dk and dv with key tiles stationary, dq with query tiles stationary. */
bn_status bn_attn_backward(const bn_attn_desc* desc, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* scratch, bn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BOOSTATTN_H */
