/*
 * boostblk.h -- C ABI of the GB300 low-rank bottleneck block library.
 *
 * One CoLA-style decoder block, forward and backward, on one GPU (sm_103a).
 * Every linear layer of the block is a bottleneck  out = B . sigma(A . x)
 * with A [r, d_in] (down-projection) and B [d_out, r] (up-projection);
 * "BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank Large
 * Language Models", project page, section "Move the chunk boundary to the
 * bottleneck" (first paragraph and the decoder-block figure).
 *
 * The block (full kind), with sigma = SiLU or identity:
 *   z_qkv = OnlineRMSNorm_S(x; w_norm1) . A_qkv^T         [T, 3r]  grouped Q/K/V down
 *   Q, K, V = sigma(z_q) B_q^T, sigma(z_k) B_k^T, sigma(z_v) B_v^T   [T, d] each
 *   x1 = x + sigma(V A_o^T) B_o^T        (attention core outside the block; with
 *                                          desc.attn = 1, O = attention(Q, K, V) replaces V)
 *   z_gu = OnlineRMSNorm_S(x1; w_norm2) . A_gu^T           [T, 2r]  grouped gate/up down
 *   G, U = sigma(z_g) B_g^T, sigma(z_u) B_u^T              [T, d_ff]
 *   m = SiLU(G) * U ;  y = x1 + sigma(m A_d^T) B_d^T
 * The MLP kind is the second half alone with x1 = x.
 *
 * Online RMSNorm: the hidden dimension is split into S equal column shards;
 * each shard's slice of the down-projection is normalised by the shard's own
 * RMS and the per-row correction alpha = RMS_local / RMS_global is applied in
 * the GEMM epilogue, which gives plain RMSNorm exactly (project page, "Three
 * supporting changes" -> Online RMSNorm; BOOST-MLSys26 summary page, core
 * method -> Online RMSNorm). RMS = sqrt(mean of squares + eps), eps inside
 * both the local and the global square root.
 * Grouping (project page, "Three supporting changes" -> Linear layer
 * grouping): the Q/K/V down-projections are one GEMM over
 * A_qkv = [A_q; A_k; A_v], the gate/up ones one GEMM over A_gu = [A_g; A_u];
 * the up-projections of a group run in one launch.
 * Checkpointing (same section -> Checkpointing without communication): with
 * desc.checkpoint = 1 the forward saves only the r-wide pre-activations
 * z_qkv, z_o, z_gu, z_d and the backward recomputes everything else.
 *
 * Conventions (all entry points):
 *  - Row-major everywhere. Weights are [out, in]. Token rows are T.
 *  - All pointers are device pointers owned by the caller; the library
 *    allocates no device memory and keeps no state except cached device
 *    properties. Every pointer must be 16-byte aligned.
 *  - The element type of every tensor is desc.dtype (fp32 or bf16). bf16 runs
 *    multiply on the tensor cores and accumulate in fp32; fp32 runs use plain
 *    fp32 FFMA.
 *  - Argument errors return synchronously, before anything is launched.
 *    Launches are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). A kernel whose internal wait exceeds its time limit
 *    records a timeout in the status word at the start of `scratch`, which
 *    bn_get_device_status() reads.
 *  - Gradients are overwritten, never accumulated.
 *  - d_ff-wide tensors (A_d, its gradient, and internal G, U, m) use the
 *    leading dimension desc.ld_ff >= d_ff; columns d_ff .. ld_ff-1 are neither
 *    read nor written.
 */
#ifndef BOOSTBLK_H
#define BOOSTBLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bn_stream_t; /* the same type as cudaStream_t */

typedef enum {
  BN_OK = 0,
  BN_ERR_INVALID_ARG = 1, /* a size, enum or pointer is out of range */
  BN_ERR_ALIGNMENT = 2,   /* a pointer or leading dimension breaks the 16-byte rule */
  BN_ERR_UNSUPPORTED = 3, /* valid, but outside what this build implements */
  BN_ERR_CUDA = 4,        /* a CUDA runtime call failed (see bn_last_cuda_error) */
  BN_ERR_TIMEOUT = 5      /* a kernel gave up on an internal wait (device status) */
} bn_status;

typedef enum { BN_F32 = 0, BN_BF16 = 1 } bn_dtype;
typedef enum { BN_SIGMA_IDENTITY = 0, BN_SIGMA_SILU = 1 } bn_sigma;
typedef enum { BN_BLOCK_FULL = 0, BN_BLOCK_MLP = 1 } bn_kind;

/* Shapes and options of one block. */
typedef struct {
  int64_t T;      /* tokens (micro-batch x sequence), >= 1 */
  int64_t d;      /* hidden width; d % S == 0; bf16 also needs (d / S) % 64 == 0 */
  int64_t r;      /* bottleneck rank; a multiple of 8 */
  int64_t d_ff;   /* MLP width, >= 1 */
  int64_t ld_ff;  /* leading dimension of d_ff-wide tensors: >= d_ff, a multiple of 8 */
  int32_t S;      /* emulated column shards of Online RMSNorm, 1 .. 16 */
  int32_t sigma;  /* bn_sigma: the bottleneck nonlinearity */
  int32_t dtype;  /* bn_dtype */
  int32_t kind;   /* bn_kind */
  int32_t dense;  /* 1 = full-rank baseline block: A_* hold the dense W, B_* are NULL */
  int32_t checkpoint; /* 1 = save only the r-wide pre-activations (factorised block only) */
  float eps;      /* RMSNorm epsilon, e.g. 1e-5 */
  /* 1 = bottleneck-aware tensor parallelism emulated over the S shards (factorised
   * block only; BOOST page, "Move the chunk boundary to the bottleneck"): every
   * row-parallel down-projection (also the O and down-projection ones) and every
   * up-projection's input gradient sums S per-shard partial products in its
   * epilogue, in shard order -- the chunk's r-wide all-reduce, 7r values per
   * token and pass. The d_ff shards are whole 64-column blocks (the last ones one
   * block shorter when 64 S does not divide d_ff). Results equal the plain
   * block's up to rounding. 0 = each of those GEMMs sums over all of K at once. */
  int32_t btp;
  /* 1 = the attention core runs inside the block (full kind, bf16, d a multiple
   * of 128; see boostattn.h): T = (T / seq_len) causal sequences of seq_len
   * tokens, d / 128 heads of 128; the O projection reads
   * O = softmax(Q K^T / sqrt(128) + causal mask) V instead of V. The block is
   * then the whole decoder layer: q_out, k_out (forward) and dq, dk (backward)
   * must be NULL, and Q, K, O and the attention's row log-sum-exp join the saved
   * activations (recomputed in checkpoint mode). 0 = the attention core runs
   * outside: the O projection reads V, Q and K leave through q_out and k_out. */
  int32_t attn;
  int32_t seq_len; /* tokens per sequence when attn = 1 (T % seq_len == 0); else ignored */
  /* Bottlenecks of uneven size (BOOST page, Limitations -> "Untested extensions":
   * the design also covers bottlenecks of different sizes): the rank of each
   * factorised layer, in the order q, k, v, o, gate, up, down; 0 = r. Each is a
   * multiple of 8. The grouped factors stack their layers' rows: A_qkv is
   * [r_q + r_k + r_v, d], A_gu [r_g + r_u, d]. All zero for the dense block. */
  int64_t r_layer[7];
} bn_block_desc;

/* Parameters (forward) or their gradients (backward). Shapes, low-rank block
 * (every layer of rank r; with desc.r_layer, layer i's r_i in its place):
 *   w_norm1 [d], A_qkv [3r, d], B_q/B_k/B_v [d, r], A_o [r, d], B_o [d, r],
 *   w_norm2 [d], A_gu [2r, d], B_g/B_u [d_ff, r], A_d [r, ld_ff], B_d [d, r].
 * Dense block: A_qkv [3d, d], A_o [d, d], A_gu [2 d_ff, d], A_d [d, ld_ff], B_* NULL.
 * MLP kind: w_norm1, A_qkv, B_q, B_k, B_v, A_o, B_o are NULL. */
typedef struct {
  void* w_norm1; void* A_qkv; void* B_q; void* B_k; void* B_v; void* A_o; void* B_o;
  void* w_norm2; void* A_gu; void* B_g; void* B_u; void* A_d; void* B_d;
} bn_block_params;

/* Bytes the caller must provide: `saved` (activations kept from forward to
 * backward) and `scratch` (temporaries of either pass). The first 256 bytes of
 * `scratch` hold the device status word and the kernels' own counters: zero
 * them once before the first call (the library keeps them consistent after
 * that). Both sizes depend on desc only. */
bn_status bn_block_workspace_size(const bn_block_desc* desc, size_t* saved_bytes,
                                  size_t* scratch_bytes);

/* Forward pass. x [T, d] in; y [T, d] out; q_out, k_out [T, d] out for the
 * full kind (NULL for the MLP kind). `saved` receives what the backward reads. */
bn_status bn_block_forward(const bn_block_desc* desc, const bn_block_params* W,
                           const void* x, void* y, void* q_out, void* k_out,
                           void* saved, void* scratch, bn_stream_t stream);

/* Backward pass for upstream gradients dy [T, d] and dq, dk [T, d] (full kind;
 * either may be NULL, meaning zero). `saved` must come from bn_block_forward
 * with the same desc, W and x. Writes dx [T, d] and every gradient in dW
 * (same shapes as W). Outputs may not alias inputs. */
bn_status bn_block_backward(const bn_block_desc* desc, const bn_block_params* W,
                            const void* x, const void* saved, const void* dy,
                            const void* dq, const void* dk, void* dx,
                            const bn_block_params* dW, void* scratch, bn_stream_t stream);

/* Synchronises `stream`, reads and clears the device status word at the start
 * of `scratch`, and returns BN_OK or BN_ERR_TIMEOUT (BN_ERR_CUDA if the
 * synchronisation itself failed). */
bn_status bn_get_device_status(void* scratch, bn_stream_t stream);

/* Number of kernels the last bn_block_forward / bn_block_backward call made by
 * this thread launched. */
int bn_last_launch_count(void);

/* Launch timing (for benchmarks; off by default). After bn_profile_start(),
 * every kernel the library launches from this thread is bracketed by two CUDA
 * events on its stream and recorded with its kind (0 tcgen05 GEMM, 1 fp32 GEMM,
 * 2 split-K reduction, 3 norm statistics, 4 weight fold, 5 RMSNorm backward,
 * 6 dw column sum, 7 elementwise, 8 attention core with epi 0 forward, 1 dK/dV,
 * 2 dQ, 3 row terms), its GEMM epilogue (or -1) and its
 * algorithmic FLOPs and bytes (each input read once, each output written once).
 * bn_profile_stop() ends recording, waits for the recorded events, copies up to
 * max_records records (device time in ms) into `out` (host memory) and returns
 * how many launches were recorded. The events keep each launch from overlapping
 * the one before it, so while recording the GEMM engine's consumers deal their
 * units in plain round robin (no lead rounds: no group of theirs starts late). */
typedef struct {
  int32_t kernel;
  int32_t epi;
  double flops;
  double bytes;
  float ms;
} bn_launch_record;

bn_status bn_profile_start(void);
int bn_profile_stop(bn_launch_record* out, int max_records);

/* Weight gradient without any caller-provided scratch: for callers that cannot
 * allocate GPU memory (their memory is reserved up front by their own pool, or
 * a cudaMalloc is forbidden or would synchronise where they run). The paper has
 * no counterpart; this is the weight-gradient GEMM of bn_block_backward
 * (dA = dz^T X, dB = dY^T h) offered on its own.
 *   dW[i, j] = colscale[j] * sum_{t < T} A[t, i] * B[t, j],  i < M, j < N
 * A [T, lda] and B [T, ldb] are row-major bf16 (token rows), dW [M, ldw] bf16;
 * colscale (bf16, N values) may be NULL; fp32 accumulation on the tensor cores.
 * Pointers 16-byte aligned, leading dimensions multiples of 8.
 * Scratch: a 32 MiB array inside the library (held on every GPU that loads
 * it until the process exits) holds the status word and the fp32 partial
 * tiles of the K split: at most one 128 x 256 tile per SM, whatever M, N and T
 * are (a GPU with more than 255 SMs returns BN_ERR_UNSUPPORTED). No device
 * memory is allocated. The first call on each
 * device looks the array's device address up (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. All calls
 * share the array, which keeps the last call's contents: calls whose kernels
 * overlap on the GPU (other streams, other threads) race and must be ordered
 * by the caller. Each call clears the array's status word first; a kernel whose
 * internal wait runs out (dW is then incomplete) records a time-out there, which
 * bn_weight_grad_noalloc_status() reports.
 * Asynchronous on `stream`; argument errors return before any launch; a failed
 * CUDA call returns BN_ERR_CUDA with its text in bn_last_cuda_error(). */
bn_status bn_weight_grad_noalloc(int64_t M, int64_t N, int64_t T, const void* A, int64_t lda,
                                 const void* B, int64_t ldb, const void* colscale, void* dW,
                                 int64_t ldw, bn_stream_t stream);

/* Status of the last bn_weight_grad_noalloc call on the current device, for the
 * same callers (the paper has no counterpart either): synchronises `stream`,
 * reads and clears the status word of the library's fixed array, and returns
 * BN_OK, or BN_ERR_TIMEOUT if that call's kernel gave up on a wait (its dW is
 * then incomplete), or BN_ERR_CUDA if the synchronisation failed. Allocates
 * nothing. */
bn_status bn_weight_grad_noalloc_status(bn_stream_t stream);

/* Name of a status code (static storage). */
const char* bn_status_string(bn_status s);

/* Text of the last CUDA error this library saw on this thread (static storage). */
const char* bn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* BOOSTBLK_H */
