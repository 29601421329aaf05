// Internal interface between the block scheduler and the two GEMM engines
// (tcgen05 tensor cores for bf16, FFMA for fp32). Not part of the public ABI.
//
// Every GEMM computes, per problem, acc[i, j] = sum_k Aop[i, k] * Bop[j, k]
// for i < M, j < N, k < K, and hands acc to a fused epilogue.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace bn {

enum Epi : int {
  // out0 = acc * rowv[i] * colv[j]  (rowv fp32, colv element type; each optional).
  // With allow_split the tensor-core engine may cut the tiles left over after
  // whole rounds of CTA groups into K ranges, summed by a reduction kernel.
  EPI_STORE = 0,
  // out0 = z = acc; out1 = h = sigma(z), sigma evaluated on z as stored.
  EPI_SIGMA = 1,
  // Online RMSNorm over S emulated shards of K (see ONLINE NORM below), then as
  // EPI_SIGMA; out1 may be null (no sigma: the dense block). With rowv null: the
  // S shards' partial products are summed with no normalisation (a row-parallel
  // down-projection of bottleneck-aware tensor parallelism), then as EPI_SIGMA.
  EPI_NORM = 2,
  // out0 = in0 + acc (residual add).
  EPI_RESID = 3,
  // Two segments: G from (a[0], b[0]), U from (a[1], b[1]).
  // out0 = G, out1 = U (each optional), out2 = m = SiLU(G) * U (G, U as stored).
  EPI_SWIGLU = 4,
  // out0 = acc * sigma'(in0) * rowv[i]  (rowv optional): the bottleneck gradient dz.
  EPI_DSIGMA = 5,
  // dm = acc; in0 = G, in1 = U: out0 = dm U SiLU'(G) * rowv[i], out1 = dm SiLU(G) * rowv[i].
  EPI_DSWIGLU = 6,
  // Two segments accumulated into one sum (K split over two operand pairs), then as EPI_STORE.
  EPI_STORE_CHAIN = 7,
  // As EPI_DSIGMA, with K (the output dimension of the up-projection B) cut into S
  // emulated shards whose partial products are summed in the epilogue: the
  // r-wide all-reduce of bottleneck-aware tensor parallelism.
  EPI_SHARD_DSIGMA = 8,
};
// ONLINE NORM. rowv = ss [M, S] fp32 holds each row's sum of squares over each
// of S equal shards of K (the raw input, before the norm weight). For shard s:
//   rms_s = sqrt(ss_s / (K/S) + eps),  rms_g = sqrt(sum_s ss_s / K + eps)
//   L_s   = P_s / rms_s           (the shard's partial product, locally normalised)
//   z    += (rms_s / rms_g) * L_s (the per-row correction alpha = rms_s / rms_g)
// where P_s is the GEMM over shard s's K range. The norm weight is folded into
// the B operand by the caller.

struct Operand {
  const void* ptr = nullptr;
  int64_t ld = 0;         // elements between consecutive stored rows
  bool mn_major = false;  // false: stored [MN, K] (K contiguous); true: stored [K, MN]
};

struct GemmProblem {
  int64_t M = 0, N = 0, K = 0;
  int64_t K2 = 0;  // K of the second operand pair (SwiGLU, chain); 0 = the same K
  Operand a[2], b[2];
  void* out[3] = {nullptr, nullptr, nullptr};
  int64_t ldo[3] = {0, 0, 0};
  const void* in[2] = {nullptr, nullptr};
  int64_t ldi[2] = {0, 0};
  const float* rowv = nullptr;
  const void* colv = nullptr;
};

struct TileReduce;

struct GemmLaunch {
  Epi epi = EPI_STORE;
  int sigma = 0;      // bn_sigma
  int S = 1;          // shards of the online norm
  float eps = 1e-5f;
  bool allow_split = false;  // EPI_STORE only: K may be split (deterministic reduction)
  // tcgen05 engine: when set, the reduction of split tiles is described here
  // (rem_tiles = 0: none) for the caller to launch (launch_finish), not launched
  TileReduce* finish = nullptr;
  int nprob = 0;
  GemmProblem p[kMaxProblems];
};

struct Ctx {
  cudaStream_t stream = nullptr;
  int* status = nullptr;       // device status word
  int num_sms = 148;
  float* partial = nullptr;    // split-K workspace (fp32)
  size_t partial_bytes = 0;
  int launches = 0;
  // targets a consumer of the last tcgen05 launch waits for (ChainLink)
  int chain_entered_target = 0, chain_rows_target = 0;
  // that producer's units, CTA groups and estimated cost of one unit (lead
  // rounds of its consumer)
  int chain_prod_units = 0, chain_prod_groups = 0;
  double chain_prod_cost = 0;
  // links for the next tcgen05 launch (taken and cleared by it)
  ChainLink chain_out, chain_in;
  cudaError_t err = cudaSuccess;
  int bad = 0;                 // a bn_status other than BN_OK raised inside a launcher
};

// Kernel families, as reported by the launch-timing facility (bn_profile_*).
enum KernelKind : int {
  KK_GEMM_TC = 0,        // tcgen05 GEMM engine
  KK_GEMM_FFMA = 1,      // fp32 GEMM engine
  KK_SPLITK_REDUCE = 2,  // reduction of K-split tiles
  KK_STATS = 3,          // Online RMSNorm shard statistics
  KK_FOLD = 4,           // norm weight folded into a down-projection
  KK_NORM_BWD = 5,       // RMSNorm backward
  KK_COLSUM = 6,         // dw column reduction
  KK_ELEMENTWISE = 7,    // sigma recompute / SwiGLU / row scaling
  KK_ATTN = 8,           // attention core (epi: 0 forward, 1 dK/dV, 2 dQ, 3 row terms)
};

// Call right before a kernel launch: starts its timing record when the
// launch-timing facility is on for this thread.
void prof_start(Ctx& c);
// Whether this thread's launches are being timed one by one (bn_profile_start).
bool prof_active();
// Call right after a kernel launch: counts it, records a launch error, and
// closes its timing record with the launch's algorithmic FLOPs and bytes.
void note_launch(Ctx& c, int kind, int epi, double flops, double bytes);
// keep the first launch error of a sequence
inline void track(Ctx& c, cudaError_t e) {
  if (e != cudaSuccess && c.err == cudaSuccess) c.err = e;
}

// Algorithmic work of one GEMM launch: 2 M N K FLOPs per operand pair, every
// operand and epilogue input read once, every output written once.
inline void gemm_work(const GemmLaunch& g, int esize, double& flops, double& bytes) {
  flops = 0;
  bytes = 0;
  const int npair = (g.epi == EPI_SWIGLU || g.epi == EPI_STORE_CHAIN) ? 2 : 1;
  for (int i = 0; i < g.nprob; ++i) {
    const GemmProblem& p = g.p[i];
    const double M = static_cast<double>(p.M), N = static_cast<double>(p.N);
    for (int j = 0; j < npair; ++j) {
      const double K = static_cast<double>((j == 1 && p.K2 > 0) ? p.K2 : p.K);
      flops += 2.0 * M * N * K;
      bytes += (M + N) * K * esize;
    }
    for (int j = 0; j < 3; ++j)
      if (p.out[j]) bytes += M * N * esize;
    for (int j = 0; j < 2; ++j)
      if (p.in[j]) bytes += M * N * esize;
    if (p.rowv) bytes += M * 4.0 * (g.epi == EPI_NORM ? g.S : 1);
    if (p.colv) bytes += N * esize;
  }
}

// Keep the text of a failed CUDA call for bn_last_cuda_error (this thread) and
// return BN_ERR_CUDA (as an int: this header does not include the public ABI).
int record_cuda_error(cudaError_t e);

void gemm_tc(Ctx& c, const GemmLaunch& g);    // bf16 operands, tcgen05
void gemm_simt(Ctx& c, const GemmLaunch& g);  // fp32 operands, FFMA

// fp32 partial tiles gemm_tc may use (Ctx::partial) for a K split on a GPU with
// num_sms SMs; with less, it runs whole tiles only.
size_t gemm_tc_partial_bytes(int num_sms);

}  // namespace bn
