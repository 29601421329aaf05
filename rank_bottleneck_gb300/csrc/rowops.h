// Launchers of the row-wise (HBM-bound) kernels of the block.
#pragma once

#include <cuda_bf16.h>
#include "gemm.h"

namespace bn {

// ss[t, s] = sum of x[t, j]^2 over shard s (S equal column shards of d);
// rstd[t] = 1 / sqrt(sum_s ss[t, s] / d + eps). x is [rows, d], row stride d.
template <typename T>
void launch_stats(Ctx& c, const T* x, int64_t rows, int64_t d, int S, float eps, float* ss,
                  float* rstd);

// out[j, k] = A[j, k] * w[k] for j < rows, k < cols (row stride cols): a norm
// weight folded into a down-projection. A null A is no job.
template <typename T>
struct FoldJob {
  const T* A = nullptr;
  const T* w = nullptr;
  int64_t rows = 0, cols = 0;
  T* out = nullptr;
};

// launch_stats and, in the same launch, up to two weight folds.
template <typename T>
void launch_stats_fold(Ctx& c, const T* x, int64_t rows, int64_t d, int S, float eps, float* ss,
                       float* rstd, const FoldJob<T>& f0, const FoldJob<T>& f1);

// RMSNorm backward from dn' = rstd * dn (the gradient of the normalised input
// times the row's 1/rms):
//   dx[t, j] = dres[t, j] + dn'[t, j] w[j] - x[t, j] rstd[t]^2 sum_k(dn' w x)[t, k] / d
//   dw[j]    = sum_t dn'[t, j] x[t, j]
// dw is reduced deterministically through `part` (nblk x d fp32): in a second
// launch when `colsum`, else by the caller (launch_finish). Returns the rows of
// `part` written (at most nblk). `unfed` (a test hook, bf16 rows of at most
// 5120 columns) never loads the first row of the first warp, so that its
// bounded wait runs out and the kernel records a timeout.
template <typename T>
int launch_norm_bwd(Ctx& c, const T* dn, const T* x, const T* w, const float* rstd,
                    const T* dres, int64_t rows, int64_t d, T* dx, float* part, int nblk, T* dw,
                    bool colsum, bool unfed = false);
int norm_bwd_blocks(int num_sms);

// End of a bf16 backward, one launch: the reduction of the GEMM's split tiles
// and the RMSNorm dw column sums.
// Tiles [0, full_units) of the GEMM launch were whole; tile full_units + t
// (t < rem_tiles) was cut into rem_split k-ranges whose fp32 partial tiles sit
// in slots rem_split t + s, each [tile_rows][BN]. For those tiles
// out[i, j] = colv[j] * sum_s partial_s[i, j] (fixed order over s, bf16
// output, colv optional), clipped to the problem's M x N.
// Column-sum job j: out[col] = sum_b part[b][col] over nblk rows of d columns
// (what launch_norm_bwd leaves in `part` when it is told not to sum it).
struct TileReduceProb {
  int64_t M, N;
  int tiles_n, tile_begin;
  const __nv_bfloat16* colv;
  __nv_bfloat16* out;
  int64_t ldo;
};
struct ColsumJob {
  const float* part = nullptr;
  int nblk = 0, d = 0;
  __nv_bfloat16* out = nullptr;
};
struct TileReduce {
  TileReduceProb p[kMaxProblems];
  int nprob = 0;
  int full_units = 0, rem_split = 0, rem_tiles = 0, tile_rows = 0, BN = 0;
  const float* part = nullptr;
  ColsumJob col[2];
  int ncol = 0;
};
void launch_finish(Ctx& c, const TileReduce& r);

// Zero the counters of a pass's chained launches (one small launch). `early`
// must belong to launches that completed before the kernel ahead of this one
// started its dependency wait: it is cleared at once, overlapping that kernel's
// tail. `late` may still be read by the kernel ahead and is cleared after the
// dependency wait. The launch completes only after the kernel ahead.
void launch_zero_counters(Ctx& c, int* early, int64_t n_early, int* late, int64_t n_late);

// h = sigma(z) elementwise, rounded exactly like the GEMM epilogues round it.
template <typename T>
void launch_sigma(Ctx& c, const T* z, int64_t rows, int64_t cols, int64_t ldz, T* h, int64_t ldh,
                  int sigma);

// m = SiLU(G) * U elementwise.
template <typename T>
void launch_swiglu(Ctx& c, const T* G, const T* U, int64_t rows, int64_t cols, int64_t ld, T* m,
                   int64_t ldm);

// out[i, j] = in[i, j] * rowv[i]; in == nullptr writes zeros.
template <typename T>
void launch_rowscale(Ctx& c, const T* in, int64_t ldi, const float* rowv, int64_t rows,
                     int64_t cols, T* out, int64_t ldo);

}  // namespace bn
