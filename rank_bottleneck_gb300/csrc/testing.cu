// bn_testing_gemm: one launch of the GEMM engine, for unit tests of each
// epilogue and operand layout.
#include <cstdio>

#include "../../include/boostblk_testing.h"
#include "gemm.h"
#include "rowops.h"

using namespace bn;

extern "C" bn_status bn_testing_gemm(int32_t dtype, int32_t epi, int32_t sigma, int32_t S,
                                     float eps, int32_t allow_split, int32_t nprob,
                                     const bn_gemm_problem* probs, void* scratch,
                                     size_t scratch_bytes, bn_stream_t stream) {
  if (probs == nullptr || nprob < 1 || nprob > kMaxProblems || epi < 0 || epi > 7 || S < 1 || S > 16 ||
      (dtype != BN_F32 && dtype != BN_BF16) || scratch == nullptr || scratch_bytes < 256)
    return BN_ERR_INVALID_ARG;
  GemmLaunch g;
  g.epi = static_cast<Epi>(epi);
  g.sigma = sigma;
  g.S = S;
  g.eps = eps;
  g.allow_split = allow_split != 0;
  g.nprob = nprob;
  for (int i = 0; i < nprob; ++i) {
    const bn_gemm_problem& q = probs[i];
    GemmProblem& p = g.p[i];
    p.M = q.M;
    p.N = q.N;
    p.K = q.K;
    p.a[0].ptr = q.a;
    p.a[1].ptr = q.a2;
    p.b[0].ptr = q.b;
    p.b[1].ptr = q.b2;
    for (int j = 0; j < 2; ++j) {
      p.a[j].ld = q.lda;
      p.a[j].mn_major = q.a_mn_major != 0;
      p.b[j].ld = q.ldb;
      p.b[j].mn_major = q.b_mn_major != 0;
    }
    p.out[0] = q.out0;
    p.out[1] = q.out1;
    p.out[2] = q.out2;
    p.ldo[0] = p.ldo[1] = p.ldo[2] = q.ldo;
    p.in[0] = q.in0;
    p.in[1] = q.in1;
    p.ldi[0] = p.ldi[1] = q.ldi;
    p.rowv = q.rowv;
    p.colv = q.colv;
    if (q.M < 1 || q.N < 1 || q.K < 1) return BN_ERR_INVALID_ARG;
  }
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.status = static_cast<int*>(scratch);
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    c.num_sms = n;
  c.partial = reinterpret_cast<float*>(static_cast<char*>(scratch) + 256);
  c.partial_bytes = scratch_bytes - 256;
  if (dtype == BN_BF16)
    gemm_tc(c, g);
  else
    gemm_simt(c, g);
  if (c.bad) return BN_ERR_UNSUPPORTED;
  if (c.err != cudaSuccess) return BN_ERR_CUDA;
  return BN_OK;
}

extern "C" bn_status bn_testing_gemm_unfed(const bn_gemm_problem* prob, int* counters,
                                           void* scratch, size_t scratch_bytes,
                                           bn_stream_t stream) {
  if (prob == nullptr || counters == nullptr || scratch == nullptr || scratch_bytes < 256 ||
      prob->M < 1 || prob->M > 256 || prob->N < 1 || prob->K < 1)
    return BN_ERR_INVALID_ARG;
  GemmLaunch g;
  g.epi = EPI_STORE;
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = prob->M;
  p.N = prob->N;
  p.K = prob->K;
  p.a[0].ptr = prob->a;
  p.a[0].ld = prob->lda;
  p.a[0].mn_major = prob->a_mn_major != 0;
  p.b[0].ptr = prob->b;
  p.b[0].ld = prob->ldb;
  p.b[0].mn_major = prob->b_mn_major != 0;
  p.out[0] = prob->out0;
  p.ldo[0] = prob->ldo;
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.status = static_cast<int*>(scratch);
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    c.num_sms = n;
  // an upstream launch that never enters: entered counter and the one row block's
  c.chain_in.entered = counters;
  c.chain_in.rows = counters + 1;
  c.chain_in.entered_target = 1;
  c.chain_in.rows_target = 1;
  gemm_tc(c, g);
  if (c.bad) return BN_ERR_UNSUPPORTED;
  if (c.err != cudaSuccess) return BN_ERR_CUDA;
  return BN_OK;
}

extern "C" bn_status bn_testing_norm_bwd(int64_t rows, int64_t d, const void* dn, const void* x,
                                         const void* w, const float* rstd, const void* dres,
                                         void* dx, void* dw, float* part, int64_t part_elems,
                                         int32_t unfed, void* scratch, bn_stream_t stream) {
  if (rows < 1 || d < 8 || d % 8 != 0 || (unfed && d > 5120) || dn == nullptr || x == nullptr ||
      w == nullptr || rstd == nullptr || dres == nullptr || dx == nullptr || dw == nullptr ||
      part == nullptr || scratch == nullptr)
    return BN_ERR_INVALID_ARG;
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.status = static_cast<int*>(scratch);
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    c.num_sms = n;
  const int nblk = norm_bwd_blocks(c.num_sms);
  if (part_elems < static_cast<int64_t>(nblk) * d) return BN_ERR_INVALID_ARG;
  using bf = __nv_bfloat16;
  launch_norm_bwd<bf>(c, static_cast<const bf*>(dn), static_cast<const bf*>(x),
                      static_cast<const bf*>(w), rstd, static_cast<const bf*>(dres), rows, d,
                      static_cast<bf*>(dx), part, nblk, static_cast<bf*>(dw), true, unfed != 0);
  if (c.err != cudaSuccess) return BN_ERR_CUDA;
  return BN_OK;
}
