// fp32 GEMM engine on the FP32 pipes, for fp32 blocks (tf32 tensor cores would
// not meet fp32 accuracy). Same problem/epilogue contract as the tcgen05 engine:
// 64 x 64 output tiles, 16-deep K steps through shared memory, 4 x 4 outputs
// per thread, segments folded exactly as the tensor-core epilogues fold them.
//
// Each dot product is accumulated with the compensated scheme "Dot2" of Ogita,
// Rump and Oishi ("Accurate Sum and Dot Product", SIAM J. Sci. Comput. 2005):
// the rounding error of every product (recovered exactly with an FMA) and of
// every addition (recovered exactly with the TwoSum of Knuth) is summed into a
// second accumulator. The result is as accurate as if computed in twice the
// working precision and then rounded, so splitting K into the S shards of
// Online RMSNorm changes it only by the final roundings of the fold.
#include <algorithm>

#include "common.cuh"
#include "gemm.h"

namespace bn {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16, THREADS = 256;

struct Op {
  const float* p;
  int64_t s_mn, s_k;  // element (i, k) at p[i * s_mn + k * s_k]
};
struct Prob {
  Op a[2], b[2];
  int64_t M, N, K;
  int64_t K2;  // K of the second operand pair (SwiGLU, chain)
  float* out[3];
  int64_t ldo[3];
  const float* in[2];
  int64_t ldi[2];
  const float* rowv;
  const float* colv;
};
struct Params {
  Prob p[kMaxProblems];
  int S, sigma;
  float eps;
};

__device__ __forceinline__ void load_tile(float (*dst)[TM + 4], const Op& op, int64_t mn0,
                                          int64_t MN, int k0, int k_end) {
  const bool mn_fast = op.s_mn == 1;
  for (int e = threadIdx.x; e < TM * TK; e += THREADS) {
    int i, k;
    if (mn_fast) {
      k = e / TM;
      i = e % TM;
    } else {
      i = e / TK;
      k = e % TK;
    }
    const int64_t gi = mn0 + i;
    const int gk = k0 + k;
    dst[k][i] = (gi < MN && gk < k_end) ? op.p[gi * op.s_mn + static_cast<int64_t>(gk) * op.s_k] : 0.f;
  }
}

// s + c += a * b, with the product's and the sum's rounding errors kept in c.
__device__ __forceinline__ void dot2_step(float& s, float& c, float a, float b) {
  const float p = __fmul_rn(a, b);
  const float pe = __fmaf_rn(a, b, -p);        // a * b - p, exactly
  const float t = __fadd_rn(s, p);
  const float z = __fsub_rn(t, s);
  const float se = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(p, z));  // s + p - t, exactly
  s = t;
  c = __fadd_rn(c, __fadd_rn(se, pe));
}

template <int EK>
__global__ void __launch_bounds__(THREADS) simt_kernel(const __grid_constant__ Params P) {
  grid_dependency_sync();
  const Prob& pr = P.p[blockIdx.z];
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM, n0 = static_cast<int64_t>(blockIdx.x) * TN;
  if (m0 >= pr.M || n0 >= pr.N) return;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4], cmp[4][4], R[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = R[i][j] = 0.f;

  constexpr bool kFold = EK == EPI_NORM || EK == EPI_SHARD_DSIGMA;  // shard-summed kinds
  const int nseg = kFold ? P.S : (EK == EPI_SWIGLU || EK == EPI_STORE_CHAIN) ? 2 : 1;
  for (int s = 0; s < nseg; ++s) {
    const int pair = (EK == EPI_SWIGLU || EK == EPI_STORE_CHAIN) ? s : 0;
    int k_lo = 0, k_hi = static_cast<int>(pair == 1 ? pr.K2 : pr.K);
    if (kFold) {  // emulated shard s of K
      k_lo = static_cast<int>(s * pr.K / P.S);
      k_hi = static_cast<int>((s + 1) * pr.K / P.S);
    }
    if (!(EK == EPI_STORE_CHAIN && s == 1)) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = 0.f;
    }
    for (int k0 = k_lo; k0 < k_hi; k0 += TK) {
      load_tile(As, pr.a[pair], m0, pr.M, k0, k_hi);
      load_tile(Bs, pr.b[pair], n0, pr.N, k0, k_hi);
      __syncthreads();
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[k][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[k][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) dot2_step(acc[i][j], cmp[i][j], av[i], bv[j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[i][j] = __fadd_rn(acc[i][j], cmp[i][j]);
        cmp[i][j] = 0.f;
      }
    if (EK == EPI_NORM && pr.rowv != nullptr) {
      // Online RMSNorm: local normalisation, then the per-row correction alpha
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = m0 + ty * 4 + i;
        float tot = 0.f, ss_s = 0.f;
        if (row < pr.M) {
          for (int t = 0; t < P.S; ++t) tot += pr.rowv[row * P.S + t];
          ss_s = pr.rowv[row * P.S + s];
        }
        const float shard_w = static_cast<float>(pr.K / P.S);
        const float rms_g = sqrtf(tot / static_cast<float>(pr.K) + P.eps);
        const float rms_s = sqrtf(ss_s / shard_w + P.eps);
        const float inv_local = 1.0f / rms_s;
        const float alpha = rms_s / rms_g;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float local = acc[i][j] * inv_local;
          R[i][j] = (s == 0) ? alpha * local : fmaf(alpha, local, R[i][j]);
        }
      }
    } else if (kFold) {
      // the shards' partial products summed in shard order (emulated all-reduce)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) R[i][j] = (s == 0) ? acc[i][j] : __fadd_rn(R[i][j], acc[i][j]);
    } else if (EK == EPI_SWIGLU && s == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) R[i][j] = acc[i][j];
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = m0 + ty * 4 + i;
    if (row >= pr.M) continue;
    const float rs = (pr.rowv != nullptr && EK != EPI_NORM) ? pr.rowv[row] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t col = n0 + tx * 4 + j;
      if (col >= pr.N) continue;
      const float v = acc[i][j];
      if (EK == EPI_STORE || EK == EPI_STORE_CHAIN) {
        float o = v;
        if (pr.colv != nullptr) o *= pr.colv[col];
        if (pr.rowv != nullptr) o *= rs;
        pr.out[0][row * pr.ldo[0] + col] = o;
      } else if (EK == EPI_SIGMA || EK == EPI_NORM) {
        const float z = (EK == EPI_NORM) ? R[i][j] : v;
        pr.out[0][row * pr.ldo[0] + col] = z;
        if (pr.out[1] != nullptr) pr.out[1][row * pr.ldo[1] + col] = act_f(z, P.sigma);
      } else if (EK == EPI_RESID) {
        pr.out[0][row * pr.ldo[0] + col] = pr.in[0][row * pr.ldi[0] + col] + v;
      } else if (EK == EPI_SWIGLU) {
        const float G = R[i][j], U = v;
        if (pr.out[0] != nullptr) pr.out[0][row * pr.ldo[0] + col] = G;
        if (pr.out[1] != nullptr) pr.out[1][row * pr.ldo[1] + col] = U;
        pr.out[2][row * pr.ldo[2] + col] = __fmul_rn(silu_f(G), U);
      } else if (EK == EPI_DSIGMA || EK == EPI_SHARD_DSIGMA) {
        const float z = pr.in[0][row * pr.ldi[0] + col];
        const float dh = (EK == EPI_SHARD_DSIGMA) ? R[i][j] : v;
        pr.out[0][row * pr.ldo[0] + col] = (dh * act_grad_f(z, P.sigma)) * rs;
      } else if (EK == EPI_DSWIGLU) {
        const float G = pr.in[0][row * pr.ldi[0] + col];
        const float U = pr.in[1][row * pr.ldi[1] + col];
        pr.out[0][row * pr.ldo[0] + col] = ((v * U) * silu_grad_f(G)) * rs;
        pr.out[1][row * pr.ldo[1] + col] = (v * silu_f(G)) * rs;
      }
    }
  }
}

static Op make_op(const Operand& o) {
  Op r;
  r.p = static_cast<const float*>(o.ptr);
  if (o.mn_major) {
    r.s_mn = 1;
    r.s_k = o.ld;
  } else {
    r.s_mn = o.ld;
    r.s_k = 1;
  }
  return r;
}

template <int EK>
static cudaError_t go(const Params& P, dim3 grid, cudaStream_t s) {
  return launch_pdl(simt_kernel<EK>, grid, THREADS, 0, s, P);
}

}  // namespace simt

void gemm_simt(Ctx& c, const GemmLaunch& g) {
  using namespace simt;
  Params P{};
  P.S = g.S;
  P.sigma = g.sigma;
  P.eps = g.eps;
  int64_t gm = 0, gn = 0;
  for (int i = 0; i < g.nprob; ++i) {
    const GemmProblem& q = g.p[i];
    Prob& p = P.p[i];
    for (int j = 0; j < 2; ++j) {
      p.a[j] = make_op(q.a[j]);
      p.b[j] = make_op(q.b[j]);
    }
    p.M = q.M;
    p.N = q.N;
    p.K = q.K;
    p.K2 = q.K2 > 0 ? q.K2 : q.K;
    for (int j = 0; j < 3; ++j) {
      p.out[j] = static_cast<float*>(q.out[j]);
      p.ldo[j] = q.ldo[j];
    }
    for (int j = 0; j < 2; ++j) {
      p.in[j] = static_cast<const float*>(q.in[j]);
      p.ldi[j] = q.ldi[j];
    }
    p.rowv = q.rowv;
    p.colv = static_cast<const float*>(q.colv);
    gm = std::max(gm, (q.M + TM - 1) / TM);
    gn = std::max(gn, (q.N + TN - 1) / TN);
  }
  dim3 grid(static_cast<unsigned>(gn), static_cast<unsigned>(gm), static_cast<unsigned>(g.nprob));
  double flops, bytes;
  gemm_work(g, 4, flops, bytes);
  prof_start(c);
  switch (g.epi) {
    case EPI_STORE: track(c, go<EPI_STORE>(P, grid, c.stream)); break;
    case EPI_SIGMA: track(c, go<EPI_SIGMA>(P, grid, c.stream)); break;
    case EPI_NORM: track(c, go<EPI_NORM>(P, grid, c.stream)); break;
    case EPI_RESID: track(c, go<EPI_RESID>(P, grid, c.stream)); break;
    case EPI_SWIGLU: track(c, go<EPI_SWIGLU>(P, grid, c.stream)); break;
    case EPI_DSIGMA: track(c, go<EPI_DSIGMA>(P, grid, c.stream)); break;
    case EPI_DSWIGLU: track(c, go<EPI_DSWIGLU>(P, grid, c.stream)); break;
    case EPI_STORE_CHAIN: track(c, go<EPI_STORE_CHAIN>(P, grid, c.stream)); break;
    case EPI_SHARD_DSIGMA: track(c, go<EPI_SHARD_DSIGMA>(P, grid, c.stream)); break;
  }
  note_launch(c, KK_GEMM_FFMA, static_cast<int>(g.epi), flops, bytes);
}

}  // namespace bn
