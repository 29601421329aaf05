// Block scheduler and C ABI: validates a bn_block_desc, lays out the caller's
// `saved` / `scratch` buffers, and issues the forward / backward kernel
// sequence of one low-rank (or dense) decoder block on the caller's stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/boostblk.h"
#include "common.cuh"
#include "attn.h"
#include "gemm.h"
#include "rowops.h"

namespace bn {

thread_local char g_cuda_err[256] = "no error";

int record_cuda_error(cudaError_t e) {
  std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s", cudaGetErrorString(e));
  return BN_ERR_CUDA;
}

namespace {

using bf16 = __nv_bfloat16;

thread_local int g_last_launches = 0;

// the factorised layers, in the order of bn_block_desc.r_layer
enum Layer : int { LQ = 0, LK, LV, LO, LG, LU, LD };

struct Shape {
  int64_t T, d, r, d_ff, ld_ff;
  int64_t rl[7];        // each factorised layer's rank (bottlenecks of uneven size)
  int64_t rqkv, rgu;    // widths of the grouped Q/K/V and gate/up bottlenecks
  int64_t off[3];       // column offsets of the Q, K, V slices in the grouped tensors
  int64_t ld_act;  // row stride of the [T, d_ff] activations G, U, m, dG, dU: whole 128-byte lines
  int S, sigma, dtype, kind, dense, ckpt, btp;
  int attn;        // the attention core runs inside the block (H heads of 128, sequences of L)
  int64_t L, H;
  float eps;
  int64_t E;  // bytes per element
  bool full() const { return kind == BN_BLOCK_FULL; }
};

// activations written by the forward and read by the backward
struct Acts {
  float *ss1 = nullptr, *rstd1 = nullptr, *ss2 = nullptr, *rstd2 = nullptr;
  void *z_qkv = nullptr, *h_qkv = nullptr, *V = nullptr, *z_o = nullptr, *h_o = nullptr;
  void *x1 = nullptr, *z_gu = nullptr, *h_gu = nullptr, *G = nullptr, *U = nullptr, *m = nullptr;
  void *z_d = nullptr, *h_d = nullptr;
  void *Q = nullptr, *K = nullptr, *O = nullptr;  // attention core: its inputs and output
  float* lse = nullptr;                            // and its row log-sum-exp
};
// temporaries in `scratch`
struct Tmp {
  int* status = nullptr;
  void *A1f = nullptr, *A2f = nullptr;  // down-projections with the norm weight folded in
  void *dz_d = nullptr, *dG = nullptr, *dU = nullptr, *dz_gu = nullptr, *dn = nullptr;
  void *dx1 = nullptr, *dz_o = nullptr, *dV = nullptr, *dz_qkv = nullptr, *dqkv = nullptr;
  float *dw_part1 = nullptr, *dw_part2 = nullptr;  // RMSNorm dw partial column sums
  void *dO = nullptr, *dQ = nullptr, *dK = nullptr;  // attention core gradients
  float* attn_rows = nullptr;                        // and its backward's row terms
  float* partial = nullptr;
  size_t partial_bytes = 0;
  int nblk = 0;
  int* chain = nullptr;  // counters of the chained launches (ChainLink), kChainLinks links
};

// Chained launch pairs: an r-wide GEMM (the producer, whose tile count leaves
// part of the GPU idle in its last round) and the up-projection that reads its
// output. Links 0..3 are the forward's, 4..7 the backward's.
constexpr int kChainLinks = 8;
int64_t chain_stride(const Shape& s) { return 32 + (s.T + 127) / 128 / 32 * 32 + 32; }

struct Bump {
  char* base;
  size_t off = 0;
  explicit Bump(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~static_cast<size_t>(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

int device_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// the attention core's shapes: T / L causal sequences of L tokens, d / 128 heads
bn_attn_desc attn_desc(const Shape& s) {
  bn_attn_desc a;
  a.B = s.L > 0 ? s.T / s.L : 0;
  a.L = s.L;
  a.H = s.H;
  a.d_head = 128;
  a.causal = 1;
  return a;
}

void plan(const Shape& s, void* saved_base, void* scratch_base, Acts& A, Tmp& B,
          size_t* saved_bytes, size_t* scratch_bytes) {
  Bump sv(saved_base), sc(scratch_base);
  const int64_t T = s.T, E = s.E;
  B.status = static_cast<int*>(sc.take(256));
  // in checkpoint mode only the pre-activations go to `saved`
  Bump& keep = sv;
  Bump& rest = s.ckpt ? sc : sv;
  if (s.full()) {
    A.ss1 = static_cast<float*>(rest.take(T * s.S * 4));
    A.rstd1 = static_cast<float*>(rest.take(T * 4));
    if (!s.dense) {
      A.z_qkv = keep.take(T * s.rqkv * E);
      A.h_qkv = rest.take(T * s.rqkv * E);
      A.z_o = keep.take(T * s.rl[LO] * E);
      A.h_o = rest.take(T * s.rl[LO] * E);
    }
    A.V = rest.take(T * s.d * E);
    A.x1 = rest.take(T * s.d * E);
    if (s.attn) {
      A.Q = rest.take(T * s.d * E);
      A.K = rest.take(T * s.d * E);
      A.O = rest.take(T * s.d * E);
      const bn_attn_desc a = attn_desc(s);
      A.lse = static_cast<float*>(rest.take(static_cast<size_t>(a.B * a.H * bn_attn_lse_stride(a.L)) * 4));
    }
  }
  A.ss2 = static_cast<float*>(rest.take(T * s.S * 4));
  A.rstd2 = static_cast<float*>(rest.take(T * 4));
  if (!s.dense) {
    A.z_gu = keep.take(T * s.rgu * E);
    A.h_gu = rest.take(T * s.rgu * E);
    A.z_d = keep.take(T * s.rl[LD] * E);
    A.h_d = rest.take(T * s.rl[LD] * E);
  }
  A.G = rest.take(T * s.ld_act * E);
  A.U = rest.take(T * s.ld_act * E);
  A.m = rest.take(T * s.ld_act * E);

  const int64_t n1 = s.dense ? 3 * s.d : s.rqkv, n2 = s.dense ? 2 * s.d_ff : s.rgu;
  if (s.full()) B.A1f = sc.take(n1 * s.d * E);
  B.A2f = sc.take(n2 * s.d * E);
  if (!s.dense) {
    B.dz_d = sc.take(T * s.rl[LD] * E);
    B.dz_gu = sc.take(T * s.rgu * E);
  }
  B.dG = sc.take(T * s.ld_act * E);
  B.dU = sc.take(T * s.ld_act * E);
  B.dn = sc.take(T * s.d * E);
  if (s.full()) {
    B.dx1 = sc.take(T * s.d * E);
    if (s.dense) {
      B.dqkv = sc.take(T * 3 * s.d * E);
    } else {
      B.dz_o = sc.take(T * s.rl[LO] * E);
      B.dV = sc.take(T * s.d * E);
      B.dz_qkv = sc.take(T * s.rqkv * E);
    }
  }
  if (s.attn) {
    B.dO = sc.take(T * s.d * E);
    B.dQ = sc.take(T * s.d * E);
    B.dK = sc.take(T * s.d * E);
    if (s.dense) B.dV = sc.take(T * s.d * E);
    B.attn_rows = static_cast<float*>(sc.take(attn_scratch_floats(attn_desc(s)) * 4));
  }
  B.nblk = norm_bwd_blocks(device_sms());
  B.dw_part2 = static_cast<float*>(sc.take(static_cast<size_t>(B.nblk) * s.d * 4));
  if (s.full()) B.dw_part1 = static_cast<float*>(sc.take(static_cast<size_t>(B.nblk) * s.d * 4));
  if (s.dtype == BN_BF16) {
    B.partial_bytes = gemm_tc_partial_bytes(device_sms());
    B.partial = static_cast<float*>(sc.take(B.partial_bytes));
    B.chain = static_cast<int*>(sc.take(kChainLinks * chain_stride(s) * 4));
  }
  if (saved_bytes) *saved_bytes = sv.off;
  if (scratch_bytes) *scratch_bytes = sc.off;
}

bn_status check_desc(const bn_block_desc* D, Shape& s) {
  if (D == nullptr) return BN_ERR_INVALID_ARG;
  s.T = D->T;
  s.d = D->d;
  s.r = D->r;
  s.d_ff = D->d_ff;
  s.ld_ff = D->ld_ff;
  s.ld_act = (s.d_ff + 63) / 64 * 64;
  s.S = D->S;
  s.sigma = D->sigma;
  s.dtype = D->dtype;
  s.kind = D->kind;
  s.dense = D->dense;
  s.ckpt = D->checkpoint;
  s.eps = D->eps;
  s.btp = D->btp;
  s.attn = D->attn;
  s.L = D->seq_len;
  s.H = s.d / 128;
  if (s.dtype != BN_F32 && s.dtype != BN_BF16) return BN_ERR_INVALID_ARG;
  if (s.sigma != BN_SIGMA_IDENTITY && s.sigma != BN_SIGMA_SILU) return BN_ERR_INVALID_ARG;
  if (s.kind != BN_BLOCK_FULL && s.kind != BN_BLOCK_MLP) return BN_ERR_INVALID_ARG;
  if ((s.dense != 0 && s.dense != 1) || (s.ckpt != 0 && s.ckpt != 1) || (s.btp != 0 && s.btp != 1) ||
      (s.attn != 0 && s.attn != 1))
    return BN_ERR_INVALID_ARG;
  if (s.attn) {
    // the attention core: full kind, bf16, heads of 128, whole sequences
    if (s.kind != BN_BLOCK_FULL || s.L < 1 || s.T % s.L != 0) return BN_ERR_INVALID_ARG;
    if (s.dtype != BN_BF16 || s.d % 128 != 0) return BN_ERR_UNSUPPORTED;
    const bn_status a = attn_check(attn_desc(s));
    if (a != BN_OK) return a;
  }
  if (s.T < 1 || s.d < 1 || s.d_ff < 1 || s.ld_ff < s.d_ff || s.S < 1 || s.S > 16)
    return BN_ERR_INVALID_ARG;
  if (!(s.eps >= 0.f) || s.eps > 1.f) return BN_ERR_INVALID_ARG;
  // per-layer ranks: 0 = r; the dense block has no ranks
  for (int i = 0; i < 7; ++i) {
    const int64_t ri = D->r_layer[i];
    if (ri < 0 || (s.dense && ri != 0)) return BN_ERR_INVALID_ARG;
    s.rl[i] = ri > 0 ? ri : s.r;
  }
  if (!s.dense)
    for (int i = 0; i < 7; ++i)
      if (s.rl[i] < 1) return BN_ERR_INVALID_ARG;
  // the RMSNorm backward keeps at least one row of d fp32 column sums in shared memory
  if (s.T > (int64_t(1) << 31) - 256 || s.d > 43688 || s.ld_ff > (int64_t(1) << 22))
    return BN_ERR_UNSUPPORTED;
  if (!s.dense)
    for (int i = 0; i < 7; ++i)
      if (s.rl[i] > (int64_t(1) << 20)) return BN_ERR_UNSUPPORTED;
  if (s.d % s.S != 0 || (s.d / s.S) % 8 != 0) return BN_ERR_INVALID_ARG;
  if (s.ld_ff % 8 != 0) return BN_ERR_ALIGNMENT;
  if (!s.dense)
    for (int i = 0; i < 7; ++i)
      if (s.rl[i] % 8 != 0) return BN_ERR_ALIGNMENT;
  s.rqkv = s.rl[LQ] + s.rl[LK] + s.rl[LV];
  s.rgu = s.rl[LG] + s.rl[LU];
  s.off[0] = 0;
  s.off[1] = s.rl[LQ];
  s.off[2] = s.rl[LQ] + s.rl[LK];
  if (s.dense && s.ckpt) return BN_ERR_UNSUPPORTED;
  // tensor-parallel emulation of the factorised block; each shard of d_ff gets
  // at least one 64-column block
  if (s.btp && (s.dense || (s.d_ff + 63) / 64 < s.S)) return BN_ERR_UNSUPPORTED;
  if (s.dtype == BN_BF16 && (s.d / s.S) % 64 != 0) return BN_ERR_UNSUPPORTED;
  s.E = (s.dtype == BN_BF16) ? 2 : 4;
  return BN_OK;
}

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Every pointer that must be present is non-null and aligned; every pointer
// that must be absent is null.
bn_status check_params(const Shape& s, const bn_block_params* W) {
  if (W == nullptr) return BN_ERR_INVALID_ARG;
  const bool f = s.full(), lr = !s.dense;
  const void* need[] = {W->w_norm2, W->A_gu, W->A_d};
  for (const void* p : need)
    if (p == nullptr) return BN_ERR_INVALID_ARG;
  struct Item { const void* p; bool required; };
  const Item items[] = {{W->w_norm1, f},        {W->A_qkv, f},        {W->B_q, f && lr},
                        {W->B_k, f && lr},      {W->B_v, f && lr},    {W->A_o, f},
                        {W->B_o, f && lr},      {W->w_norm2, true},   {W->A_gu, true},
                        {W->B_g, lr},           {W->B_u, lr},         {W->A_d, true},
                        {W->B_d, lr}};
  for (const Item& it : items) {
    if (it.required && it.p == nullptr) return BN_ERR_INVALID_ARG;
    if (!it.required && it.p != nullptr) return BN_ERR_INVALID_ARG;
    if (it.p != nullptr && !aligned(it.p)) return BN_ERR_ALIGNMENT;
  }
  return BN_OK;
}

// ---------------------------------------------------------------------------
// launch helpers
// ---------------------------------------------------------------------------
Operand op(const void* p, int64_t ld, bool mn_major) {
  Operand o;
  o.ptr = p;
  o.ld = ld;
  o.mn_major = mn_major;
  return o;
}
constexpr bool KM = false, MN = true;

const void* at(const void* p, int64_t elems, const Shape& s) {
  return p ? static_cast<const char*>(p) + elems * s.E : nullptr;
}
void* at(void* p, int64_t elems, const Shape& s) {
  return p ? static_cast<char*>(p) + elems * s.E : nullptr;
}

void gemm(Ctx& c, const Shape& s, const GemmLaunch& g) {
  if (s.dtype == BN_BF16) {
    gemm_tc(c, g);
  } else {
    c.chain_out = ChainLink{};
    c.chain_in = ChainLink{};
    gemm_simt(c, g);
  }
}

// Chained launches (ChainLink). BN_GEMM_CHAIN=0 in the environment turns them off.
bool chains_on(const Shape& s, const Tmp& B) {
  static const bool off = [] {
    const char* v = std::getenv("BN_GEMM_CHAIN");
    return v != nullptr && v[0] == '0';
  }();
  return !off && s.dtype == BN_BF16 && B.chain != nullptr;
}
ChainLink chain_link(const Shape& s, const Tmp& B, int i) {
  ChainLink l;
  l.entered = B.chain + i * chain_stride(s);
  l.rows = l.entered + 32;
  return l;
}
// zero links [first, first + n) before the launches that use them; the last
// n_late of them after the kernel ahead has completed (it may be the consumer
// of one of them, still reading its counters: the previous forward's last
// launch is link 3's consumer), the others at once
void chain_reset(Ctx& c, const Shape& s, const Tmp& B, int first, int n, int n_late) {
  if (!chains_on(s, B)) return;
  const int64_t st = chain_stride(s);
  launch_zero_counters(c, B.chain + first * st, (n - n_late) * st, B.chain + (first + n - n_late) * st,
                       n_late * st);
}
// the next GEMM launch produces rows for link i
void produce(Ctx& c, const Shape& s, const Tmp& B, int i) {
  if (chains_on(s, B)) c.chain_out = chain_link(s, B, i);
}
// the next GEMM launch consumes link i, filled by the launch just before it
void consume(Ctx& c, const Shape& s, const Tmp& B, int i) {
  if (!chains_on(s, B) || c.chain_rows_target <= 0) return;
  ChainLink l = chain_link(s, B, i);
  l.entered_target = c.chain_entered_target;
  l.rows_target = c.chain_rows_target;
  c.chain_in = l;
}

GemmLaunch launch(Epi e, const Shape& s) {
  GemmLaunch g;
  g.epi = e;
  g.sigma = s.sigma;
  g.S = s.S;
  g.eps = s.eps;
  return g;
}

// weight gradient: out[M, N] = colv[j] * sum_t Aop[t, i] Bop[t, j]
GemmProblem wgrad(int64_t M, int64_t N, int64_t T, const void* a, int64_t lda, const void* b,
                  int64_t ldb, void* out, int64_t ldo, const void* colv = nullptr) {
  GemmProblem p;
  p.M = M;
  p.N = N;
  p.K = T;
  p.a[0] = op(a, lda, MN);
  p.b[0] = op(b, ldb, MN);
  p.out[0] = out;
  p.ldo[0] = ldo;
  p.colv = colv;
  return p;
}

// The weight gradients of a backward pass, gathered and launched together at its
// end: they read only tensors the backward has already written (nothing later
// overwrites them), and one launch over all their tiles fills whole rounds of
// the CTA groups, with only the last few tiles split along K.
// The RMSNorm dw column sums of a bf16 backward go out in the same final
// launch as the reduction of the weight-gradient GEMM's split tiles.
struct Wgrads {
  GemmProblem p[kMaxProblems];
  int n = 0;
  ColsumJob col[2];
  int ncol = 0;
};
void flush_wgrads(Ctx& c, const Shape& s, Wgrads& w, bool final = false);
void add_wgrad(Ctx& c, const Shape& s, Wgrads& w, const GemmProblem& q) {
  if (w.n == kMaxProblems) flush_wgrads(c, s, w);
  w.p[w.n++] = q;
}

#define DT_CALL(s, FN, ...)                                          \
  do {                                                               \
    if ((s).dtype == BN_BF16)                                        \
      FN<bf16>(__VA_ARGS__);                                         \
    else                                                             \
      FN<float>(__VA_ARGS__);                                        \
  } while (0)

template <typename T>
void stats(Ctx& c, const void* x, const Shape& s, float* ss, float* rstd) {
  launch_stats<T>(c, static_cast<const T*>(x), s.T, s.d, s.S, s.eps, ss, rstd);
}
// a norm weight folded into a down-projection: out = A diag(w), A [rows, cols]
struct Fold {
  const void* A = nullptr;
  const void* w = nullptr;
  int64_t rows = 0, cols = 0;
  void* out = nullptr;
};
// stats(x) and up to two weight folds in one launch
template <typename T>
void stats_fold(Ctx& c, const void* x, const Shape& s, float* ss, float* rstd, const Fold& a,
                const Fold& b) {
  auto job = [](const Fold& f) {
    FoldJob<T> j;
    j.A = static_cast<const T*>(f.A);
    j.w = static_cast<const T*>(f.w);
    j.rows = f.rows;
    j.cols = f.cols;
    j.out = static_cast<T*>(f.out);
    return j;
  };
  launch_stats_fold<T>(c, static_cast<const T*>(x), s.T, s.d, s.S, s.eps, ss, rstd, job(a), job(b));
}
// RMSNorm backward; `part` holds its dw partial sums until they are summed
// (bf16: in the backward's final launch, see Wgrads)
template <typename T>
void normbwd(Ctx& c, const Shape& s, const Tmp& B, Wgrads& wg, float* part, const void* dn,
             const void* x, const void* w, const float* rstd, const void* dres, void* dx,
             void* dw) {
  const bool defer = s.dtype == BN_BF16;
  const int rows_written = launch_norm_bwd<T>(
      c, static_cast<const T*>(dn), static_cast<const T*>(x), static_cast<const T*>(w), rstd,
      static_cast<const T*>(dres), s.T, s.d, static_cast<T*>(dx), part, B.nblk,
      static_cast<T*>(dw), !defer);
  if (defer) {
    ColsumJob& j = wg.col[wg.ncol++];
    j.part = part;
    j.nblk = rows_written;
    j.d = static_cast<int>(s.d);
    j.out = static_cast<bf16*>(dw);
  }
}
template <typename T>
void sigma_ew(Ctx& c, const Shape& s, const void* z, int64_t cols, int64_t ld, void* h) {
  launch_sigma<T>(c, static_cast<const T*>(z), s.T, cols, ld, static_cast<T*>(h), ld, s.sigma);
}
template <typename T>
void swiglu_ew(Ctx& c, const Shape& s, const void* G, const void* U, void* m) {
  launch_swiglu<T>(c, static_cast<const T*>(G), static_cast<const T*>(U), s.T, s.d_ff, s.ld_act,
                   static_cast<T*>(m), s.ld_act);
}
template <typename T>
void rowscale(Ctx& c, const Shape& s, const void* in, int64_t ldi, const float* rowv, int64_t cols,
              void* out, int64_t ldo) {
  launch_rowscale<T>(c, static_cast<const T*>(in), ldi, rowv, s.T, cols, static_cast<T*>(out), ldo);
}

void zero2d(Ctx& c, void* p, int64_t ld_bytes, int64_t width_bytes, int64_t rows) {
  cudaError_t e = cudaMemset2DAsync(p, ld_bytes, 0, width_bytes, rows, c.stream);
  if (e != cudaSuccess && c.err == cudaSuccess) c.err = e;
}

bn_status finish(Ctx& c) {
  g_last_launches = c.launches;
  if (c.bad) return BN_ERR_UNSUPPORTED;
  if (c.err != cudaSuccess) return static_cast<bn_status>(record_cuda_error(c.err));
  return BN_OK;
}

// ---------------------------------------------------------------------------
// forward pieces (shared by the forward and the checkpoint recompute)
// ---------------------------------------------------------------------------

// O = causal softmax attention of (Q, K, V), and its row log-sum-exp
void attention(Ctx& c, const Shape& s, const Acts& A, const Tmp& B) {
  track(c, attn_forward(c, attn_desc(s), A.Q, A.K, A.V, A.O, A.lse, B.status));
}

// V (and Q, K when wanted) = sigma(z) B^T for the grouped Q/K/V bottlenecks.
void qkv_up(Ctx& c, const Shape& s, const bn_block_params* W, const Acts& A, void* q, void* k) {
  GemmLaunch g = launch(EPI_STORE, s);
  const void* Bs[3] = {W->B_q, W->B_k, W->B_v};
  void* outs[3] = {q, k, A.V};
  for (int i = 0; i < 3; ++i) {
    if (outs[i] == nullptr) continue;
    GemmProblem& p = g.p[g.nprob++];
    p.M = s.T;
    p.N = s.d;
    p.K = s.rl[LQ + i];
    p.a[0] = op(at(A.h_qkv, s.off[i], s), s.rqkv, KM);
    p.b[0] = op(Bs[i], s.rl[LQ + i], KM);
    p.out[0] = outs[i];
    p.ldo[0] = s.d;
  }
  gemm(c, s, g);
}

// x1 = x + sigma(z_o) B_o^T
void o_up(Ctx& c, const Shape& s, const bn_block_params* W, const void* x, const Acts& A) {
  GemmLaunch g = launch(EPI_RESID, s);
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = s.d;
  p.K = s.rl[LO];
  p.a[0] = op(A.h_o, s.rl[LO], KM);
  p.b[0] = op(W->B_o, s.rl[LO], KM);
  p.in[0] = x;
  p.ldi[0] = s.d;
  p.out[0] = A.x1;
  p.ldo[0] = s.d;
  gemm(c, s, g);
}

// G, U = sigma(z_g) B_g^T, sigma(z_u) B_u^T; m = SiLU(G) U
void gu_up(Ctx& c, const Shape& s, const bn_block_params* W, const Acts& A, bool keep_gu) {
  GemmLaunch g = launch(EPI_SWIGLU, s);
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = s.d_ff;
  p.K = s.rl[LG];
  p.K2 = s.rl[LU];
  p.a[0] = op(A.h_gu, s.rgu, KM);
  p.b[0] = op(W->B_g, s.rl[LG], KM);
  p.a[1] = op(at(A.h_gu, s.rl[LG], s), s.rgu, KM);
  p.b[1] = op(W->B_u, s.rl[LU], KM);
  p.out[0] = keep_gu ? A.G : nullptr;
  p.out[1] = keep_gu ? A.U : nullptr;
  p.out[2] = A.m;
  p.ldo[0] = p.ldo[1] = p.ldo[2] = s.ld_act;
  gemm(c, s, g);
}

// y = x1 + sigma(z_d) B_d^T
void down_up(Ctx& c, const Shape& s, const bn_block_params* W, const Acts& A, const void* x1,
             void* y) {
  GemmLaunch g = launch(EPI_RESID, s);
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = s.d;
  p.K = s.rl[LD];
  p.a[0] = op(A.h_d, s.rl[LD], KM);
  p.b[0] = op(W->B_d, s.rl[LD], KM);
  p.in[0] = x1;
  p.ldi[0] = s.d;
  p.out[0] = y;
  p.ldo[0] = s.d;
  gemm(c, s, g);
}

// z = OnlineRMSNorm_S(x) Af^T (Af has the norm weight folded in), h = sigma(z)
void norm_down(Ctx& c, const Shape& s, const void* x, const float* ss, const void* Af, int64_t n,
               void* z, void* h) {
  GemmLaunch g = launch(EPI_NORM, s);
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = n;
  p.K = s.d;
  p.a[0] = op(x, s.d, KM);
  p.b[0] = op(Af, s.d, KM);
  p.rowv = ss;
  p.out[0] = z;
  p.ldo[0] = n;
  p.out[1] = h;
  p.ldo[1] = n;
  gemm(c, s, g);
}

// z = X A^T, h = sigma(z)   (X [T, K] with leading dimension ldx). Emulated
// bottleneck-aware TP: a row-parallel down-projection, the S shards' partial
// products summed in the epilogue (the chunk's all-reduce).
void plain_down(Ctx& c, const Shape& s, const void* X, int64_t K, int64_t ldx, const void* Adown,
                int64_t lda, int64_t n, void* z, void* h) {
  GemmLaunch g = launch(s.btp ? EPI_NORM : EPI_SIGMA, s);  // EPI_NORM with no rowv: shard sum
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = n;
  p.K = K;
  p.a[0] = op(X, ldx, KM);
  p.b[0] = op(Adown, lda, KM);
  p.out[0] = z;
  p.ldo[0] = n;
  p.out[1] = h;
  p.ldo[1] = n;
  gemm(c, s, g);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
void forward_lowrank(Ctx& c, const Shape& s, const bn_block_params* W, const void* x, void* y,
                     void* q, void* k, const Acts& A, const Tmp& B) {
  const void* x1 = x;
  const Fold f2{W->A_gu, W->w_norm2, s.rgu, s.d, B.A2f};
  chain_reset(c, s, B, 0, 4, 1);
  if (s.full()) {
    const Fold f1{W->A_qkv, W->w_norm1, s.rqkv, s.d, B.A1f};
    DT_CALL(s, stats_fold, c, x, s, A.ss1, A.rstd1, f1, f2);
    produce(c, s, B, 0);
    norm_down(c, s, x, A.ss1, B.A1f, s.rqkv, A.z_qkv, A.h_qkv);
    consume(c, s, B, 0);
    qkv_up(c, s, W, A, s.attn ? A.Q : q, s.attn ? A.K : k);
    if (s.attn) attention(c, s, A, B);
    produce(c, s, B, 1);
    plain_down(c, s, s.attn ? A.O : A.V, s.d, s.d, W->A_o, s.d, s.rl[LO], A.z_o, A.h_o);
    consume(c, s, B, 1);
    o_up(c, s, W, x, A);
    x1 = A.x1;
    DT_CALL(s, stats, c, x1, s, A.ss2, A.rstd2);
  } else {
    DT_CALL(s, stats_fold, c, x1, s, A.ss2, A.rstd2, f2, Fold{});
  }
  produce(c, s, B, 2);
  norm_down(c, s, x1, A.ss2, B.A2f, s.rgu, A.z_gu, A.h_gu);
  consume(c, s, B, 2);
  gu_up(c, s, W, A, !s.ckpt);
  produce(c, s, B, 3);
  plain_down(c, s, A.m, s.d_ff, s.ld_act, W->A_d, s.ld_ff, s.rl[LD], A.z_d, A.h_d);
  consume(c, s, B, 3);
  down_up(c, s, W, A, x1, y);
}

void forward_dense(Ctx& c, const Shape& s, const bn_block_params* W, const void* x, void* y,
                   void* q, void* k, const Acts& A, const Tmp& B) {
  const void* x1 = x;
  const Fold f2{W->A_gu, W->w_norm2, 2 * s.d_ff, s.d, B.A2f};
  if (s.full()) {
    const Fold f1{W->A_qkv, W->w_norm1, 3 * s.d, s.d, B.A1f};
    DT_CALL(s, stats_fold, c, x, s, A.ss1, A.rstd1, f1, f2);
    GemmLaunch g = launch(EPI_NORM, s);
    void* outs[3] = {s.attn ? A.Q : q, s.attn ? A.K : k, A.V};
    for (int i = 0; i < 3; ++i) {
      GemmProblem& p = g.p[g.nprob++];
      p.M = s.T;
      p.N = s.d;
      p.K = s.d;
      p.a[0] = op(x, s.d, KM);
      p.b[0] = op(at(B.A1f, i * s.d * s.d, s), s.d, KM);
      p.rowv = A.ss1;
      p.out[0] = outs[i];
      p.ldo[0] = s.d;
    }
    gemm(c, s, g);
    if (s.attn) attention(c, s, A, B);
    GemmLaunch o = launch(EPI_RESID, s);
    o.nprob = 1;
    GemmProblem& p = o.p[0];
    p.M = s.T;
    p.N = s.d;
    p.K = s.d;
    p.a[0] = op(s.attn ? A.O : A.V, s.d, KM);
    p.b[0] = op(W->A_o, s.d, KM);
    p.in[0] = x;
    p.ldi[0] = s.d;
    p.out[0] = A.x1;
    p.ldo[0] = s.d;
    gemm(c, s, o);
    x1 = A.x1;
    DT_CALL(s, stats, c, x1, s, A.ss2, A.rstd2);
  } else {
    DT_CALL(s, stats_fold, c, x1, s, A.ss2, A.rstd2, f2, Fold{});
  }
  GemmLaunch g = launch(EPI_NORM, s);
  void* outs[2] = {A.G, A.U};
  for (int i = 0; i < 2; ++i) {
    GemmProblem& p = g.p[g.nprob++];
    p.M = s.T;
    p.N = s.d_ff;
    p.K = s.d;
    p.a[0] = op(x1, s.d, KM);
    p.b[0] = op(at(B.A2f, i * s.d_ff * s.d, s), s.d, KM);
    p.rowv = A.ss2;
    p.out[0] = outs[i];
    p.ldo[0] = s.ld_act;
  }
  gemm(c, s, g);
  DT_CALL(s, swiglu_ew, c, s, A.G, A.U, A.m);
  GemmLaunch d = launch(EPI_RESID, s);
  d.nprob = 1;
  GemmProblem& p = d.p[0];
  p.M = s.T;
  p.N = s.d;
  p.K = s.d_ff;
  p.a[0] = op(A.m, s.ld_act, KM);
  p.b[0] = op(W->A_d, s.ld_ff, KM);
  p.in[0] = x1;
  p.ldi[0] = s.d;
  p.out[0] = y;
  p.ldo[0] = s.d;
  gemm(c, s, d);
}

// Checkpoint mode: rebuild every activation the backward reads from the saved
// pre-activations, with the same kernels (bit-identical to the forward).
void recompute(Ctx& c, const Shape& s, const bn_block_params* W, const void* x, const Acts& A,
               const Tmp& B) {
  const void* x1 = x;
  if (s.full()) {
    DT_CALL(s, stats, c, x, s, A.ss1, A.rstd1);
    DT_CALL(s, sigma_ew, c, s, A.z_qkv, s.rqkv, s.rqkv, A.h_qkv);
    qkv_up(c, s, W, A, s.attn ? A.Q : nullptr, s.attn ? A.K : nullptr);
    if (s.attn) attention(c, s, A, B);  // O for the O bottleneck's backward
    DT_CALL(s, sigma_ew, c, s, A.z_o, s.rl[LO], s.rl[LO], A.h_o);
    o_up(c, s, W, x, A);
    x1 = A.x1;
  }
  DT_CALL(s, stats, c, x1, s, A.ss2, A.rstd2);
  DT_CALL(s, sigma_ew, c, s, A.z_gu, s.rgu, s.rgu, A.h_gu);
  gu_up(c, s, W, A, true);
  DT_CALL(s, sigma_ew, c, s, A.z_d, s.rl[LD], s.rl[LD], A.h_d);
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
// The sigma-backward of a low-rank layer: dh = dY Bup summed over all of dY's
// columns at once, or (emulated bottleneck-aware TP) over the S shards of the
// column-parallel up-projection's outputs, summed in the epilogue (the
// backward's r-wide all-reduce).
Epi dsigma_epi(const Shape& s) { return s.btp ? EPI_SHARD_DSIGMA : EPI_DSIGMA; }

// dz = (dY Bup) * sigma'(z) * rowv: one problem of a grouped DSIGMA launch
// (Bup [K, n]: the layer's up-projection, n its rank)
GemmProblem dsigma(const Shape& s, const void* dY, int64_t ldy, int64_t K, const void* Bup,
                   int64_t n, const void* z, int64_t ldz, void* dz, const float* rowv) {
  GemmProblem p;
  p.M = s.T;
  p.N = n;
  p.K = K;
  p.a[0] = op(dY, ldy, KM);
  p.b[0] = op(Bup, n, MN);
  p.in[0] = z;
  p.ldi[0] = ldz;
  p.out[0] = dz;
  p.ldo[0] = ldz;
  p.rowv = rowv;
  return p;
}

// dX = dz A  (dz [T, K] K-major, A [K, N] row-major)
void dx_gemm(Ctx& c, const Shape& s, const void* dz, int64_t K, const void* A, int64_t lda,
             int64_t N, void* out, int64_t ldo, const float* rowv = nullptr) {
  GemmLaunch g = launch(EPI_STORE, s);
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = s.T;
  p.N = N;
  p.K = K;
  p.a[0] = op(dz, K, KM);
  p.b[0] = op(A, lda, MN);
  p.out[0] = out;
  p.ldo[0] = ldo;
  p.rowv = rowv;
  gemm(c, s, g);
}

void flush_wgrads(Ctx& c, const Shape& s, Wgrads& w, bool final) {
  TileReduce tr;
  if (w.n > 0) {
    GemmLaunch g = launch(EPI_STORE, s);
    g.allow_split = true;
    if (final) g.finish = &tr;
    g.nprob = w.n;
    for (int i = 0; i < w.n; ++i) g.p[i] = w.p[i];
    gemm(c, s, g);
    w.n = 0;
  }
  if (!final) return;
  for (int j = 0; j < w.ncol; ++j) tr.col[j] = w.col[j];
  tr.ncol = w.ncol;
  w.ncol = 0;
  launch_finish(c, tr);
}

void backward_lowrank(Ctx& c, const Shape& s, const bn_block_params* W, const void* x,
                      const void* dy, const void* dq, const void* dk, void* dx,
                      const bn_block_params* dW, const Acts& A, const Tmp& B) {
  const int64_t T = s.T, d = s.d;
  const int64_t ro = s.rl[LO], rg = s.rl[LG], ru = s.rl[LU], rd = s.rl[LD];
  const int64_t rqkv = s.rqkv, rgu = s.rgu;
  Wgrads wg;
  const void* x1 = s.full() ? A.x1 : x;
  chain_reset(c, s, B, 4, 4, 0);
  // ---- down bottleneck: y = x1 + B_d sigma(A_d m)
  add_wgrad(c, s, wg, wgrad(d, rd, T, dy, d, A.h_d, rd, dW->B_d, rd));
  {
    GemmLaunch g = launch(dsigma_epi(s), s);
    g.nprob = 1;
    g.p[0] = dsigma(s, dy, d, d, W->B_d, rd, A.z_d, rd, B.dz_d, nullptr);
    produce(c, s, B, 4);
    gemm(c, s, g);
  }
  add_wgrad(c, s, wg, wgrad(rd, s.d_ff, T, B.dz_d, rd, A.m, s.ld_act, dW->A_d, s.ld_ff));
  consume(c, s, B, 4);
  {
    // dm = dz_d A_d, then the SwiGLU backward in the epilogue
    GemmLaunch g = launch(EPI_DSWIGLU, s);
    g.nprob = 1;
    GemmProblem& p = g.p[0];
    p.M = T;
    p.N = s.d_ff;
    p.K = rd;
    p.a[0] = op(B.dz_d, rd, KM);
    p.b[0] = op(W->A_d, s.ld_ff, MN);
    p.in[0] = A.G;
    p.in[1] = A.U;
    p.ldi[0] = p.ldi[1] = s.ld_act;
    p.out[0] = B.dG;
    p.out[1] = B.dU;
    p.ldo[0] = p.ldo[1] = s.ld_act;
    gemm(c, s, g);
  }
  // ---- gate / up bottlenecks
  add_wgrad(c, s, wg, wgrad(s.d_ff, rg, T, B.dG, s.ld_act, A.h_gu, rgu, dW->B_g, rg));
  add_wgrad(c, s, wg, wgrad(s.d_ff, ru, T, B.dU, s.ld_act, at(A.h_gu, rg, s), rgu, dW->B_u, ru));
  {
    GemmLaunch g = launch(dsigma_epi(s), s);
    g.nprob = 2;
    g.p[0] = dsigma(s, B.dG, s.ld_act, s.d_ff, W->B_g, rg, A.z_gu, rgu, B.dz_gu, A.rstd2);
    g.p[1] = dsigma(s, B.dU, s.ld_act, s.d_ff, W->B_u, ru, at(A.z_gu, rg, s), rgu,
                    at(B.dz_gu, rg, s), A.rstd2);
    produce(c, s, B, 5);
    gemm(c, s, g);
  }
  add_wgrad(c, s, wg, wgrad(rgu, d, T, B.dz_gu, rgu, x1, d, dW->A_gu, d, W->w_norm2));
  consume(c, s, B, 5);
  dx_gemm(c, s, B.dz_gu, rgu, W->A_gu, d, d, B.dn, d);
  void* dx1 = s.full() ? B.dx1 : dx;
  DT_CALL(s, normbwd, c, s, B, wg, B.dw_part2, B.dn, x1, W->w_norm2, A.rstd2, dy, dx1,
          dW->w_norm2);
  if (!s.full()) {
    flush_wgrads(c, s, wg, true);
    return;
  }

  // ---- O bottleneck: x1 = x + B_o sigma(A_o V)
  add_wgrad(c, s, wg, wgrad(d, ro, T, dx1, d, A.h_o, ro, dW->B_o, ro));
  {
    GemmLaunch g = launch(dsigma_epi(s), s);
    g.nprob = 1;
    g.p[0] = dsigma(s, dx1, d, d, W->B_o, ro, A.z_o, ro, B.dz_o, nullptr);
    produce(c, s, B, 6);
    gemm(c, s, g);
  }
  add_wgrad(c, s, wg, wgrad(ro, d, T, B.dz_o, ro, s.attn ? A.O : A.V, d, dW->A_o, d));
  consume(c, s, B, 6);
  dx_gemm(c, s, B.dz_o, ro, W->A_o, d, d, s.attn ? B.dO : B.dV, d);
  if (s.attn)
    track(c, attn_backward(c, attn_desc(s), A.Q, A.K, A.V, A.O, A.lse, B.dO, B.dQ, B.dK, B.dV,
                           B.attn_rows, B.status));

  // ---- Q / K / V bottlenecks
  const void* dQKV[3] = {s.attn ? B.dQ : dq, s.attn ? B.dK : dk, B.dV};
  const void* Bup[3] = {W->B_q, W->B_k, W->B_v};
  void* dB[3] = {dW->B_q, dW->B_k, dW->B_v};
  for (int i = 0; i < 3; ++i) {
    const int64_t ri = s.rl[LQ + i];
    if (dQKV[i] == nullptr)
      zero2d(c, dB[i], ri * s.E, ri * s.E, d);
    else
      add_wgrad(c, s, wg, wgrad(d, ri, T, dQKV[i], d, at(A.h_qkv, s.off[i], s), rqkv, dB[i], ri));
  }
  {
    GemmLaunch g = launch(dsigma_epi(s), s);
    for (int i = 0; i < 3; ++i) {
      const int64_t ri = s.rl[LQ + i];
      if (dQKV[i] == nullptr) {
        zero2d(c, at(B.dz_qkv, s.off[i], s), rqkv * s.E, ri * s.E, T);
        continue;
      }
      g.p[g.nprob++] = dsigma(s, dQKV[i], d, d, Bup[i], ri, at(A.z_qkv, s.off[i], s), rqkv,
                              at(B.dz_qkv, s.off[i], s), A.rstd1);
    }
    // with a zeroed slice (dq or dk absent) not every row block is counted
    if (g.nprob == 3) produce(c, s, B, 7);
    gemm(c, s, g);
  }
  add_wgrad(c, s, wg, wgrad(rqkv, d, T, B.dz_qkv, rqkv, x, d, dW->A_qkv, d, W->w_norm1));
  consume(c, s, B, 7);
  dx_gemm(c, s, B.dz_qkv, rqkv, W->A_qkv, d, d, B.dn, d);
  DT_CALL(s, normbwd, c, s, B, wg, B.dw_part1, B.dn, x, W->w_norm1, A.rstd1, dx1, dx,
          dW->w_norm1);
  flush_wgrads(c, s, wg, true);
}

void backward_dense(Ctx& c, const Shape& s, const bn_block_params* W, const void* x,
                    const void* dy, const void* dq, const void* dk, void* dx,
                    const bn_block_params* dW, const Acts& A, const Tmp& B) {
  const int64_t T = s.T, d = s.d, dff = s.d_ff;
  const void* x1 = s.full() ? A.x1 : x;
  Wgrads wg;
  add_wgrad(c, s, wg, wgrad(d, dff, T, dy, d, A.m, s.ld_act, dW->A_d, s.ld_ff));
  {
    // dm = dy W_d with the SwiGLU backward; rows scaled by rstd2 for the norm GEMMs
    GemmLaunch g = launch(EPI_DSWIGLU, s);
    g.nprob = 1;
    GemmProblem& p = g.p[0];
    p.M = T;
    p.N = dff;
    p.K = d;
    p.a[0] = op(dy, d, KM);
    p.b[0] = op(W->A_d, s.ld_ff, MN);
    p.in[0] = A.G;
    p.in[1] = A.U;
    p.ldi[0] = p.ldi[1] = s.ld_act;
    p.out[0] = B.dG;
    p.out[1] = B.dU;
    p.ldo[0] = p.ldo[1] = s.ld_act;
    p.rowv = A.rstd2;
    gemm(c, s, g);
  }
  add_wgrad(c, s, wg, wgrad(dff, d, T, B.dG, s.ld_act, x1, d, dW->A_gu, d, W->w_norm2));
  add_wgrad(c, s, wg, wgrad(dff, d, T, B.dU, s.ld_act, x1, d, at(dW->A_gu, dff * d, s), d, W->w_norm2));
  {
    GemmLaunch g = launch(EPI_STORE_CHAIN, s);
    g.nprob = 1;
    GemmProblem& p = g.p[0];
    p.M = T;
    p.N = d;
    p.K = dff;
    p.a[0] = op(B.dG, s.ld_act, KM);
    p.b[0] = op(W->A_gu, d, MN);
    p.a[1] = op(B.dU, s.ld_act, KM);
    p.b[1] = op(at(W->A_gu, dff * d, s), d, MN);
    p.out[0] = B.dn;
    p.ldo[0] = d;
    gemm(c, s, g);
  }
  void* dx1 = s.full() ? B.dx1 : dx;
  DT_CALL(s, normbwd, c, s, B, wg, B.dw_part2, B.dn, x1, W->w_norm2, A.rstd2, dy, dx1,
          dW->w_norm2);
  if (!s.full()) {
    flush_wgrads(c, s, wg, true);
    return;
  }
  add_wgrad(c, s, wg, wgrad(d, d, T, dx1, d, s.attn ? A.O : A.V, d, dW->A_o, d));
  if (s.attn) {
    dx_gemm(c, s, dx1, d, W->A_o, d, d, B.dO, d);
    track(c, attn_backward(c, attn_desc(s), A.Q, A.K, A.V, A.O, A.lse, B.dO, B.dQ, B.dK, B.dV,
                           B.attn_rows, B.status));
    DT_CALL(s, rowscale, c, s, B.dQ, d, A.rstd1, d, B.dqkv, 3 * d);
    DT_CALL(s, rowscale, c, s, B.dK, d, A.rstd1, d, at(B.dqkv, d, s), 3 * d);
    DT_CALL(s, rowscale, c, s, B.dV, d, A.rstd1, d, at(B.dqkv, 2 * d, s), 3 * d);
  } else {
    DT_CALL(s, rowscale, c, s, dq, d, A.rstd1, d, B.dqkv, 3 * d);
    DT_CALL(s, rowscale, c, s, dk, d, A.rstd1, d, at(B.dqkv, d, s), 3 * d);
    dx_gemm(c, s, dx1, d, W->A_o, d, d, at(B.dqkv, 2 * d, s), 3 * d, A.rstd1);
  }
  add_wgrad(c, s, wg, wgrad(3 * d, d, T, B.dqkv, 3 * d, x, d, dW->A_qkv, d, W->w_norm1));
  dx_gemm(c, s, B.dqkv, 3 * d, W->A_qkv, d, d, B.dn, d);
  DT_CALL(s, normbwd, c, s, B, wg, B.dw_part1, B.dn, x, W->w_norm1, A.rstd1, dx1, dx,
          dW->w_norm1);
  flush_wgrads(c, s, wg, true);
}

Ctx make_ctx(void* scratch, bn_stream_t stream, const Tmp& B) {
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.status = B.status;
  c.num_sms = device_sms();
  c.partial = B.partial;
  c.partial_bytes = B.partial_bytes;
  (void)scratch;
  return c;
}

}  // namespace
}  // namespace bn

using namespace bn;

extern "C" {

bn_status bn_block_workspace_size(const bn_block_desc* desc, size_t* saved_bytes,
                                  size_t* scratch_bytes) {
  Shape s;
  bn_status st = check_desc(desc, s);
  if (st != BN_OK) return st;
  if (saved_bytes == nullptr || scratch_bytes == nullptr) return BN_ERR_INVALID_ARG;
  Acts A;
  Tmp B;
  plan(s, nullptr, nullptr, A, B, saved_bytes, scratch_bytes);
  return BN_OK;
}

bn_status bn_block_forward(const bn_block_desc* desc, const bn_block_params* W, const void* x,
                           void* y, void* q_out, void* k_out, void* saved, void* scratch,
                           bn_stream_t stream) {
  g_last_launches = 0;
  Shape s;
  bn_status st = check_desc(desc, s);
  if (st != BN_OK) return st;
  if ((st = check_params(s, W)) != BN_OK) return st;
  if (!x || !y || !saved || !scratch) return BN_ERR_INVALID_ARG;
  // q and k leave the block only when the attention core runs outside it
  const bool qk_out = s.full() && !s.attn;
  if (qk_out != (q_out != nullptr) || qk_out != (k_out != nullptr)) return BN_ERR_INVALID_ARG;
  for (const void* p : {x, static_cast<const void*>(y), static_cast<const void*>(q_out),
                        static_cast<const void*>(k_out), static_cast<const void*>(saved),
                        static_cast<const void*>(scratch)})
    if (p && !aligned(p)) return BN_ERR_ALIGNMENT;
  Acts A;
  Tmp B;
  plan(s, saved, scratch, A, B, nullptr, nullptr);
  Ctx c = make_ctx(scratch, stream, B);
  if (s.dense)
    forward_dense(c, s, W, x, y, q_out, k_out, A, B);
  else
    forward_lowrank(c, s, W, x, y, q_out, k_out, A, B);
  return finish(c);
}

bn_status bn_block_backward(const bn_block_desc* desc, const bn_block_params* W, const void* x,
                            const void* saved, const void* dy, const void* dq, const void* dk,
                            void* dx, const bn_block_params* dW, void* scratch,
                            bn_stream_t stream) {
  g_last_launches = 0;
  Shape s;
  bn_status st = check_desc(desc, s);
  if (st != BN_OK) return st;
  if ((st = check_params(s, W)) != BN_OK) return st;
  if ((st = check_params(s, dW)) != BN_OK) return st;
  if (!x || !saved || !dy || !dx || !scratch) return BN_ERR_INVALID_ARG;
  if ((!s.full() || s.attn) && (dq || dk)) return BN_ERR_INVALID_ARG;
  for (const void* p : {x, saved, dy, dq, dk, static_cast<const void*>(dx),
                        static_cast<const void*>(scratch)})
    if (p && !aligned(p)) return BN_ERR_ALIGNMENT;
  Acts A;
  Tmp B;
  plan(s, const_cast<void*>(saved), scratch, A, B, nullptr, nullptr);
  Ctx c = make_ctx(scratch, stream, B);
  if (s.ckpt) recompute(c, s, W, x, A, B);
  if (s.dense)
    backward_dense(c, s, W, x, dy, dq, dk, dx, dW, A, B);
  else
    backward_lowrank(c, s, W, x, dy, dq, dk, dx, dW, A, B);
  return finish(c);
}

bn_status bn_get_device_status(void* scratch, bn_stream_t stream) {
  if (scratch == nullptr) return BN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(scratch, 0, sizeof(int));
  if (e != cudaSuccess) return static_cast<bn_status>(record_cuda_error(e));
  return (word & kStatusTimeout) ? BN_ERR_TIMEOUT : BN_OK;
}

int bn_last_launch_count(void) { return g_last_launches; }

const char* bn_status_string(bn_status s) {
  switch (s) {
    case BN_OK: return "BN_OK";
    case BN_ERR_INVALID_ARG: return "BN_ERR_INVALID_ARG";
    case BN_ERR_ALIGNMENT: return "BN_ERR_ALIGNMENT";
    case BN_ERR_UNSUPPORTED: return "BN_ERR_UNSUPPORTED";
    case BN_ERR_CUDA: return "BN_ERR_CUDA";
    case BN_ERR_TIMEOUT: return "BN_ERR_TIMEOUT";
  }
  return "unknown bn_status";
}

const char* bn_last_cuda_error(void) { return g_cuda_err; }

}  // extern "C"
