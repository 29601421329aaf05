// Host side of the tcgen05 GEMM engine: tensor-map encoding, tile width, the
// K split of left-over tiles, launch, and the deterministic partial-tile reduction.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm.h"
#include "gemm_tc_launch.h"
#include "rowops.h"

namespace bn {
namespace tc {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D tensor map over a row-major matrix [outer, inner] with row stride ld
// (elements of `esize` bytes: 2 = bf16, 4 = fp32).
static bool encode(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
                   uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B, int esize = 2) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15) ||
      (ld * esize) % 16)
    return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand of logical shape [mn, K]: K-major tiles are one box of 64 (K) x box_mn
// rows; MN-major tiles are boxes of 64 (MN) x 64 (K).
static bool encode_operand(CUtensorMap* m, const Operand& op, int64_t mn, int64_t K, int box_mn) {
  if (op.ptr == nullptr || (reinterpret_cast<uintptr_t>(op.ptr) & 15) || (op.ld * 2) % 16)
    return false;
  if (!op.mn_major) return encode(m, op.ptr, K, mn, op.ld, 64, static_cast<uint32_t>(box_mn));
  return encode(m, op.ptr, mn, K, op.ld, 64, 64);
}

static int epi_kind(Epi e) {
  switch (e) {
    case EPI_STORE: return K_STORE;
    case EPI_SIGMA: return K_SIGMA;
    case EPI_NORM: return K_NORM;
    case EPI_RESID: return K_RESID;
    case EPI_SWIGLU: return K_SWIGLU;
    case EPI_DSIGMA: return K_DSIGMA;
    case EPI_DSWIGLU: return K_DSWIGLU;
    case EPI_STORE_CHAIN: return K_CHAIN;
    case EPI_SHARD_DSIGMA: return K_SDSIGMA;
  }
  return -1;
}

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace tc

size_t gemm_tc_partial_bytes(int num_sms) {
  // at most one split unit per CTA group, each a [CG x 128][256] fp32 tile
  return static_cast<size_t>(num_sms) * tc::BM * 256 * 4;
}

namespace {
// CTA pairs (2-SM MMA) unless the problems are at most one 128-row tile tall,
// or BN_GEMM_CTA_PAIR=0 is set in the environment.
int cta_group_for(const GemmLaunch& g) {
  static const bool pairs_off = [] {
    const char* v = std::getenv("BN_GEMM_CTA_PAIR");
    return v != nullptr && v[0] == '0';
  }();
  if (pairs_off) return 1;
  for (int i = 0; i < g.nprob; ++i)
    if (g.p[i].M > tc::BM) return 2;
  return 1;
}
}  // namespace

// Estimated time of one tile of an epilogue kind, in units of k-elements of a
// plain 256 x 256 tile: the k extent (both operand pairs of SwiGLU) times a
// per-kind factor from the kinds' measured rates at the 1B and 7B shapes (the
// epilogues that read inputs or write two outputs are the slower ones).
static double unit_cost(int ek, const GemmProblem& q) {
  double k = static_cast<double>(q.K);
  if (ek == tc::K_SWIGLU || ek == tc::K_CHAIN) k += static_cast<double>(q.K2 > 0 ? q.K2 : q.K);
  switch (ek) {
    case tc::K_NORM: return 1.15 * k;
    case tc::K_SIGMA: return 0.9 * k;
    case tc::K_STORE: return 0.95 * k;
    case tc::K_SWIGLU: return 1.15 * k;
    case tc::K_RESID: return 1.5 * k;
    case tc::K_DSWIGLU: return 1.9 * k;
    default: return k;
  }
}

void gemm_tc(Ctx& c, const GemmLaunch& g) {
  using namespace tc;
  // this launch's chain links, if any (none carry over to a later launch)
  const ChainLink chain_out = c.chain_out, chain_in = c.chain_in;
  const int prod_units = c.chain_prod_units, prod_groups = c.chain_prod_groups;
  const double prod_cost = c.chain_prod_cost;
  c.chain_out = ChainLink{};
  c.chain_in = ChainLink{};
  c.chain_entered_target = 0;
  c.chain_rows_target = 0;
  c.chain_prod_units = c.chain_prod_groups = 0;
  c.chain_prod_cost = 0;
  int ek = epi_kind(g.epi);
  if (ek < 0 || g.nprob < 1 || g.nprob > kMaxProblems) {
    c.bad = 1;
    return;
  }
  // tile width: 256 columns (the MMA's most efficient shape) unless a problem is narrower
  int BN = 256;
  for (int i = 0; i < g.nprob; ++i)
    if (g.p[i].N < 256) BN = 128;
  static const int forced_bn = [] {  // BN_GEMM_TILE_N=128 forces narrow tiles (tuning experiments)
    const char* v = std::getenv("BN_GEMM_TILE_N");
    return (v != nullptr && v[0] == '1') ? 128 : 0;
  }();
  if (forced_bn) BN = forced_bn;

  const int CG = cta_group_for(g);
  const int BMP = BM * CG;  // rows per tile
  thread_local static Params P;  // large kernel parameter block, filled per call
  std::memset(&P, 0, sizeof(P));
  P.nprob = g.nprob;
  P.S = g.S;
  P.sigma = g.sigma;
  P.eps = g.eps;
  P.status = c.status;

  const bool a_mn = g.p[0].a[0].mn_major, b_mn = g.p[0].b[0].mn_major;
  int64_t tiles_total = 0, nkb_min = INT64_MAX;
  bool plain = true;  // no row scale: the reduction kernel applies only colv
  for (int i = 0; i < g.nprob; ++i) {
    const GemmProblem& q = g.p[i];
    if (q.M <= 0 || q.N <= 0 || q.K <= 0 || q.a[0].mn_major != a_mn || q.b[0].mn_major != b_mn) {
      c.bad = 1;
      return;
    }
    tiles_total += cdiv(q.M, BMP) * cdiv(q.N, BN);
    nkb_min = std::min(nkb_min, cdiv(q.K, BK));
    plain = plain && q.rowv == nullptr;
  }
  // K split (weight gradients, K = T): whole tiles fill complete rounds of the CTA
  // groups; the tiles left over are each cut into rem_split k-ranges of at least
  // 8 k-blocks that share one last round.
  const int groups = c.num_sms / CG;
  int64_t rem = 0;
  int rem_split = 1;
  if (ek == K_STORE && g.allow_split && plain) {
    rem = tiles_total % groups;
    if (rem > 0) {
      rem_split = static_cast<int>(std::min<int64_t>(groups / rem, nkb_min / 8));
      const size_t need = static_cast<size_t>(rem) * rem_split * BMP * BN * 4;
      if (rem_split < 2 || c.partial == nullptr || need > c.partial_bytes) rem_split = 1;
    }
  }
  if (rem_split == 1) rem = 0;
  const bool split = rem > 0;
  P.full_units = static_cast<int>(tiles_total - rem);
  P.rem_split = rem_split;
  P.part = split ? c.partial : nullptr;

  int units = 0;
  for (int i = 0; i < g.nprob; ++i) {
    const GemmProblem& q = g.p[i];
    Prob& p = P.p[i];
    const int npair = (ek == K_SWIGLU || ek == K_CHAIN) ? 2 : 1;
    for (int j = 0; j < npair; ++j) {
      // each CTA of a pair loads its own 128 rows of A and BN / CG rows of B
      const int64_t Kj = (j == 1 && q.K2 > 0) ? q.K2 : q.K;
      if (!encode_operand(&p.ma[j], q.a[j], q.M, Kj, BM) ||
          !encode_operand(&p.mb[j], q.b[j], q.N, Kj, BN / CG)) {
        c.bad = 2;
        return;
      }
      p.nkb[j] = static_cast<int>(cdiv(Kj, BK));
    }
    // Online RMSNorm's shards are equal, whole k-blocks; a plain shard sum needs
    // at least one k-block per shard
    if ((ek == K_NORM && q.rowv != nullptr && q.K % (BK * g.S) != 0) ||
        ((ek == K_NORM || ek == K_SDSIGMA) && (g.S < 1 || cdiv(q.K, BK) < g.S))) {
      c.bad = 3;
      return;
    }
    p.M = q.M;
    p.N = q.N;
    p.K = q.K;
    // epilogue outputs: 32 x 32 boxes (bf16, 64-byte swizzle; fp32 partials, 128-byte)
    const int nout = (ek == K_SWIGLU) ? 3 : (ek == K_SIGMA || ek == K_NORM || ek == K_DSWIGLU) ? 2 : 1;
    const int nin = (ek == K_RESID) ? 1 : (ek == K_DSWIGLU) ? 2 : 0;  // through the TMA ring
    p.out_mask = 0;
    p.N8 = q.N / 8 * 8;
    for (int j = 0; j < 3; ++j) {
      p.out[j] = q.out[j];
      p.ldo[j] = q.ldo[j];
    }
    for (int j = 0; j < nout; ++j) {
      if (q.out[j] == nullptr) continue;
      // TMA bounds the innermost dimension in 16-byte units: the map stops at N8
      // and the epilogue writes columns [N8, N) itself
      if (p.N8 > 0 &&
          !encode(&p.mo[j], q.out[j], p.N8, q.M, q.ldo[j], 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, 2)) {
        c.bad = 2;
        return;
      }
      p.out_mask |= 1 << j;
    }
    if (nout == 1 && !(p.out_mask & 1)) {
      c.bad = 2;
      return;
    }
    // epilogue inputs: 32-column x 128-row boxes
    for (int j = 0; j < nin; ++j) {
      if (!encode(&p.mi[j], q.in[j], q.N, q.M, q.ldi[j], 32, 128, CU_TENSOR_MAP_SWIZZLE_64B, 2)) {
        c.bad = 2;
        return;
      }
    }
    p.rowv = q.rowv;
    p.colv = q.colv;
    p.in_raw = (ek == K_DSIGMA || ek == K_SDSIGMA) ? q.in[0] : nullptr;
    p.ldi_raw = q.ldi[0];
    p.tiles_m = static_cast<int>(cdiv(q.M, BMP));
    p.tiles_n = static_cast<int>(cdiv(q.N, BN));
    p.tile_begin = units;
    units += p.tiles_m * p.tiles_n;
  }
  units = P.full_units + static_cast<int>(rem) * rem_split;
  P.total_units = units;
  double flops, bytes;
  gemm_work(g, 2, flops, bytes);
  // chained launches: kinds that take part, every problem spanning the same row blocks
  const bool producer = ek == K_NORM || ek == K_SIGMA || ek == K_DSIGMA || ek == K_SDSIGMA;
  const bool consumer = ek == K_STORE || ek == K_RESID || ek == K_SWIGLU || ek == K_DSWIGLU;
  P.out = producer ? chain_out : ChainLink{};
  P.in = consumer ? chain_in : ChainLink{};
  int tiles_per_row_block = 0;
  for (int i = 0; i < g.nprob; ++i) {
    if (g.p[i].M != g.p[0].M) {
      P.out = ChainLink{};
      P.in = ChainLink{};
    }
    tiles_per_row_block += P.p[i].tiles_n;
  }
  // A chained consumer after a producer whose last round was partial: the
  // producer's last (units mod groups) groups hold their SMs about one producer
  // unit longer, and the consumer CTAs that land there (its last groups, as
  // CTAs are placed in index order) start that much later. The other groups
  // take the first lead_rounds rounds alone: about as many of this launch's
  // units as fit in one producer unit (rounded down). While launches are timed
  // one by one, the events between them keep a launch from overlapping the one
  // before it: no consumer group starts late, and there is no lead.
  const double cost = unit_cost(ek, g.p[0]);
  static const bool lead_off = [] {
    const char* v = std::getenv("BN_GEMM_LEAD");
    return v != nullptr && v[0] == '0';
  }();
  if (P.in.rows != nullptr && !lead_off && !prof_active() && prod_groups > 0 && prod_units > prod_groups &&
      prod_units % prod_groups > 0 && cost > 0) {
    P.lead_late = prod_units % prod_groups;
    P.lead_rounds = static_cast<int>(std::min(16.0, std::floor(prod_cost / cost)));
  }
  prof_start(c);
  int ctas;
  if (CG == 2)
    ctas = (BN == 256) ? launch_bn256_cg2(ek, a_mn, b_mn, P, units, c.num_sms, c.stream)
                       : launch_bn128_cg2(ek, a_mn, b_mn, P, units, c.num_sms, c.stream);
  else
    ctas = (BN == 256) ? launch_bn256_cg1(ek, a_mn, b_mn, P, units, c.num_sms, c.stream)
                       : launch_bn128_cg1(ek, a_mn, b_mn, P, units, c.num_sms, c.stream);
  if (ctas == 0) {
    c.bad = 5;
    return;
  }
  // what a consumer of this launch waits for: all its CTAs past their dependency
  // wait, and per row block one count from each epilogue warp of each tile
  c.chain_entered_target = P.out.rows ? ctas : 0;
  c.chain_rows_target = P.out.rows ? tiles_per_row_block * NUM_EPI_WARPS * CG : 0;
  if (P.out.rows != nullptr) {
    c.chain_prod_units = P.total_units;
    c.chain_prod_groups = ctas / CG;
    c.chain_prod_cost = cost;
  }
  note_launch(c, KK_GEMM_TC, static_cast<int>(g.epi), flops, bytes);
  TileReduce local;
  TileReduce& r = g.finish ? *g.finish : local;
  r.rem_tiles = 0;
  if (split) {
    r.nprob = g.nprob;
    r.full_units = P.full_units;
    r.rem_split = rem_split;
    r.rem_tiles = static_cast<int>(rem);
    r.tile_rows = BMP;
    r.BN = BN;
    r.part = c.partial;
    for (int i = 0; i < g.nprob; ++i) {
      const Prob& p = P.p[i];
      TileReduceProb& q = r.p[i];
      q.M = p.M;
      q.N = p.N;
      q.tiles_n = p.tiles_n;
      q.tile_begin = p.tile_begin;
      q.colv = static_cast<const __nv_bfloat16*>(g.p[i].colv);
      q.out = static_cast<__nv_bfloat16*>(g.p[i].out[0]);
      q.ldo = g.p[i].ldo[0];
    }
    if (g.finish == nullptr) launch_finish(c, r);
  }
}

}  // namespace bn
