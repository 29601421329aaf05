// tcgen05 / TMA / TMEM GEMM engine for sm_103a with fused epilogues.
//
// Persistent CTAs, one per SM (352 threads). With CG = 2 the CTAs run in
// clusters of two and each pair computes one 256 x BN tile with the 2-SM MMA
// (tcgen05.mma.cta_group::2): each CTA loads its own 128 rows of A and half of
// B, the leader CTA (rank 0) issues the MMAs, the accumulator rows of each CTA
// land in its own TMEM. Per CTA:
//   warp 0        operand producer: TMA loads into a ring of shared-memory
//                 stages, each one 128 x 64 tile of A and one BN x 64 tile of
//                 B (bf16, 128-byte swizzle), one mbarrier per stage;
//   warp 1        owns the TMEM allocation (all 512 columns) and, from one
//                 thread, issues tcgen05.mma (M = 128, N = BN, K = 16, fp32
//                 accumulate) into a ring of TMEM accumulator slots of BN
//                 columns; tcgen05.commit frees a stage / publishes a slot;
//   warps 2..9    epilogue, two groups of four: tcgen05.ld (warp w reads TMEM
//                 lanes 32 (w % 4) .. +31: one tile row per thread; group g
//                 takes the tile's 32-column subtiles c with c % 2 == g), fused
//                 math, results written to a swizzled shared-memory subtile and
//                 stored with TMA;
//   warp 10       epilogue-input producer: TMA loads of the tensors an
//                 epilogue reads (residual, z, G and U) into the same
//                 subtile ring, ahead of the epilogue.
// Online RMSNorm's kernel moves the epilogue to warps 4..11 (warps 2 and 3 are
// idle) and shifts registers to it with setmaxnreg: it keeps each row's running
// sum over the shards in registers.
// The epilogue works on 128 x 32 subtiles; warp w owns rows 32 (w % 4) .. +31
// of each and stores them as one 32 x 32 TMA box, so every global access is a
// bulk copy and the threads only touch conflict-free swizzled shared memory.
//
// A work unit is one 128 x BN output tile (or one K split of it), a sequence
// of segments; each segment is a K range, possibly of another operand pair,
// accumulated in the next TMEM slot of the ring: this is how Online RMSNorm sees
// each emulated shard's partial product and how SwiGLU sees G and U side by side.
//
// Every mbarrier wait is bounded by wall time (kWaitLimitNs). On expiry the
// thread sets a CTA-wide abort flag and the device status word, all roles
// unwind, outstanding TMA copies and MMAs are drained (bounded), TMEM is
// freed and the kernel returns.
#pragma once

#include <cuda.h>
#include "common.cuh"
#include "tc_ptx.cuh"

namespace bn {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int NUM_EPI_WARPS = 8;                 // two groups of four
constexpr int NUM_THREADS = 32 * (3 + NUM_EPI_WARPS);
constexpr int EPI_GROUPS = NUM_EPI_WARPS / 4;
constexpr int EPI_N = 32;  // columns per epilogue subtile

// epilogue kinds of the kernel template
enum : int {
  K_STORE = 0, K_SIGMA = 2, K_NORM = 3, K_RESID = 4, K_SWIGLU = 5,
  K_DSIGMA = 6, K_DSWIGLU = 7, K_CHAIN = 8, K_SDSIGMA = 9
};
// Shard-summed kinds: K is cut into S segments (emulated shards), each
// segment's partial product goes to the next TMEM slot and the epilogue sums
// them in registers -- the emulated all-reduce. K_NORM applies Online RMSNorm's
// per-shard normalisation and correction while summing (or none, for a plain
// row-parallel down-projection, when rowv is null) and stores z and sigma(z);
// K_SDSIGMA sums dY B over the shards of B's output dimension and stores
// dz = sum * sigma'(z) * rowv.
template <int EK>
constexpr bool is_fold() {
  return EK == K_NORM || EK == K_SDSIGMA;
}

template <int EK>
struct EpiShape {
  // epilogue inputs staged through the ring by the input warp (the sigma-backward's
  // z is instead read straight into registers: its GEMMs are long in K, so the
  // read hides behind the next tile's MMAs, and the ring's space goes to stages)
  static constexpr int NIN = (EK == K_RESID) ? 1 : (EK == K_DSWIGLU) ? 2 : 0;
  static constexpr int NOUT =
      (EK == K_SWIGLU) ? 3 : (EK == K_SIGMA || EK == K_NORM || EK == K_DSWIGLU) ? 2 : 1;
  // subtiles per ring entry. SwiGLU's three outputs share two: G leaves its
  // subtile (stored while the U MMAs run) before m, formed from G and U later,
  // takes it over; the space saved goes to operand stages
  static constexpr int NT = (EK == K_SWIGLU) ? 2 : (NIN > NOUT ? NIN : NOUT);
  static constexpr int ELEM = 2;                             // output element bytes (bf16)
  static constexpr int SUB_BYTES = BM * EPI_N * ELEM;        // one 128 x 32 subtile
  static constexpr int WARP_BYTES = 32 * EPI_N * ELEM;       // one warp's 32 rows of it
  // ring entries: kinds that read epilogue inputs keep several subtiles of them in
  // flight; the others only need each warp's previous store to have left shared
  // memory, and leave the rest to operand stages
  // (the sigma down-projection's tiles are long in K: its light epilogue keeps up
  // with one entry per warp, and the space goes to a sixth operand stage)
  static constexpr int NE = (NIN > 0) ? 8 : (EK == K_SIGMA ? 2 : 4);
  static constexpr int BYTES = NE * NT * SUB_BYTES;
};

// Chained launches (ChainLink): the kinds that may produce rows for the next
// launch (the r-wide GEMMs) and the kinds that may consume the previous
// launch's rows (the up-projections and the dX GEMMs).
template <int EK>
constexpr bool can_produce() {
  return EK == K_NORM || EK == K_SIGMA || EK == K_DSIGMA || EK == K_SDSIGMA;
}
template <int EK>
constexpr bool can_consume() {
  return EK == K_STORE || EK == K_RESID || EK == K_SWIGLU || EK == K_DSWIGLU;
}

// First epilogue warp. Online RMSNorm keeps each row's running sum in the
// epilogue's registers, so its epilogue warps form whole warpgroups (4..11)
// that take registers from warpgroup 0 (warps 0..3: the producer, the MMA
// issuer and two idle warps) with setmaxnreg, which acts per warpgroup.
template <int EK>
constexpr int epi_warp0() {
  return is_fold<EK>() ? 4 : 2;
}
// threads of a CTA: kinds without epilogue inputs leave out the input-producer
// warp, which leaves the epilogue more registers
template <int EK>
constexpr int kernel_threads() {
  return is_fold<EK>() ? 32 * (4 + NUM_EPI_WARPS)
                      : (EpiShape<EK>::NIN > 0 ? NUM_THREADS : NUM_THREADS - 32);
}
// Online RMSNorm register split. At launch, 12 warps get 168 registers a thread
// (3 warps per SM sub-partition): 384 x 168 = 64512 in all. Warpgroup 0 drops to
// kNormRegsLow and the two epilogue warpgroups rise to kNormRegsHigh:
// 128 x 56 + 256 x 224 = 64512, no more than the launch's total, and 56 + 2 x 224
// = 504 of the 512 a sub-partition holds per lane. That increase is the only one:
// it asks for exactly what warpgroup 0 gives up, whatever the order in which the
// warps get there. At the end the epilogue drops to kNormRegsLow too (a decrease
// never waits), so every warp reaches the common exit path with the same count.
constexpr int kNormRegsLaunch = 168;
constexpr int kNormRegsLow = 56;
constexpr int kNormRegsHigh = 224;
static_assert(128 * kNormRegsLow + 256 * kNormRegsHigh <= 384 * kNormRegsLaunch,
              "register split too large");
static_assert(kNormRegsLow + 2 * kNormRegsHigh <= 512, "register split exceeds a sub-partition");

template <int BN, int EK, int CG = 1>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / CG) * BK * 2;  // each CTA holds BN / CG rows of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TX_BYTES = CG * STAGE_BYTES;    // bytes one stage receives, whole pair
  static constexpr int NSLOT = 512 / BN;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int EPI_BYTES = EpiShape<EK>::BYTES;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(STAGES >= 2, "shared memory too small for the pipeline");
};

struct Prob {
  CUtensorMap ma[2];  // A operand of segment pair 0 / 1
  CUtensorMap mb[2];  // B operand of segment pair 0 / 1
  CUtensorMap mo[3];  // outputs: 32 x 32 boxes
  CUtensorMap mi[2];  // epilogue inputs: 32-column x 128-row boxes
  int64_t M, N, K;
  int64_t N8;         // N rounded down to a multiple of 8: TMA stores cover [0, N8)
  void* out[3];       // raw outputs, for the ragged columns [N8, N)
  int64_t ldo[3];
  const float* rowv;
  const void* colv;
  int tiles_m, tiles_n;
  int tile_begin;     // tiles of the problems before this one
  int nkb[2];         // k-blocks of operand pair 0 / 1
  int out_mask;       // bit k: output k is written
  const void* in_raw; // sigma-backward: z, read directly (row stride ldi_raw)
  int64_t ldi_raw;
};

struct Params {
  Prob p[kMaxProblems];
  int nprob, total_units, S, sigma;
  float eps;
  int* status;
  // Units [0, full_units) are whole tiles, in tile order over the problems,
  // dealt round-robin to the CTA groups. Each remaining tile (STORE with K split)
  // is cut into rem_split k-ranges, units full_units + rem_split t + s, whose
  // fp32 partial tiles go to `part` and are summed by a reduction kernel: the
  // whole tiles fill complete rounds and the split tiles one last round.
  int full_units, rem_split;
  float* part;  // per split unit j: [CG x 128][BN] fp32 at j * CG * 128 * BN
  ChainLink out;  // this launch produces rows for the next launch (counts them)
  ChainLink in;   // this launch consumes the previous launch's rows (waits on them)
  // Lead rounds of a chained consumer: its last lead_late groups start on the
  // SMs its producer's partial last round holds, about one producer tile late,
  // so the first lead_rounds rounds go to the other groups only (see
  // first_unit / next_unit). 0: plain round robin.
  int lead_late, lead_rounds;
};

// The units of group `pair` of `npairs`, in increasing order. With E = npairs -
// lead_late early groups and base = lead_rounds x E, units [0, base) are dealt
// round robin to the early groups, then units from base round robin to all
// groups; without a lead (base = 0) that is plain round robin.
struct UnitSeq {
  int pair, npairs, early, base;
  __device__ __forceinline__ UnitSeq(const Params& P, int pair_, int npairs_)
      : pair(pair_), npairs(npairs_), early(npairs_ - P.lead_late), base(0) {
    if (P.lead_late > 0 && P.lead_rounds > 0 && early > 0) base = P.lead_rounds * early;
  }
  __device__ __forceinline__ int first() const { return pair < early ? pair : base + pair; }
  __device__ __forceinline__ int next(int u) const {
    if (u < base) {
      u += early;
      return u < base ? u : base + pair;
    }
    return u + npairs;
  }
};

// ---------------------------------------------------------------------------
// barrier waits of the engine (the PTX wrappers are in tc_ptx.cuh)
// ---------------------------------------------------------------------------
template <int EK>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status, unsigned long long limit_ns = kWaitLimitNs) {
  if constexpr (is_fold<EK>())
    return wait_bar_inline(bar, parity, abort_flag, status, limit_ns);
  else
    return wait_bar_call(bar, parity, abort_flag, status, limit_ns);
}

// ---------------------------------------------------------------------------
// one thread's row of a warp's 32 x 32 subtile block in shared memory
//  bf16: 64-byte rows, 64-byte swizzle (16-byte chunk c of row t at c ^ ((t >> 1) & 3))
//  fp32: 128-byte rows, 128-byte swizzle (chunk c of row t at c ^ (t & 7))
// These are the layouts TMA reads and writes for boxes of 32 columns with
// SWIZZLE_64B / SWIZZLE_128B, and a warp's 16-byte accesses are conflict free.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void smem_row_store_bf16(uint8_t* blk, int t, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[8 * c + 2 * i], v[8 * c + 2 * i + 1]);
    *reinterpret_cast<uint4*>(blk + t * 64 + ((c ^ ((t >> 1) & 3)) << 4)) = u;
  }
}
// the same row layout from 16 packed bf16 pairs
__device__ __forceinline__ void smem_row_store_packed(uint8_t* blk, int t, const uint32_t* pk) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(blk + t * 64 + ((c ^ ((t >> 1) & 3)) << 4)) =
        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}
__device__ __forceinline__ void smem_row_load_bf16(const uint8_t* blk, int t, float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(blk + t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * c + 2 * i] = f.x;
      v[8 * c + 2 * i + 1] = f.y;
    }
  }
}
// Columns [max(col0, N8), min(col0 + 32, N)) of one row, written directly: TMA
// bounds the innermost dimension in 16-byte units, so the maps stop at N8 and
// this covers the last (N mod 8) columns.
__device__ __forceinline__ void store_tail_bf16(void* base, int64_t ld, int64_t row, int64_t col0,
                                                int64_t N8, int64_t N, const float* v) {
  __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + row * ld;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int64_t col = col0 + i;
    if (col >= N8 && col < N) p[col] = __float2bfloat16_rn(v[i]);
  }
}
// Row `row`, columns [col0, col0 + 32) of a bf16 matrix with row stride ld and N
// columns, zero beyond N or when the row is outside the matrix.
__device__ __forceinline__ void ld_row32_bf16(const __nv_bfloat16* p, int64_t ld, int64_t row,
                                              bool row_ok, int64_t col0, int64_t N, float* v) {
  const __nv_bfloat16* r = p + (row_ok ? row : 0) * ld;
  if (row_ok && col0 + 32 <= N) {
#pragma unroll
    for (int i = 0; i < 4; ++i) Vec8<__nv_bfloat16>::load(r + col0 + 8 * i, v + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = (row_ok && col0 + i < N) ? __bfloat162float(r[col0 + i]) : 0.f;
  }
}
// 32 bf16 values starting at column col0 of a vector of length N (zero beyond N)
__device__ __forceinline__ void ld_vec_bf16(const __nv_bfloat16* p, int64_t col0, int64_t N,
                                            float* v) {
  if (col0 + 32 <= N) {
#pragma unroll
    for (int i = 0; i < 4; ++i) Vec8<__nv_bfloat16>::load(p + col0 + 8 * i, v + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = (col0 + i < N) ? __bfloat162float(p[col0 + i]) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// work decomposition
// ---------------------------------------------------------------------------
struct Work {
  int pi;
  int64_t m0, nb;
  int kb0, kb1;   // k-blocks [kb0, kb1)
  int part_slot;  // -1: a whole tile; else its fp32 partial goes to this slot
};

// Unit u -> problem, first row m0 of the (CG x 128)-row tile, n-block, k-range.
template <int CG>
__device__ __forceinline__ Work decode(const Params& P, int u) {
  Work w;
  int t = u;
  int sp = 0;
  w.part_slot = -1;
  if (u >= P.full_units) {
    const int j = u - P.full_units;
    t = P.full_units + j / P.rem_split;
    sp = j % P.rem_split;
    w.part_slot = j;
  }
  int pi = 0;
  while (pi + 1 < P.nprob && t >= P.p[pi + 1].tile_begin) ++pi;
  const Prob& pr = P.p[pi];
  const int local = t - pr.tile_begin;
  w.pi = pi;
  w.m0 = static_cast<int64_t>(local / pr.tiles_n) * BM * CG;
  w.nb = local % pr.tiles_n;  // n-block index; the kernel scales it by BN
  const int nkb = pr.nkb[0];
  w.kb0 = (w.part_slot < 0) ? 0 : sp * nkb / P.rem_split;
  w.kb1 = (w.part_slot < 0) ? nkb : (sp + 1) * nkb / P.rem_split;
  return w;
}

template <int EK>
__device__ __forceinline__ int num_segments(const Params& P) {
  return is_fold<EK>() ? P.S : (EK == K_SWIGLU || EK == K_CHAIN) ? 2 : 1;
}
// k-block range and operand pair of segment s of a unit
template <int EK>
__device__ __forceinline__ void segment(const Params& P, const Prob& pr, const Work& w, int s,
                                        int& kb0, int& nkb, int& pair) {
  if (is_fold<EK>()) {
    // S segments of k-blocks (equal when S divides the k-blocks, as Online
    // RMSNorm's shards require; otherwise the first ones one shorter)
    kb0 = s * pr.nkb[0] / P.S;
    nkb = (s + 1) * pr.nkb[0] / P.S - kb0;
    pair = 0;
  } else if (EK == K_SWIGLU || EK == K_CHAIN) {
    kb0 = 0;
    nkb = pr.nkb[s];
    pair = s;
  } else {
    kb0 = w.kb0;
    nkb = w.kb1 - w.kb0;
    pair = 0;
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BN, int EK, bool AMN, bool BMN, int CG>
__global__ void __launch_bounds__(kernel_threads<EK>(), 1) gemm_kernel(const __grid_constant__ Params P) {
  using C = Cfg<BN, EK, CG>;
  using E = EpiShape<EK>;
  constexpr int NCH = BN / EPI_N;  // epilogue subtiles per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* epi = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::EPI_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = full + C::STAGES;
  uint64_t* accf = empty + C::STAGES;
  uint64_t* acce = accf + C::NSLOT;
  uint64_t* epi_full = acce + C::NSLOT;
  uint64_t* epi_empty = epi_full + E::NE;
  uint64_t* drain = epi_empty + E::NE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: both CTAs of a pair walk the same units; rank 1 adds 128 rows
  const uint32_t rank = (CG == 2) ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x) / CG;
  const int npairs = static_cast<int>(gridDim.x) / CG;
  const int row_off = BM * static_cast<int>(rank);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), NUM_EPI_WARPS * CG);  // the pair's epilogue warps
    }
    for (int i = 0; i < E::NE; ++i) {
      mbar_init(smem_u32(&epi_full[i]), 1);
      mbar_init(smem_u32(&epi_empty[i]), 4);  // the four warps of the group that used it
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers are initialised
  if (warp == 1) tmem_alloc<CG>(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // setup above touches no global memory; from here on the previous kernel's
  // results are read and its inputs may be overwritten
  // A chained consumer starts during its producer's last round: it triggers its
  // own dependents but does not wait for the producer grid to finish; its roles
  // wait below for the producer's CTAs to be past their own dependency wait
  // (so every earlier kernel is complete) and, per tile, for the rows they read.
  if (!can_consume<EK>() || P.in.rows == nullptr)
    grid_dependency_sync();
  else
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if constexpr (can_produce<EK>())
    if (P.out.entered != nullptr && threadIdx.x == 0) red_release_add(P.out.entered, 1);
  const uint32_t tmem = *tmem_slot;
  const int nseg = num_segments<EK>(P);
  const UnitSeq seq(P, pair, npairs);

  // Online RMSNorm's register split is made per warpgroup, in one place for
  // each: a point where the register count differs between the branches
  // cannot be shared code.
  if (warp == 0 || warp == 1 || warp == epi_warp0<EK>() + NUM_EPI_WARPS ||
      (is_fold<EK>() && warp < 4)) {
  if constexpr (is_fold<EK>()) setmaxnreg_dec<kNormRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ operand producer
    if (lane == 0) {
      for (int i = 0; i < P.nprob; ++i) {
        tma_prefetch_desc(&P.p[i].ma[0]);
        tma_prefetch_desc(&P.p[i].mb[0]);
      }
      int stage = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = !can_consume<EK>() || P.in.entered == nullptr ||
                wait_count(P.in.entered, P.in.entered_target, abort_flag, P.status);
      for (int u = seq.first(); ok && u < P.total_units; u = seq.next(u)) {
        const Work w = decode<CG>(P, u);
        const Prob& pr = P.p[w.pi];
        if (can_consume<EK>() && P.in.rows != nullptr) {
          // the producer's tiles of these rows have all been stored
          if (!wait_count(P.in.rows + w.m0 / (BM * CG), P.in.rows_target, abort_flag, P.status)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const int m0 = static_cast<int>(w.m0) + row_off;                  // this CTA's A rows
        const int n0 = static_cast<int>(w.nb) * BN + static_cast<int>(rank) * (BN / CG);  // B rows
        for (int s = 0; ok && s < nseg; ++s) {
          int kb0, nkb, opair;
          segment<EK>(P, pr, w, s, kb0, nkb, opair);
          const CUtensorMap* ma = &pr.ma[opair];
          const CUtensorMap* mb = &pr.mb[opair];
          for (int kb = kb0; kb < kb0 + nkb; ++kb) {
            if (!wait_bar<EK>(smem_u32(&empty[stage]), ph ^ 1u, abort_flag, P.status)) {
              ok = false;
              break;
            }
            const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
            // the stage's completion is counted on the leader's barrier, for the whole pair
            const uint32_t fb = smem_u32(&full[stage]);
            const uint32_t fbc = (CG == 2) ? mapa(fb, 0) : fb;
            if (leader) mbar_expect_tx(fb, C::TX_BYTES);
            const int k0 = kb * BK;
            auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1) {
              if constexpr (CG == 2)
                tma_load_2d_pair(dst, map, c0, c1, fbc);
              else
                tma_load_2d(dst, map, c0, c1, fb);
            };
            if (AMN) {
              load(sa, ma, m0, k0);
              load(sa + 8192, ma, m0 + 64, k0);
            } else {
              load(sa, ma, k0, m0);
            }
            if (BMN) {
#pragma unroll
              for (int j = 0; j < BN / CG / 64; ++j) load(sb + j * 8192, mb, n0 + 64 * j, k0);
            } else {
              load(sb, mb, k0, n0);
            }
            ++issued;
            if (++stage == C::STAGES) {
              stage = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        // drain: the last phase issued on each stage must land before the CTA exits
        int st = stage;
        uint32_t p = ph;
        for (int i = 0; i < C::STAGES && i < issued; ++i) {
          if (--st < 0) {
            st = C::STAGES - 1;
            p ^= 1u;
          }
          wait_bar<EK>(smem_u32(&full[st]), p, abort_flag, P.status, 50ull * 1000 * 1000);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t IDESC = instr_desc(BM * CG, BN, AMN, BMN);
      int stage = 0;
      uint32_t ph = 0;
      int slot = 0;
      uint32_t sph = 0;
      bool ok = true;
      for (int u = seq.first(); ok && u < P.total_units; u = seq.next(u)) {
        const Work w = decode<CG>(P, u);
        const Prob& pr = P.p[w.pi];
        for (int s = 0; ok && s < nseg; ++s) {
          int kb0, nkb, opair;
          segment<EK>(P, pr, w, s, kb0, nkb, opair);
          const bool fresh = !(EK == K_CHAIN && s == 1);
          if (fresh) {
            if (!wait_bar<EK>(smem_u32(&acce[slot]), sph ^ 1u, abort_flag, P.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(slot * BN);
          for (int i = 0; i < nkb; ++i) {
            if (!wait_bar<EK>(smem_u32(&full[stage]), ph, abort_flag, P.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = smem_desc(sa + (AMN ? kk * 2048 : kk * 32), AMN);
              const uint64_t bd = smem_desc(sb + (BMN ? kk * 2048 : kk * 32), BMN);
              mma_bf16<CG>(d_tmem, ad, bd, IDESC, (fresh && i == 0 && kk == 0) ? 0u : 1u);
            }
            mma_commit<CG>(smem_u32(&empty[stage]));
            if (++stage == C::STAGES) {
              stage = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if (!(EK == K_CHAIN && s == 0)) {
            // each segment's accumulator (for Online RMSNorm: each shard's partial
            // product) takes the next slot of the ring
            mma_commit<CG>(smem_u32(&accf[slot]));
            if (++slot == C::NSLOT) {
              slot = 0;
              sph ^= 1u;
            }
          }
        }
      }
      // every MMA issued must complete before TMEM is released
      mma_commit_local<CG>(smem_u32(drain));
      wait_bar<EK>(smem_u32(drain), 0, abort_flag, P.status, ok ? kWaitLimitNs : 50ull * 1000 * 1000);
    }
  } else if (warp == epi_warp0<EK>() + NUM_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue-input producer
    if (E::NIN > 0 && lane == 0) {
      int e = 0;
      uint32_t eph = 0;
      int issued = 0;
      bool ok = !can_consume<EK>() || P.in.entered == nullptr ||
                wait_count(P.in.entered, P.in.entered_target, abort_flag, P.status);
      if (can_consume<EK>() && ok && P.in.entered != nullptr) fence_proxy_async_global();
      for (int u = seq.first(); ok && u < P.total_units; u = seq.next(u)) {
        const Work w = decode<CG>(P, u);
        const Prob& pr = P.p[w.pi];
        const int m0 = static_cast<int>(w.m0) + row_off;
        const int n0 = static_cast<int>(w.nb) * BN;
        for (int c = 0; c < NCH; ++c) {
          if (!wait_bar<EK>(smem_u32(&epi_empty[e]), eph ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&epi_full[e]);
          mbar_expect_tx(fb, E::NIN * E::SUB_BYTES);
#pragma unroll
          for (int k = 0; k < E::NIN; ++k)
            tma_load_2d(smem_u32(epi + (e * E::NT + k) * E::SUB_BYTES), &pr.mi[k], n0 + c * EPI_N,
                        m0, fb);
          ++issued;
          if (++e == E::NE) {
            e = 0;
            eph ^= 1u;
          }
        }
      }
      if (!ok) {
        // drain the loads in flight before the CTA exits
        int st = e;
        uint32_t p = eph;
        for (int i = 0; i < E::NE && i < issued; ++i) {
          if (--st < 0) {
            st = E::NE - 1;
            p ^= 1u;
          }
          wait_bar<EK>(smem_u32(&epi_full[st]), p, abort_flag, P.status, 50ull * 1000 * 1000);
        }
      }
    }
  }  // Online RMSNorm: warps 2 and 3 only lend their registers
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (is_fold<EK>()) setmaxnreg_inc<kNormRegsHigh>();
    const int q = warp & 3;                 // TMEM lane quarter = tile rows 32q .. 32q + 31
    const int grp = (warp - epi_warp0<EK>()) >> 2;  // this warp's subtiles: c % EPI_GROUPS == grp
    constexpr int MYCH = NCH / EPI_GROUPS;  // subtiles per warp per tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int slot = 0;
    uint32_t sph = 0;
    int prev_e = 0, mine = 0;
    int64_t tile_no = 0;                    // tiles this CTA has finished
    bool ok = true;
    auto acquire = [&](int sl, uint32_t p) -> bool {
      if (!wait_bar<EK>(smem_u32(&accf[sl]), p, abort_flag, P.status)) return false;
      tc_fence_after();
      return true;
    };
    auto release = [&](int sl) {  // on the leader's barrier: its MMA warp refills the slot
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 1 || leader)
          mbar_arrive(smem_u32(&acce[sl]));
        else
          mbar_arrive_cluster(mapa(smem_u32(&acce[sl]), 0));
      }
    };
    auto advance = [&]() {
      if (++slot == C::NSLOT) {
        slot = 0;
        sph ^= 1u;
      }
    };
    // Chained producer: once this warp's stores of a tile have landed, count
    // them for the tile's row block (the next launch reads those rows). Online
    // RMSNorm's epilogue, which must drain the next tile's shards while the MMAs
    // run on, counts a tile when it is about to store the next one (or exits),
    // by when the stores have long landed; the other kinds wait for their
    // stores at the end of the tile, hidden behind the next tile's long K loop.
    int64_t pending_rb = -1;
    auto signal_pending = [&]() {
      if (!can_produce<EK>() || pending_rb < 0) return;
      if (lane == 0) {
        bulk_wait_all();
        fence_proxy_async_global();
        red_release_add(P.out.rows + pending_rb, 1);
      }
      __syncwarp();
      pending_rb = -1;
    };
    auto signal_rows = [&](const Work& w) {
      if (can_produce<EK>() && P.out.rows != nullptr) pending_rb = w.m0 / (BM * CG);
    };
    // (a chained consumer's epilogue needs no wait of its own: it touches global
    // memory only after its accumulators are complete, i.e. after the operand
    // producer's waits)
    for (int u = seq.first(); ok && u < P.total_units; u = seq.next(u), ++tile_no) {
      const Work w = decode<CG>(P, u);
      const Prob& pr = P.p[w.pi];
      const int64_t row = w.m0 + row_off + q * 32 + lane;
      const int64_t n0 = w.nb * BN;
      const int64_t M = pr.M, N = pr.N;
      const bool row_ok = row < M;
      uint32_t gpk[EK == K_SWIGLU ? MYCH : 1][16];  // SwiGLU: this warp's G, bf16 pairs
      int sl0 = slot, sl1 = slot;  // TMEM slot(s) of this tile's accumulator(s)
      if constexpr (is_fold<EK>()) {
        // Shard s's partial product P_s arrives in the next TMEM slot of the
        // ring; the epilogue folds it into the running sum R, kept in registers
        // (this thread's row, this group's columns). Online RMSNorm (K_NORM with
        // the sums of squares in rowv) folds R += alpha_s * (P_s / rms_s): local
        // normalisation, then the per-row correction alpha_s = rms_s / rms_g.
        // Otherwise R += P_s: the plain sum of the shards' partials. The slot is
        // free again as soon as P_s is in registers, so the MMAs of shard s + 1
        // run during the fold.
        const int S = P.S;
        const bool norm = EK == K_NORM && pr.rowv != nullptr;
        const float* ss = norm ? pr.rowv + (row_ok ? row : 0) * S : nullptr;
        float tot = 0.f;
        if (norm)
          for (int s = 0; s < S; ++s) tot += row_ok ? ss[s] : 0.f;
        const float shard_w = static_cast<float>(pr.K / S);
        const float rms_g = sqrtf(tot / static_cast<float>(pr.K) + P.eps);
        float R[MYCH][32];
        for (int s = 0; s < S; ++s) {
          const int sl = slot;
          if (!acquire(sl, sph)) {
            ok = false;
            break;
          }
          advance();
          float inv_local = 1.f, alpha = 1.f;
          if (norm) {
            const float ss_s = row_ok ? ss[s] : 0.f;
            const float rms_s = sqrtf(ss_s / shard_w + P.eps);
            inv_local = 1.0f / rms_s;
            alpha = rms_s / rms_g;
          }
          const uint32_t tP = tmem + lane_base + static_cast<uint32_t>(sl * BN);
#pragma unroll
          for (int k = 0; k < MYCH; ++k) {
            float v[32];
            tmem_ld32(tP + static_cast<uint32_t>((k * EPI_GROUPS + grp) * 32), v);
            if (k == MYCH - 1) release(sl);  // every column of P_s is in registers
            if (s == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) R[k][i] = alpha * (v[i] * inv_local);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) R[k][i] = fmaf(alpha, v[i] * inv_local, R[k][i]);
            }
          }
        }
        if (!ok) break;
        signal_pending();
        const int rt = static_cast<int>(w.m0) + row_off + q * 32;
        if constexpr (EK == K_SDSIGMA) {
          // dz = (sum over shards of dY_s B_s) * sigma'(z) * rowv
          const float rs = (pr.rowv != nullptr && row_ok) ? pr.rowv[row] : 1.f;
#pragma unroll
          for (int k = 0; k < MYCH; ++k) {
            // one chunk's z at a time: its loads stay below the previous chunk's
            // stores (the running sum already holds 128 registers)
            asm volatile("" ::: "memory");
            const int c = k * EPI_GROUPS + grp;
            const int64_t col0 = n0 + c * EPI_N;
            const int e = static_cast<int>((tile_no * NCH + c) % E::NE);
            uint8_t* ent = epi + e * E::NT * E::SUB_BYTES + q * E::WARP_BYTES;
            float v[32];  // z, then dz in place
            ld_row32_bf16(static_cast<const __nv_bfloat16*>(pr.in_raw), pr.ldi_raw, row, row_ok,
                          col0, N, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (R[k][i] * act_grad_fast(v[i], P.sigma)) * rs;
            smem_row_store_bf16(ent, lane, v);
            if (row_ok && col0 + EPI_N > pr.N8 && col0 < N)
              store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, v);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              if (rt < M && col0 < pr.N8)
                tma_store_2d(&pr.mo[0], smem_u32(ent), static_cast<int>(col0), rt);
              bulk_commit();
              bulk_wait_read<E::NE / EPI_GROUPS - 1>();
            }
            __syncwarp();
          }
          signal_rows(w);
          continue;  // the tile is done
        }
#pragma unroll
        for (int k = 0; k < MYCH; ++k) {
          const int c = k * EPI_GROUPS + grp;
          const int64_t col0 = n0 + c * EPI_N;
          const int e = static_cast<int>((tile_no * NCH + c) % E::NE);
          uint8_t* ent = epi + e * E::NT * E::SUB_BYTES + q * E::WARP_BYTES;
          uint32_t zpk[16], hpk[16];  // z = R rounded to bf16, h = sigma(z): bf16 pairs
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(R[k][2 * i], R[k][2 * i + 1]);
            zpk[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float z0 = __uint_as_float(zpk[i] << 16);
            const float z1 = __uint_as_float(zpk[i] & 0xFFFF0000u);
            const __nv_bfloat162 h = __floats2bfloat162_rn(act_fast(z0, P.sigma), act_fast(z1, P.sigma));
            hpk[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
          smem_row_store_packed(ent, lane, zpk);
          smem_row_store_packed(ent + E::SUB_BYTES, lane, hpk);
          if (row_ok && col0 + EPI_N > pr.N8 && col0 < N) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              f[2 * i] = __uint_as_float(zpk[i] << 16);
              f[2 * i + 1] = __uint_as_float(zpk[i] & 0xFFFF0000u);
            }
            if (pr.out_mask & 1) store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, f);
            if (pr.out_mask & 2) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                f[2 * i] = __uint_as_float(hpk[i] << 16);
                f[2 * i + 1] = __uint_as_float(hpk[i] & 0xFFFF0000u);
              }
              store_tail_bf16(pr.out[1], pr.ldo[1], row, col0, pr.N8, N, f);
            }
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (rt < M && col0 < pr.N8) {
              if (pr.out_mask & 1)
                tma_store_2d(&pr.mo[0], smem_u32(ent), static_cast<int>(col0), rt);
              if (pr.out_mask & 2)
                tma_store_2d(&pr.mo[1], smem_u32(ent + E::SUB_BYTES), static_cast<int>(col0), rt);
            }
            bulk_commit();
            bulk_wait_read<E::NE / EPI_GROUPS - 1>();
          }
          __syncwarp();
        }
        signal_rows(w);
        continue;  // the tile is done
      } else if constexpr (EK == K_SWIGLU) {
        sl0 = slot;
        const uint32_t p0 = sph;
        advance();
        sl1 = slot;
        const uint32_t p1 = sph;
        advance();
        // G first: keep this warp's columns of it as bf16 pairs and free its slot
        // at once, so the MMAs of the next tile's G overlap this tile's epilogue
        if (!acquire(sl0, p0)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < MYCH; ++k) {
          float g[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(sl0 * BN + (k * EPI_GROUPS + grp) * 32),
                    g);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * i], g[2 * i + 1]);
            gpk[k][i] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
        release(sl0);
        // store G while the MMAs of U run: each chunk goes to subtile 0 of its ring
        // entry; U (subtile 1) and m (subtile 0 again) follow once U has arrived
        if (pr.out_mask & 1) {
          const int rt = static_cast<int>(w.m0) + row_off + q * 32;
#pragma unroll
          for (int k = 0; k < MYCH; ++k) {
            const int c = k * EPI_GROUPS + grp;
            const int64_t col0 = n0 + c * EPI_N;
            const int e = static_cast<int>((tile_no * NCH + c) % E::NE);
            uint8_t* ent = epi + e * E::NT * E::SUB_BYTES + q * E::WARP_BYTES;
            smem_row_store_packed(ent, lane, gpk[k]);
            if (row_ok && col0 + EPI_N > pr.N8 && col0 < N) {
              float g[32];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                g[2 * i] = __uint_as_float(gpk[k][i] << 16);
                g[2 * i + 1] = __uint_as_float(gpk[k][i] & 0xFFFF0000u);
              }
              store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, g);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              if (rt < M && col0 < pr.N8)
                tma_store_2d(&pr.mo[0], smem_u32(ent), static_cast<int>(col0), rt);
              bulk_commit();
              bulk_wait_read<E::NE / EPI_GROUPS - 1>();
            }
            __syncwarp();
          }
        }
        if (!acquire(sl1, p1)) {
          ok = false;
          break;
        }
        // U: all of this warp's columns into registers too, then its slot is free
        // and the MMAs run a tile ahead while m = SiLU(G) * U is formed and stored
        uint32_t upk[MYCH][16];
#pragma unroll
        for (int k = 0; k < MYCH; ++k) {
          float u[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(sl1 * BN + (k * EPI_GROUPS + grp) * 32),
                    u);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(u[2 * i], u[2 * i + 1]);
            upk[k][i] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
        release(sl1);
        const int rt = static_cast<int>(w.m0) + row_off + q * 32;
#pragma unroll
        for (int k = 0; k < MYCH; ++k) {
          const int c = k * EPI_GROUPS + grp;
          const int64_t col0 = n0 + c * EPI_N;
          const int e = static_cast<int>((tile_no * NCH + c) % E::NE);
          uint8_t* ent = epi + e * E::NT * E::SUB_BYTES + q * E::WARP_BYTES;
          uint32_t mpk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(gpk[k][i] << 16);
            const float g1 = __uint_as_float(gpk[k][i] & 0xFFFF0000u);
            const float u0 = __uint_as_float(upk[k][i] << 16);
            const float u1 = __uint_as_float(upk[k][i] & 0xFFFF0000u);
            const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(silu_fast(g0), u0),
                                                           __fmul_rn(silu_fast(g1), u1));
            mpk[i] = *reinterpret_cast<const uint32_t*>(&h);
          }
          // U in subtile 1, m in subtile 0: G's store from it was issued before
          // every later bulk group of this warp, and each commit below waits for
          // all but the newest group to have left shared memory
          smem_row_store_packed(ent + E::SUB_BYTES, lane, upk[k]);
          smem_row_store_packed(ent, lane, mpk);
          if (row_ok && col0 + EPI_N > pr.N8 && col0 < N) {
            float f[32];
            if (pr.out_mask & 2) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                f[2 * i] = __uint_as_float(upk[k][i] << 16);
                f[2 * i + 1] = __uint_as_float(upk[k][i] & 0xFFFF0000u);
              }
              store_tail_bf16(pr.out[1], pr.ldo[1], row, col0, pr.N8, N, f);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              f[2 * i] = __uint_as_float(mpk[i] << 16);
              f[2 * i + 1] = __uint_as_float(mpk[i] & 0xFFFF0000u);
            }
            store_tail_bf16(pr.out[2], pr.ldo[2], row, col0, pr.N8, N, f);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (rt < M && col0 < pr.N8) {
              if (pr.out_mask & 2)
                tma_store_2d(&pr.mo[1], smem_u32(ent + E::SUB_BYTES), static_cast<int>(col0), rt);
              if (pr.out_mask & 4)
                tma_store_2d(&pr.mo[2], smem_u32(ent), static_cast<int>(col0), rt);
            }
            bulk_commit();
            bulk_wait_read<E::NE / EPI_GROUPS - 1>();
          }
          __syncwarp();
        }
        continue;  // the tile is done
      } else {
        sl0 = slot;
        if (!acquire(slot, sph)) {
          ok = false;
          break;
        }
        advance();
      }
      float rs = 1.f;
      if ((EK == K_STORE || EK == K_CHAIN || EK == K_DSIGMA || EK == K_DSWIGLU) &&
          pr.rowv != nullptr && row_ok)
        rs = pr.rowv[row];

#pragma unroll 1
      for (int k = 0; k < MYCH; ++k) {
        const int c = k * EPI_GROUPS + grp;            // subtile within the tile
        const int64_t col0 = n0 + c * EPI_N;
        const int64_t j = tile_no * NCH + c;           // subtile sequence number of this CTA
        const int e = static_cast<int>(j % E::NE);
        const uint32_t eph = static_cast<uint32_t>((j / E::NE) & 1);
        if (E::NIN > 0) {
          if (!wait_bar<EK>(smem_u32(&epi_full[e]), eph, abort_flag, P.status)) {
            ok = false;
            break;
          }
        }
        float zin[EK == K_DSIGMA ? 32 : 1];
        if constexpr (EK == K_DSIGMA)  // issued first: in flight during the TMEM load
          ld_row32_bf16(static_cast<const __nv_bfloat16*>(pr.in_raw), pr.ldi_raw, row, row_ok,
                        col0, N, zin);
        float v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(sl0 * BN + c * 32), v);
        if (k == MYCH - 1) release(sl0);
        uint8_t* ent = epi + e * E::NT * E::SUB_BYTES + q * E::WARP_BYTES;
        if (EK == K_STORE && w.part_slot >= 0) {
          // fp32 partial tile of a split unit, written in whole 128-byte rows: this
          // warp's 32 x 32 block goes through its ring entry, 16 rows at a time,
          // transposed so that lane = column. A split unit issues no TMA stores;
          // the ones still reading the ring from earlier units are waited for once.
          if (k == 0) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
          float* dst = P.part + (static_cast<int64_t>(w.part_slot) * CG * BM + row_off + q * 32) * BN +
                       c * 32 + lane;
          auto cell = [&](int rr, int col) -> float* {  // row rr, column col of the block
            return reinterpret_cast<float*>(ent + rr * 128 + ((((col >> 2) ^ (rr & 7)) << 4) |
                                                              ((col & 3) << 2)));
          };
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            if ((lane >> 4) == h) {
              const int rr = lane & 15;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(cell(rr, 4 * i)) =
                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            __syncwarp();
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
              dst[static_cast<int64_t>(h * 16 + rr) * BN] = *cell(rr, lane);
            __syncwarp();
          }
          continue;  // summed, scaled and stored by the reduction kernel
        }
        // this row holds some of the ragged columns [N8, N)
        const bool tail = row_ok && col0 + EPI_N > pr.N8 && col0 < N;
        if constexpr (EK == K_STORE || EK == K_CHAIN) {
          if (pr.colv != nullptr) {
            float cv[32];
            ld_vec_bf16(static_cast<const __nv_bfloat16*>(pr.colv), col0, N, cv);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= cv[i];
          }
          if (pr.rowv != nullptr) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= rs;
          }
          smem_row_store_bf16(ent, lane, v);
          if (tail) store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, v);
        } else if constexpr (EK == K_SIGMA || EK == K_NORM) {
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = round_to<__nv_bfloat16>(v[i]);
            h[i] = act_fast(v[i], P.sigma);
          }
          smem_row_store_bf16(ent, lane, v);
          smem_row_store_bf16(ent + E::SUB_BYTES, lane, h);
          if (tail) {
            store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, v);
            if (pr.out_mask & 2) store_tail_bf16(pr.out[1], pr.ldo[1], row, col0, pr.N8, N, h);
          }
        } else if constexpr (EK == K_RESID) {
          float r[32];
          smem_row_load_bf16(ent, lane, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += r[i];
          smem_row_store_bf16(ent, lane, v);
          if (tail) store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, v);
        } else if constexpr (EK == K_DSIGMA) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (v[i] * act_grad_fast(zin[i], P.sigma)) * rs;
          smem_row_store_bf16(ent, lane, v);
          if (tail) store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, v);
        } else if constexpr (EK == K_DSWIGLU) {
          float G[32], U[32];
          smem_row_load_bf16(ent, lane, G);
          smem_row_load_bf16(ent + E::SUB_BYTES, lane, U);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float sg = sigmoid_fast(G[i]);
            const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(G[i], __fsub_rn(1.0f, sg))));
            U[i] = ((v[i] * U[i]) * dsilu) * rs;          // dG
            G[i] = (v[i] * __fmul_rn(G[i], sg)) * rs;     // dU
          }
          smem_row_store_bf16(ent, lane, U);
          smem_row_store_bf16(ent + E::SUB_BYTES, lane, G);
          if (tail) {
            store_tail_bf16(pr.out[0], pr.ldo[0], row, col0, pr.N8, N, U);
            store_tail_bf16(pr.out[1], pr.ldo[1], row, col0, pr.N8, N, G);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          const uint32_t src = smem_u32(ent);
          const int rt = static_cast<int>(w.m0) + row_off + q * 32;  // row within the problem
          if (rt < M && col0 < pr.N8) {  // boxes partly outside the tensor are clipped by TMA
#pragma unroll
            for (int o = 0; o < E::NOUT; ++o)
              if (pr.out_mask & (1 << o))
                tma_store_2d(&pr.mo[o], src + o * E::SUB_BYTES, static_cast<int>(col0), rt);
          }
          bulk_commit();
          // a warp reuses a ring entry every NE / EPI_GROUPS of its own subtiles: the
          // stores issued from that entry must have left shared memory by then
          bulk_wait_read<E::NE / EPI_GROUPS - 1>();
          if (E::NIN > 0 && mine > 0) mbar_arrive(smem_u32(&epi_empty[prev_e]));
        }
        __syncwarp();
        prev_e = e;
        ++mine;
      }
      if (ok) {
        signal_rows(w);
        signal_pending();
      }
    }
    if (ok) signal_pending();
    if (lane == 0) {
      bulk_wait_read<0>();
      if (E::NIN > 0 && mine > 0) mbar_arrive(smem_u32(&epi_empty[prev_e]));
      bulk_wait_all();
    }
    __syncwarp();
    if constexpr (is_fold<EK>()) setmaxnreg_dec<kNormRegsLow>();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the leader's MMAs and the peer's arrivals are done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, 512);
  }
}

}  // namespace tc
}  // namespace bn
