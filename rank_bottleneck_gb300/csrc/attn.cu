// Attention core on the tcgen05 tensor cores (sm_103a): exact multi-head
// softmax attention, causal or not, forward and backward, d_head = 128.
//
// The project page of BOOST places the attention core between the grouped
// Q/K/V up-projection and the O projection of the decoder block (section
// "Move the chunk boundary to the bottleneck", the decoder-block figure); the
// paper summary page cites FlashAttention for it. The arithmetic is the
// FlashAttention one: the forward keeps a running row maximum and sum (online
// softmax) and writes the row log-sum-exp; the backward recomputes the
// probabilities from it.
//
// One kernel template, three modes, all built on one tile shape: a stationary
// 128-row tile (one row per TMEM lane and per epilogue thread) and a stream of
// 128-row blocks of the other side, d_head = 128.
//   FWD   stationary Q;        blocks K_j, V_j.   S = Q K_j^T (TMEM), online
//         softmax in registers (the two warps of a row exchange their partial
//         row maxima through shared memory), P (bf16 pairs) written over the
//         warp's own S columns, O += P V_j in TMEM with P as the A operand;
//         O is rescaled in place only when a row maximum grows by more than
//         2^8 (lazy rescale), and divided by the row sum at the end.
//   BKV   stationary K and V;  blocks Q_i, dO_i.  S^T = K Q_i^T, dP^T = V dO_i^T;
//         dP^T is read into registers and its buffer handed back; P^T and dS^T
//         (bf16 pairs) are written into TMEM over the S^T columns already read,
//         and dV += P^T dO_i, dK += dS^T Q_i take them from there (A operand in
//         TMEM), which leaves shared memory for a two-stage ring.
//   BQ    stationary Q and dO; blocks K_j, V_j.   S = Q K_j^T, dP = dO V_j^T,
//         dQ += dS K_j in TMEM with dS (bf16 pairs) written into S's buffer
//         and read from there as the A operand. dP is read into registers
//         first and its single TMEM buffer handed back, so the next block's dP
//         runs during this block's softmax; the K ring is three deep.
// Per CTA (320 threads, persistent over the tiles, one CTA per SM):
//   warp 0      TMA producer: the stationary tile(s), then rings of streamed
//               blocks (K and V, or BKV's Q and dO, two stages each, BQ's K
//               three), in BKV with the blocks' row terms; in FWD and BQ a
//               second lane loads the V ring on its own barriers;
//   warp 1      TMEM owner (512 columns) and, from one thread, the MMA issuer;
//   warps 2..9  elementwise: warp w owns TMEM lanes 32 (w % 4) .. + 31 (one
//               tile row per thread) and one column half of every block.
// TMEM columns: S in two or three buffers so that the next blocks' S = Q K^T
// run while the current block's softmax does:
//   FWD  [0, 384) S (then P) of block buffers 0, 1 and 2; [384, 512) O
//   BKV  [0, 128) S^T (then P^T, dS^T); [128, 256) dP^T; [256, 384) dV; [384, 512) dK
//   BQ   [0, 256) S (then dS) of block buffers 0 and 1; [256, 384) dP (single); [384, 512) dQ
// Every operand is bf16 in 128-byte-swizzled shared memory: K-major for the
// S and dP products (rows of 64 elements per 128-byte line), and the streamed
// blocks' same bytes read MN-major for the accumulating products (the 64
// d_head columns of a line are the N dimension, the block's rows are K).
// Every mbarrier wait is bounded (kWaitLimitNs): on expiry the kernel records
// a timeout in the status word and every role unwinds.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "attn.h"
#include "tc_ptx.cuh"

namespace bn {
namespace attn {

using namespace tc;

constexpr int DH = 128;      // head width
constexpr int BR = 128;      // rows of the stationary tile
constexpr int BCF = 128;     // rows of a streamed block
constexpr int NTHREADS = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 elementwise
constexpr int SUB_R = BR * 128;          // one 64-column half of a stationary tile: 16 KB
constexpr int XTILE = 2 * SUB_R;         // a stationary tile: 32 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Mode : int { FWD = 0, BKV = 1, BQ = 2 };

template <int MODE>
struct Lay {
  static constexpr int BCM = BCF;                       // rows of a streamed block
  static constexpr int SUBC = BCM * 128;              // a 64-column (d_head) half of a streamed block
  static constexpr int HALF = 2 * SUBC;               // one streamed block (both d_head halves)
  static constexpr int EB = BR * BCM * 2;             // one bf16 elementwise tile [128, BCM]
  static constexpr int NX = (MODE == FWD) ? 1 : 2;   // stationary tiles
  // elementwise tiles in shared memory: none (the forward keeps P, the backward
  // P^T, dS^T and dS in TMEM, over the score columns already read)
  static constexpr int NE = 0;
  // buffers of each elementwise tile: the forward's P and dQ's dS are single
  // (shared memory); the softmax waits for the previous block's product first
  static constexpr int NPB = (MODE == BKV) ? 2 : 1;
  // Rings of streamed blocks, one for each operand half: FWD and BQ K (first)
  // and V (second), BKV Q and dO (filled and freed together). BQ's K ring is
  // three deep: K_j is read last by the dQ product, so a two-deep ring could
  // refill it only after that product.
  static constexpr int NSTK = (MODE == BQ) ? 3 : 2;
  static constexpr int NSTV = 2;
  static constexpr int AUXB = (MODE == BKV) ? 2 * BCM * 4 : 0;  // BKV: a block's lse log2 e and D
  static constexpr int X_OFF = 0;
  static constexpr int Y_OFF = X_OFF + NX * XTILE;
  static constexpr int E_OFF = Y_OFF + (NSTK + NSTV) * HALF;
  static constexpr int AUX_OFF = E_OFF + NE * NPB * EB;
  static constexpr int XCH_OFF = AUX_OFF + NSTK * AUXB;
  // FWD: row sums exchanged between the two warps of a row, [2 tile parity][2 half][128],
  // then each block's row maxima, [2 block parity][2 half][128]
  static constexpr int BAR_OFF = XCH_OFF + ((MODE == FWD) ? 2 * 2 * 2 * BR * 4 : 0);
  // stage barriers: the two halves of a FWD or BQ stage are filled and freed
  // apart (FWD: K after S, V after P V; BQ: V after dP, K after dQ), BKV's
  // stage as a whole
  static constexpr int NYB = (MODE == BKV) ? NSTK : NSTK + NSTV;
  // TMEM buffers of the scores (then P or dS): the forward's three let the MMA
  // thread issue the score products two blocks ahead of the softmax
  static constexpr int NSB = (MODE == FWD) ? 3 : 2;
  // barriers (2 + 2 NYB + 3 NSB + 21 of 8 bytes), the TMEM address and the abort flag
  static constexpr int BAR_BYTES = (2 + 2 * NYB + 3 * NSB + 21) * 8 + 8 <= 256 ? 256 : 512;
  static constexpr int BYTES = BAR_OFF + BAR_BYTES;
  static constexpr int SMEM = 1024 + BYTES;
  static_assert(E_OFF % 1024 == 0, "elementwise tiles must be 1024-byte aligned");
  static_assert(SMEM <= 232448, "shared memory over the per-CTA limit");
};

struct Params {
  CUtensorMap mx[2];  // stationary operands: boxes of 64 columns x 128 rows
  CUtensorMap my[2];  // streamed operands: boxes of 64 columns x 64 rows
  int B, L, H, Lp;
  int causal;
  int ntiles;
  float scale;        // 1 / sqrt(d_head)
  float scale_log2;   // scale * log2(e)
  __nv_bfloat16* out0;  // FWD: o; BKV: dv
  __nv_bfloat16* out1;  // BKV: dk; BQ: dq
  float* lse;           // FWD: [B H, Lp]
  const float* l2;      // backward: lse * log2(e), [B H, Lp]
  const float* dd;      // backward: D = rowsum(dO * O), [B H, Lp]
  int* status;
  int unfed;            // test hook: the first stationary tile is never loaded
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// contiguous global -> shared copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// 2^x with the hardware approximation (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 16 32-bit columns into this thread's TMEM lane (completion: tcgen05.wait::st)
__device__ __forceinline__ void tmem_st16u_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                     int* status, unsigned long long limit = kWaitLimitNs) {
  return wait_bar_call(bar, parity, abort_flag, status, limit);
}

// Tile u -> (stationary tile index, sequence*head). Causal tiles are dealt
// heaviest first: query tiles from the end of the sequence, key tiles from
// its start.
template <int MODE>
__device__ __forceinline__ void decode(const Params& P, int u, int& t, int& bh) {
  const int BH = P.B * P.H;
  const int nt = (P.L + BR - 1) / BR;
  bh = u % BH;
  t = (MODE == BKV) ? u / BH : nt - 1 - u / BH;
}
// streamed blocks [first, last) of tile t
template <int MODE>
__device__ __forceinline__ void blocks(const Params& P, int t, int& first, int& last) {
  constexpr int bcm = Lay<MODE>::BCM;
  const int nb = (P.L + bcm - 1) / bcm;
  if (MODE == BKV) {
    first = P.causal ? (t * BR) / bcm : 0;
    last = nb;
  } else {
    first = 0;
    last = P.causal ? min(nb, (t * BR + BR) / bcm) : nb;
  }
}

// One thread's 32 bf16 values (16 packed pairs) into row r, 16-byte chunks
// 4 h .. 4 h + 3, of a 128-row x 128-byte tile with the 128-byte swizzle.
__device__ __forceinline__ void put_row32(uint8_t* tile, int r, int h, const uint32_t* pk) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
// 32 fp32 values as bf16 to global memory (16-byte aligned)
__device__ __forceinline__ void store32(__nv_bfloat16* dst, const float* v, float s) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 u;
    u.x = pack2(v[8 * c] * s, v[8 * c + 1] * s);
    u.y = pack2(v[8 * c + 2] * s, v[8 * c + 3] * s);
    u.z = pack2(v[8 * c + 4] * s, v[8 * c + 5] * s);
    u.w = pack2(v[8 * c + 6] * s, v[8 * c + 7] * s);
    *reinterpret_cast<uint4*>(dst + 8 * c) = u;
  }
}

template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1) attn_kernel(const __grid_constant__ Params P) {
  using LY = Lay<MODE>;
  constexpr int BCM = LY::BCM, SUBC = LY::SUBC, HALF = LY::HALF;
  // forward: S buffers take TMEM columns [0, 3 BCM), O the 128 columns after them
  constexpr int NSB = LY::NSB;
  constexpr int OCOL = NSB * BCM;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sX = smem + LY::X_OFF;
  uint8_t* sYK = smem + LY::Y_OFF;                  // first-half ring (K; BKV: Q)
  uint8_t* sYV = sYK + LY::NSTK * HALF;              // second-half ring (V; BKV: dO)
  float* sAux = reinterpret_cast<float*>(smem + LY::AUX_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
  uint64_t* x_full = bars;
  uint64_t* x_empty = bars + 1;
  uint64_t* y_full = bars + 2;                // [NYB] (FWD, BQ: K ring, then V ring)
  uint64_t* y_empty = y_full + LY::NYB;       // [NYB]
  uint64_t* s_full = y_empty + LY::NYB;       // [NSB] scores of the buffer's block ready
  uint64_t* e_full = s_full + NSB;            // [NSB] P / dS (BKV: P^T, dS^T) written
  uint64_t* e_empty = e_full + NSB;           // [NSB] the accumulating products that read them
                                              //       done (the buffer is free again)
  uint64_t* a_full = e_empty + NSB;           // backward: [0] the tile's sums done, [1] dP ready
  uint64_t* a_empty = a_full + 2;             // FWD: [0] O read out;
                                              // backward: [0] sums read out, [1] dP read
  uint64_t* drain = a_empty + 2;
  uint64_t* lx = drain + 1;                   // FWD [4 row quarters][2 tile parity]: row sums exchanged
  uint64_t* mxb = lx + 8;                     // FWD [4 row quarters][2 block parity]: row maxima exchanged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mxb + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(x_full), 1);
    mbar_init(smem_u32(x_empty), 1);
    for (int i = 0; i < LY::NYB; ++i) {
      mbar_init(smem_u32(&y_full[i]), 1);
      mbar_init(smem_u32(&y_empty[i]), 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&e_full[i]), 8);
      mbar_init(smem_u32(&e_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&a_full[i]), 1);
      mbar_init(smem_u32(&a_empty[i]), 8);
    }
    mbar_init(smem_u32(drain), 1);
    for (int i = 0; i < 8; ++i) mbar_init(smem_u32(&lx[i]), 64);
    for (int i = 0; i < 8; ++i) mbar_init(smem_u32(&mxb[i]), 64);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<1>(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 loads the stationary tiles and the streamed blocks; in FWD and BQ
    // lane 1 loads the V blocks on their own barriers, so that each half of a
    // stage is refilled as soon as its last reader is done (FWD: K after S;
    // BQ: V after dP).
    if (lane == 0 || (MODE != BKV && lane == 1)) {
      const bool vlane = MODE != BKV && lane == 1;
      for (int i = 0; i < LY::NX; ++i) tma_prefetch_desc(&P.mx[i]);
      for (int i = 0; i < 2; ++i) tma_prefetch_desc(&P.my[i]);
      bool ok = true;
      uint32_t tn = 0, jn = 0;
      uint32_t x_loads = 0;
      for (int u = blockIdx.x; ok && u < P.ntiles; u += gridDim.x, ++tn) {
        int t, bh, first, last;
        decode<MODE>(P, u, t, bh);
        blocks<MODE>(P, t, first, last);
        const int b = bh / P.H, col = (bh % P.H) * DH;
        if (!vlane) {
          if (!bwait(smem_u32(x_empty), (tn & 1u) ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          if (P.unfed) {  // (test hook) the MMA's wait for this tile must run out
            ok = false;
            break;
          }
          const uint32_t xb = smem_u32(x_full);
          mbar_expect_tx(xb, LY::NX * XTILE);
          for (int i = 0; i < LY::NX; ++i)
            for (int c = 0; c < 2; ++c)
              tma_load_3d(smem_u32(sX + i * XTILE + c * SUB_R), &P.mx[i], col + 64 * c, t * BR,
                          b, xb);
          ++x_loads;
        }
        for (int j = first; j < last; ++j, ++jn) {
          const int st = vlane ? static_cast<int>(jn % LY::NSTV) : static_cast<int>(jn % LY::NSTK);
          const uint32_t par = vlane ? (jn / LY::NSTV) & 1u : (jn / LY::NSTK) & 1u;
          const int bi = vlane ? LY::NSTK + st : st;  // this lane's barrier of the stage
          if (!bwait(smem_u32(&y_empty[bi]), par ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          const uint32_t yb = smem_u32(&y_full[bi]);
          if constexpr (MODE != BKV) {
            // one block of K (lane 0) or of V (lane 1)
            const int i = vlane ? 1 : 0;
            uint8_t* dst = (vlane ? sYV : sYK) + st * HALF;
            mbar_expect_tx(yb, HALF);
            for (int c = 0; c < 2; ++c)
              tma_load_3d(smem_u32(dst + c * SUBC), &P.my[i], col + 64 * c, j * BCM, b, yb);
          } else {
            mbar_expect_tx(yb, 2 * HALF + LY::AUXB);
            for (int i = 0; i < 2; ++i)
              for (int c = 0; c < 2; ++c)
                tma_load_3d(smem_u32((i ? sYV : sYK) + st * HALF + c * SUBC), &P.my[i],
                            col + 64 * c, j * BCM, b, yb);
            if constexpr (MODE == BKV) {
              const int64_t off = static_cast<int64_t>(bh) * P.Lp + j * BCM;
              bulk_load(smem_u32(sAux + st * (LY::AUXB / 4)), P.l2 + off, BCM * 4, yb);
              bulk_load(smem_u32(sAux + st * (LY::AUXB / 4) + BCM), P.dd + off, BCM * 4, yb);
            }
          }
        }
      }
      if (!ok) {
        // the copies in flight must land before the CTA exits
        const unsigned long long lim = 50ull * 1000 * 1000;
        const uint32_t depth = vlane ? LY::NSTV : LY::NSTK;
        for (uint32_t i = 0; i < depth && i < jn; ++i) {
          const uint32_t k = jn - 1 - i;
          const int bi = (vlane ? LY::NSTK : 0) + static_cast<int>(k % depth);
          bwait(smem_u32(&y_full[bi]), (k / depth) & 1u, abort_flag, P.status, lim);
        }
        if (x_loads > 0) bwait(smem_u32(x_full), (x_loads - 1) & 1u, abort_flag, P.status, lim);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = instr_desc(128, BCM, false, false);  // S, dP: K-major B
      constexpr uint32_t ID_A = instr_desc(128, DH, false, true);    // sums: MN-major B
      bool ok = true;
      uint32_t tn = 0, jn = 0;
      // S (and dP) of streamed block number n into TMEM buffer n % NSB
      auto issue_sd = [&](uint32_t n) -> bool {
        const int st = n % LY::NSTK, bf = n % NSB;
        if (!bwait(smem_u32(&y_full[st]), (n / LY::NSTK) & 1u, abort_flag, P.status)) return false;
        // the buffer's previous block: its P (FWD) or dS (BQ), written over its
        // scores, read by that block's accumulating product
        uint64_t* freed = &e_empty[bf];
        if (!bwait(smem_u32(freed), ((n / NSB) & 1u) ^ 1u, abort_flag, P.status)) return false;
        tc_fence_after();
        const uint32_t y = smem_u32(sYK + st * HALF);
        const uint32_t x = smem_u32(sX);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16<1>(tmem + bf * BCM, smem_desc(x + c * SUB_R + kk * 32, false),
                        smem_desc(y + c * SUBC + kk * 32, false), ID_S, (c | kk) ? 1u : 0u);
        mma_commit<1>(smem_u32(&s_full[bf]));
        if constexpr (MODE == FWD) mma_commit<1>(smem_u32(&y_empty[st]));  // K read
        return true;
      };
      // BQ: dP = dO V_n^T of block n into its single TMEM buffer (columns 256..383),
      // once the elementwise warps hold the previous block's dP in registers
      // (a_full[1] / a_empty[1] serve as its full / empty barriers)
      auto issue_dp = [&](uint32_t n) -> bool {
        const int st = n % LY::NSTV;
        if (!bwait(smem_u32(&y_full[LY::NSTK + st]), (n / LY::NSTV) & 1u, abort_flag, P.status))
          return false;
        if (!bwait(smem_u32(&a_empty[1]), (n & 1u) ^ 1u, abort_flag, P.status)) return false;
        tc_fence_after();
        const uint32_t y = smem_u32(sYV + st * HALF);
        const uint32_t x = smem_u32(sX);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16<1>(tmem + 256, smem_desc(x + XTILE + c * SUB_R + kk * 32, false),
                        smem_desc(y + c * SUBC + kk * 32, false), ID_S, (c | kk) ? 1u : 0u);
        mma_commit<1>(smem_u32(&a_full[1]));
        mma_commit<1>(smem_u32(&y_empty[LY::NSTK + st]));  // V read
        return true;
      };
      // BKV: S^T and dP^T of block n into their single TMEM buffers; S^T's buffer
      // is free once block n - 1's dV, dK products (which read P^T, dS^T from it)
      // have completed, dP^T's once the elementwise warps hold dP^T(n - 1)
      auto kv_s = [&](uint32_t n) -> bool {
        const int st = n % LY::NSTK;
        if (!bwait(smem_u32(&y_full[st]), (n / LY::NSTK) & 1u, abort_flag, P.status)) return false;
        if (n > 0 && !bwait(smem_u32(&e_empty[0]), (n - 1) & 1u, abort_flag, P.status))
          return false;
        tc_fence_after();
        const uint32_t y = smem_u32(sYK + st * HALF);
        const uint32_t x = smem_u32(sX);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16<1>(tmem, smem_desc(x + c * SUB_R + kk * 32, false),
                        smem_desc(y + c * SUBC + kk * 32, false), ID_S, (c | kk) ? 1u : 0u);
        mma_commit<1>(smem_u32(&s_full[0]));
        return true;
      };
      auto kv_dp = [&](uint32_t n) -> bool {
        const int st = n % LY::NSTK;
        if (!bwait(smem_u32(&y_full[st]), (n / LY::NSTK) & 1u, abort_flag, P.status)) return false;
        if (!bwait(smem_u32(&a_empty[1]), (n & 1u) ^ 1u, abort_flag, P.status)) return false;
        tc_fence_after();
        const uint32_t y = smem_u32(sYV + st * HALF);
        const uint32_t x = smem_u32(sX);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16<1>(tmem + 128, smem_desc(x + XTILE + c * SUB_R + kk * 32, false),
                        smem_desc(y + c * SUBC + kk * 32, false), ID_S, (c | kk) ? 1u : 0u);
        mma_commit<1>(smem_u32(&a_full[1]));
        return true;
      };
      if constexpr (MODE == BKV) {
        for (int u = blockIdx.x; ok && u < P.ntiles; u += gridDim.x, ++tn) {
          int t, bh, first, last;
          decode<MODE>(P, u, t, bh);
          blocks<MODE>(P, t, first, last);
          if (!bwait(smem_u32(x_full), tn & 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nblk = last - first;
          if (!kv_s(jn) || !kv_dp(jn)) {
            ok = false;
            break;
          }
          for (int i = 0; i < nblk; ++i, ++jn) {
            const int st = jn % LY::NSTK;
            // the next block's dP^T first: it needs only its stage and the warps'
            // copy of this block's dP^T, both early, and so runs during this
            // block's softmax; its S^T must wait for this block's dV, dK products
            if (i + 1 < nblk && !kv_dp(jn + 1)) {
              ok = false;
              break;
            }
            if (!bwait(smem_u32(&e_full[0]), jn & 1u, abort_flag, P.status) ||
                (i == 0 && !bwait(smem_u32(&a_empty[0]), (tn & 1u) ^ 1u, abort_flag, P.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            // dV += P^T dO_i and dK += dS^T Q_i, P^T and dS^T read from TMEM: the
            // 16 queries of k-step kk are warp half kk / 4's chunk (kk % 4) / 2,
            // P^T in that chunk's first 16 columns, dS^T in the next 16
            const uint32_t yq = smem_u32(sYK + st * HALF), ydo = smem_u32(sYV + st * HALF);
            const uint32_t acc = (i > 0) ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BCM / 16; ++kk) {
              const uint32_t pa = tmem + 64 * (kk >> 2) + 32 * ((kk >> 1) & 1) + 8 * (kk & 1);
              mma_bf16_ta(tmem + 256, pa, smem_desc_mn(ydo + kk * 2048, SUBC), ID_A,
                          (acc | kk) ? 1u : 0u);
              mma_bf16_ta(tmem + 384, pa + 16, smem_desc_mn(yq + kk * 2048, SUBC), ID_A,
                          (acc | kk) ? 1u : 0u);
            }
            mma_commit<1>(smem_u32(&e_empty[0]));
            mma_commit<1>(smem_u32(&y_empty[st]));
            if (i + 1 < nblk && !kv_s(jn + 1)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          mma_commit<1>(smem_u32(&a_full[0]));
          mma_commit<1>(smem_u32(x_empty));
        }
      } else
      for (int u = blockIdx.x; ok && u < P.ntiles; u += gridDim.x, ++tn) {
        int t, bh, first, last;
        decode<MODE>(P, u, t, bh);
        blocks<MODE>(P, t, first, last);
        if (!bwait(smem_u32(x_full), tn & 1u, abort_flag, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nblk = last - first;
        // scores issued LA blocks ahead of the accumulating product (FWD: two, into
        // the third S buffer, so that a block's scores never wait behind the
        // product of the block before; BQ: one)
        constexpr int LA = NSB - 1;
        bool pre = true;
        for (int i = 0; pre && i < LA && i < nblk; ++i)
          pre = issue_sd(jn + i) && (MODE != BQ || issue_dp(jn + i));
        if (!pre) {
          ok = false;
          break;
        }
        for (int i = 0; i < nblk; ++i, ++jn) {
          // FWD: the scores LA blocks ahead are issued k-step by k-step between
          // this block's P V steps (two independent accumulators in the pipe);
          // BQ: issued whole, before this block's product
          static_assert(MODE != FWD || BCM == DH, "the interleave pairs the k-steps one to one");
          const bool s2 = MODE == FWD && i + LA < nblk;
          const uint32_t n2 = jn + LA;
          const int st2 = n2 % LY::NSTK, bf2 = n2 % NSB;
          if constexpr (MODE == FWD) {
            if (s2 && (!bwait(smem_u32(&y_full[st2]), (n2 / LY::NSTK) & 1u, abort_flag, P.status) ||
                       !bwait(smem_u32(&e_empty[bf2]), ((n2 / NSB) & 1u) ^ 1u, abort_flag,
                              P.status))) {
              ok = false;
              break;
            }
          } else if (i + LA < nblk && (!issue_sd(jn + LA) || (MODE == BQ && !issue_dp(jn + LA)))) {
            ok = false;
            break;
          }
          const int stk = jn % LY::NSTK, stv = jn % LY::NSTV, bf = jn % NSB;
          if (!bwait(smem_u32(&e_full[bf]), (jn / NSB) & 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          if constexpr (MODE == FWD) {
            // the block's V half
            if (!bwait(smem_u32(&y_full[LY::NSTK + stv]), (jn / LY::NSTV) & 1u, abort_flag,
                       P.status)) {
              ok = false;
              break;
            }
          }
          // the first accumulating product of a tile overwrites its TMEM sums: they
          // must have been read out
          if (i == 0 && !bwait(smem_u32(&a_empty[0]), (tn & 1u) ^ 1u, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc = (i > 0) ? 1u : 0u;
          if constexpr (MODE == FWD) {
            // O += P V_j: A = P in TMEM (bf16 pairs in S's buffer: the 16 keys of
            // k-step kk are warp half kk / 4's, in that half's first 32 columns),
            // B = V_j read MN-major [d_head x BCM keys] (its two d_head halves SUBC apart)
            const uint32_t y2 = smem_u32(sYK + st2 * HALF);
            const uint32_t x = smem_u32(sX);
#pragma unroll
            for (int kk = 0; kk < BCM / 16; ++kk) {
              mma_bf16_ta(tmem + OCOL, tmem + bf * BCM + 64 * (kk >> 2) + 8 * (kk & 3),
                          smem_desc_mn(smem_u32(sYV + stv * HALF) + kk * 2048, SUBC), ID_A,
                          (acc | kk) ? 1u : 0u);
              if (s2)  // k-step kk of S = Q K^T of block n2 (d_head half kk / 4)
                mma_bf16<1>(tmem + bf2 * BCM,
                            smem_desc(x + (kk >> 2) * SUB_R + (kk & 3) * 32, false),
                            smem_desc(y2 + (kk >> 2) * SUBC + (kk & 3) * 32, false), ID_S,
                            kk ? 1u : 0u);
            }
            if (s2) {
              mma_commit<1>(smem_u32(&s_full[bf2]));
              mma_commit<1>(smem_u32(&y_empty[st2]));  // K read
            }
          } else {
            // dQ += dS K_j: A = dS in TMEM (bf16 pairs in S's buffer: the 16 keys of
            // k-step kk are warp half kk / 4's, in that half's first 32 columns),
            // B = K_j read MN-major [d_head x BCM keys]
#pragma unroll
            for (int kk = 0; kk < BCM / 16; ++kk)
              mma_bf16_ta(tmem + 384, tmem + bf * BCM + 64 * (kk >> 2) + 8 * (kk & 3),
                          smem_desc_mn(smem_u32(sYK + stk * HALF) + kk * 2048, SUBC), ID_A,
                          (acc | kk) ? 1u : 0u);
          }
          // this S buffer is free again (its P / dS read), (FWD) O holds block i,
          // the stage (FWD: its V half; BQ: its K half) is no longer read
          mma_commit<1>(smem_u32(&e_empty[bf]));
          mma_commit<1>(smem_u32(&y_empty[(MODE == FWD) ? LY::NSTK + stv : stk]));
        }
        if (!ok) break;
        if constexpr (MODE != FWD) mma_commit<1>(smem_u32(&a_full[0]));
        mma_commit<1>(smem_u32(x_empty));
      }
      // every MMA issued must complete before TMEM is released
      mma_commit<1>(smem_u32(drain));
      bwait(smem_u32(drain), 0, abort_flag, P.status, ok ? kWaitLimitNs : 50ull * 1000 * 1000);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // Eight warps: warp w owns TMEM lanes 32 (w % 4) .. + 31 (tile rows) and
    // column half hf of every block and of every TMEM sum. The forward's two
    // warps of a row (w and w + 4) exchange their partial row maxima once per
    // block (mbarrier mxb) and their partial row sums once per tile (mbarrier lx).
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = 32 * q + lane;
    const uint32_t lb = static_cast<uint32_t>(32 * q) << 16;
    bool ok = true;
    uint32_t tn = 0, jn = 0;
    auto arrive = [&](uint64_t* bar) {
      if (lane == 0) mbar_arrive(smem_u32(bar));
    };
    // Every lane waits; the warp goes on only if all of them saw the phase, so
    // that no lane can reach a warp-collective tcgen05 instruction alone.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = bwait(smem_u32(bar), parity, abort_flag, P.status);
      return __all_sync(0xffffffffu, r);
    };
    const int64_t ld = static_cast<int64_t>(P.H) * DH;
    for (int u = blockIdx.x; ok && u < P.ntiles; u += gridDim.x, ++tn) {
      int t, bh, first, last;
      decode<MODE>(P, u, t, bh);
      blocks<MODE>(P, t, first, last);
      const int b = bh / P.H, col = (bh % P.H) * DH + 64 * hf;
      const int row = t * BR + r;                 // this thread's query (FWD, BQ) or key (BKV)
      const int64_t grow = static_cast<int64_t>(b) * P.L + row;  // its token row
      const bool row_ok = row < P.L;
      // visibility of the other side's index c: lo <= c <= hi
      int lo, hi;
      if constexpr (MODE == BKV) {
        lo = row_ok ? (P.causal ? row : 0) : P.L;
        hi = P.L - 1;
      } else {
        lo = 0;
        hi = (MODE == BQ && !row_ok) ? -1 : (P.causal ? min(row, P.L - 1) : P.L - 1);
      }
      if constexpr (MODE == FWD) {
        float* xl = reinterpret_cast<float*>(smem + LY::XCH_OFF);  // [2 tile parity][2 half][128]
        const int tp = static_cast<int>(tn & 1u);                    // tile parity: exchange slots
        const uint32_t ocol = OCOL + 64 * hf;                        // this warp's half of O
        float m = -INFINITY, l = 0.f;
        for (int j = first; j < last; ++j, ++jn) {
          const int bf = jn % NSB;                 // the block's S (then P) buffer
          const int bp = static_cast<int>(jn & 1u);  // block parity: max exchange slot
          if (!wwait(&s_full[bf], (jn / NSB) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Raw scores of the row: this warp's own 64 columns of the block. Scale > 0,
          // so the maximum is taken on raw scores; masked scores are -inf. The row's
          // other half comes from its other warp as a partial maximum through
          // shared memory, so that each warp reads only its own columns and can
          // write P over them.
          const int c0 = j * BCM + 64 * hf;
          const bool need_mask = (P.causal && j * BCM + BCM - 1 > t * BR) || j * BCM + BCM > P.L;
          float x[64];
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          {
            uint32_t xa[32], xb[32];
            tmem_ld32_nowait(tmem + lb + bf * BCM + 64 * hf, xa);
            tmem_ld32_nowait(tmem + lb + bf * BCM + 64 * hf + 32, xb);
            tmem_wait_ld2(xa, xb);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = __uint_as_float(xa[i]);
              x[32 + i] = __uint_as_float(xb[i]);
            }
          }
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < 64; ++i) x[i] = (c0 + i >= lo && c0 + i <= hi) ? x[i] : -INFINITY;
          }
#pragma unroll
          for (int i = 0; i < 64; i += 2) mx[(i >> 1) & 3] = max3(mx[(i >> 1) & 3], x[i], x[i + 1]);
          {
            // exchange the partial maxima with the row's other warp (block parity bp)
            float* xm = xl + 2 * 2 * BR + bp * 2 * BR;  // [2 half][128] of this block parity
            xm[hf * BR + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            mbar_arrive(smem_u32(&mxb[2 * q + bp]));
            if (!wwait(&mxb[2 * q + bp], (jn >> 1) & 1u)) {
              ok = false;
              break;
            }
            mx[0] = fmaxf(xm[hf * BR + r], xm[(1 - hf) * BR + r]);
          }
          const float bm = mx[0] * P.scale_log2;
          const float m_new = fmaxf(m, bm);
          // (a warp-wide decision: the TMEM accesses below are warp-collective;
          // the row's other warp sees the same rows and decides the same)
          const bool rescale = __any_sync(0xffffffffu, m_new > m + 8.f);
          if (j == first) {
            m = m_new;
          } else if (rescale) {
            // Lazy rescale: p = 2^(x - m) stays below 2^8 while the running maximum
            // m lags the true one by at most 8; past that, O (in TMEM, complete
            // through the previous block) and l move to the new maximum.
            const uint32_t pj = jn - 1;
            if (!wwait(&e_empty[pj % NSB], (pj / NSB) & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float a = ex2f_approx(m - m_new);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float o[32];
              tmem_ld32(tmem + lb + ocol + 32 * c, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= a;
              tmem_st32(tmem + lb + ocol + 32 * c, o);
            }
            l *= a;
            m = m_new;
          }
          // P as bf16 pairs over this warp's own score columns, already read: keys
          // 32 h .. 32 h + 31 of the half go to columns 16 h .. 16 h + 15, where the
          // P V product reads them as its A operand
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float p0 = ex2f_approx(fmaf(x[32 * h + i], P.scale_log2, -m));
              const float p1 = ex2f_approx(fmaf(x[32 * h + i + 1], P.scale_log2, -m));
              rs[(i >> 1) & 3] += p0 + p1;
              pk[i / 2] = pack2(p0, p1);
            }
            tmem_st16u_nowait(tmem + lb + bf * BCM + 64 * hf + 16 * h, pk);
          }
          l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          arrive(&e_full[bf]);
        }
        if (!ok) break;
        // O is complete once the tile's last product has committed
        const uint32_t pj = jn - 1;
        if (!wwait(&e_empty[pj % NSB], (pj / NSB) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float* ls = xl + tp * 2 * BR;
        ls[hf * BR + r] = l;
        mbar_arrive(smem_u32(&lx[2 * q + tp]));
        if (!wwait(&lx[2 * q + tp], (tn >> 1) & 1u)) {
          ok = false;
          break;
        }
        const float lt = l + ls[(1 - hf) * BR + r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float o[32];
          tmem_ld32(tmem + lb + ocol + 32 * c, o);
          if (row_ok) store32(P.out0 + grow * ld + col + 32 * c, o, inv);
        }
        if (hf == 0)
          P.lse[static_cast<int64_t>(bh) * P.Lp + row] =
              lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
        tc_fence_before();
        __syncwarp();
        arrive(&a_empty[0]);
      } else {
        // backward: per-row terms of the stationary rows (BQ) come from global memory
        float lr = 0.f, dr = 0.f;
        if constexpr (MODE == BQ) {
          lr = P.l2[static_cast<int64_t>(bh) * P.Lp + row];
          dr = P.dd[static_cast<int64_t>(bh) * P.Lp + row];
        }
        if constexpr (MODE == BQ) {
          for (int j = first; j < last; ++j, ++jn) {
            const int bf = jn & 1;
            // dP of the block into registers; its TMEM buffer goes back to the MMA
            if (!wwait(&a_full[1], jn & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            float dpv[64];
            {
              uint32_t da[32], db[32];
              tmem_ld32_nowait(tmem + lb + 256 + 64 * hf, da);
              tmem_ld32_nowait(tmem + lb + 256 + 64 * hf + 32, db);
              tmem_wait_ld2(da, db);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                dpv[i] = __uint_as_float(da[i]) - dr;
                dpv[32 + i] = __uint_as_float(db[i]) - dr;
              }
            }
            tc_fence_before();
            __syncwarp();
            arrive(&a_empty[1]);
            if (!wwait(&s_full[bf], (jn >> 1) & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool mask = (P.causal && j * BCM + BCM - 1 > t * BR) || j * BCM + BCM > P.L ||
                              t * BR + BR > P.L;
            // Per 32-key chunk h: S in, then dS as 16 columns of bf16 pairs written
            // over columns of this warp's half that are already read (the first
            // chunk's): keys 32 h .. 32 h + 31 of the half go to columns 16 h ...
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t sr[32];
              tmem_ld32_nowait(tmem + lb + bf * BCM + 64 * hf + 32 * h, sr);
              tmem_wait_ld2(sr, sr);
              if (mask) {
                const int c0 = j * BCM + 64 * hf + 32 * h;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (!(c0 + i >= lo && c0 + i <= hi)) sr[i] = __float_as_uint(-INFINITY);
              }
              uint32_t pd[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float p0 = ex2f_approx(fmaf(__uint_as_float(sr[i]), P.scale_log2, -lr));
                const float p1 = ex2f_approx(fmaf(__uint_as_float(sr[i + 1]), P.scale_log2, -lr));
                pd[i / 2] = pack2(p0 * dpv[32 * h + i], p1 * dpv[32 * h + i + 1]);
              }
              tmem_st16u_nowait(tmem + lb + bf * BCM + 64 * hf + 16 * h, pd);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            arrive(&e_full[bf]);
          }
        } else {
          // BKV: rows are keys, columns the block's 128 queries
          for (int j = first; j < last; ++j, ++jn) {
            const int st = jn % LY::NSTK;
            // the block's row terms (lse log2 e, D of its queries) came with its stage
            if (!wwait(&y_full[st], (jn / LY::NSTK) & 1u) || !wwait(&a_full[1], jn & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float* al = sAux + st * (LY::AUXB / 4) + 64 * hf;  // this half's 64 queries
            // dP^T into registers (minus D), then its TMEM buffer goes back to the MMA
            float dpv[64];
            {
              uint32_t da[32], db[32];
              tmem_ld32_nowait(tmem + lb + 128 + 64 * hf, da);
              tmem_ld32_nowait(tmem + lb + 128 + 64 * hf + 32, db);
              tmem_wait_ld2(da, db);
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 d0 = *reinterpret_cast<const float4*>(al + BCM + i);
                const float4 d1 = *reinterpret_cast<const float4*>(al + BCM + 32 + i);
                dpv[i] = __uint_as_float(da[i]) - d0.x;
                dpv[i + 1] = __uint_as_float(da[i + 1]) - d0.y;
                dpv[i + 2] = __uint_as_float(da[i + 2]) - d0.z;
                dpv[i + 3] = __uint_as_float(da[i + 3]) - d0.w;
                dpv[32 + i] = __uint_as_float(db[i]) - d1.x;
                dpv[32 + i + 1] = __uint_as_float(db[i + 1]) - d1.y;
                dpv[32 + i + 2] = __uint_as_float(db[i + 2]) - d1.z;
                dpv[32 + i + 3] = __uint_as_float(db[i + 3]) - d1.w;
              }
            }
            tc_fence_before();
            __syncwarp();
            arrive(&a_empty[1]);
            if (!wwait(&s_full[0], jn & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool mask = (P.causal && j * BCM < t * BR + BR - 1) || j * BCM + BCM > P.L ||
                              t * BR + BR > P.L;
            // Per 32-query chunk h: S^T in, then P^T (16 columns of bf16 pairs) and
            // dS^T (the next 16) written over the chunk's own columns, already read.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t sr[32];
              tmem_ld32_nowait(tmem + lb + 64 * hf + 32 * h, sr);
              tmem_wait_ld2(sr, sr);
              if (mask) {
                const int c0 = j * BCM + 64 * hf + 32 * h;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (!(c0 + i >= lo && c0 + i <= hi)) sr[i] = __float_as_uint(-INFINITY);
              }
              uint32_t o[32];
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 lv = *reinterpret_cast<const float4*>(al + 32 * h + i);
                const float l4[4] = {lv.x, lv.y, lv.z, lv.w};
                float pv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  pv[k] = ex2f_approx(fmaf(__uint_as_float(sr[i + k]), P.scale_log2, -l4[k]));
                o[i / 2] = pack2(pv[0], pv[1]);
                o[i / 2 + 1] = pack2(pv[2], pv[3]);
                o[16 + i / 2] = pack2(pv[0] * dpv[32 * h + i], pv[1] * dpv[32 * h + i + 1]);
                o[16 + i / 2 + 1] = pack2(pv[2] * dpv[32 * h + i + 2], pv[3] * dpv[32 * h + i + 3]);
              }
              tmem_st32u_nowait(tmem + lb + 64 * hf + 32 * h, o);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            arrive(&e_full[0]);
          }
        }
        if (!ok) break;
        if (!wwait(&a_full[0], tn & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (MODE == BKV) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v[32];
            tmem_ld32(tmem + lb + 256 + 64 * hf + 32 * c, v);
            if (row_ok) store32(P.out0 + grow * ld + col + 32 * c, v, 1.f);
          }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float v[32];
          tmem_ld32(tmem + lb + 384 + 64 * hf + 32 * c, v);
          if (row_ok) store32(P.out1 + grow * ld + col + 32 * c, v, P.scale);
        }
        tc_fence_before();
        __syncwarp();
        arrive(&a_empty[0]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, 512);
  }
}

// D[bh, i] = sum_e dO[i, h, e] O[i, h, e] (0 for L <= i < Lp) and
// l2[bh, i] = lse[bh, i] log2(e).
// Work items are (token row (b, i < L), group of up to 16 heads); a warp takes
// an item's O and dO (up to 16 x 128 bf16 each) through shared memory: each
// warp owns a ring of two stages, a stage holds one item of O and of dO,
// brought in by two bulk copies that complete on the stage's mbarrier, and the
// copies of the warp's next item are in flight while it works on this one.
// Each head's D is a half-warp reduction (head 2u + (lane >= 16) of the group
// at step u, 16-byte shared-memory reads). Block k takes the contiguous items
// [k n / grid, (k + 1) n / grid), its warps take them round robin. l2, and
// D = 0 on the padding rows i in [L, Lp) of the lse stride, are one coalesced
// grid-stride pass.
// Every wait is bounded; a warp that gives up waits (bounded) for its copies in
// flight before the block leaves.
constexpr size_t kRowsSmem = 227 * 1024;
constexpr int kRowsMaxWarps = 12;
__global__ void __launch_bounds__(kRowsMaxWarps * 32, 1)
    attn_rows_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                     const float* __restrict__ lse, float* __restrict__ dd,
                     float* __restrict__ l2, int B, int L, int H, int Lp, int* status) {
  extern __shared__ __align__(128) unsigned char ars[];
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HG = H < 16 ? H : 16;                        // heads of a full group
  const int ngroups = (H + 15) / 16;
  const uint32_t row_bytes = static_cast<uint32_t>(HG) * DH * 2u;  // one item of one tensor
  const uint32_t stage_bytes = 2u * row_bytes;  // O | dO
  unsigned char* ring = ars + static_cast<size_t>(warp) * 2 * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ars + static_cast<size_t>(nw) * 2 * stage_bytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * nw);
  const uint32_t bar0 = smem_u32(bars + 2 * warp);
  const uint32_t ring0 = smem_u32(ring);
  if (lane == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  grid_dependency_sync();

  // l2 = lse log2(e) for every entry, and D = 0 on the padding rows of the lse
  // stride: one coalesced grid-stride pass
  const int64_t nrow_terms = static_cast<int64_t>(B) * H * Lp;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < nrow_terms;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    l2[t] = lse[t] * kLog2e;
    if (static_cast<int>(t % Lp) >= L) dd[t] = 0.f;
  }
  const int64_t items = static_cast<int64_t>(B) * L * ngroups;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * items / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * items / gridDim.x;
  const int64_t first = r0 + warp;
  const int64_t n = first < r1 ? (r1 - first + nw - 1) / nw : 0;  // this warp's items
  const int64_t rowlen = static_cast<int64_t>(H) * DH;
  // item t: token row t / ngroups (b L + i), heads from 16 (t % ngroups)
  // (one group when H <= 16: no division)
  auto group_of = [&](int64_t t) { return ngroups == 1 ? 0 : static_cast<int>(t % ngroups); };
  auto row_of = [&](int64_t t) { return ngroups == 1 ? t : t / ngroups; };
  auto heads_of = [&](int g) { return H - 16 * g < 16 ? H - 16 * g : 16; };
  auto issue = [&](int64_t j) {  // copies of the warp's item j into stage j & 1 (lane 0)
    const int64_t t = first + j * nw;
    const int g = group_of(t);
    const int64_t off = row_of(t) * rowlen + static_cast<int64_t>(g) * 16 * DH;
    const uint32_t bytes = static_cast<uint32_t>(heads_of(g)) * DH * 2u;
    const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(j & 1);
    const uint32_t dst = ring0 + static_cast<uint32_t>(j & 1) * stage_bytes;
    mbar_expect_tx(bar, 2u * bytes);
    bulk_load(dst, o + off, bytes, bar);
    bulk_load(dst + row_bytes, dout + off, bytes, bar);
  };
  if (lane == 0) {
    if (n > 0) issue(0);
    if (n > 1) issue(1);
  }
  const int lo = (lane >> 4) * DH + (lane & 15) * 8;  // this lane's columns of head pair u
  int64_t j = 0;
  for (; j < n; ++j) {
    const int64_t t = first + j * nw;
    const int64_t row = row_of(t);
    const int g = group_of(t);
    const int g0 = 16 * g;  // the group's first head
    const int nh = heads_of(g);
    const int b = static_cast<int>(row / L), i = static_cast<int>(row % L);
    const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(j & 1);
    const bool landed =
        bwait(bar, static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status);
    if (!__all_sync(0xffffffffu, landed)) break;
    const __nv_bfloat16* so = reinterpret_cast<const __nv_bfloat16*>(ring + (j & 1) * stage_bytes);
    const __nv_bfloat16* sg = so + HG * DH;
    for (int u = 0; 2 * u < nh; ++u) {
      const int h = 2 * u + (lane >> 4);  // head within the group
      float acc = 0.f;
      if (h < nh) {
        const uint4 a = *reinterpret_cast<const uint4*>(so + 2 * u * DH + lo);
        const uint4 g = *reinterpret_cast<const uint4*>(sg + 2 * u * DH + lo);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 fa = __bfloat1622float2(a2[k]), fg = __bfloat1622float2(g2[k]);
          acc = fmaf(fa.x, fg.x, acc);
          acc = fmaf(fa.y, fg.y, acc);
        }
      }
#pragma unroll
      for (int sft = 8; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
      if ((lane & 15) == 0 && h < nh) dd[(static_cast<int64_t>(b) * H + g0 + h) * Lp + i] = acc;
    }
    __syncwarp();  // every lane has read the stage
    if (lane == 0 && j + 2 < n) {
      fence_proxy_async();
      issue(j + 2);
    }
  }
  if (j < n) {
    // a wait gave up: this warp's copies still in flight (rows j and j + 1) land
    // before the block's shared memory is released
    for (int64_t k = j; k < n && k < j + 2; ++k) {
      const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(k & 1);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, static_cast<uint32_t>(k >> 1) & 1u) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// 3-D map over [B, L, H d_head] bf16: boxes of 64 columns x `rows` token rows
// of one sequence (rows past L read as zero), 128-byte swizzle.
bool encode3(CUtensorMap* m, const void* ptr, const bn_attn_desc& d, uint32_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t D = static_cast<cuuint64_t>(d.H * d.d_head);
  cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(d.L), static_cast<cuuint64_t>(d.B)};
  cuuint64_t strides[2] = {D * 2, D * 2 * static_cast<cuuint64_t>(d.L)};
  cuuint32_t box[3] = {64, rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sms() {
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

template <int MODE>
cudaError_t launch(Ctx& c, const Params& P, double flops, double bytes) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay<MODE>::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int grid = P.ntiles < c.num_sms ? P.ntiles : c.num_sms;
  prof_start(c);
  cudaError_t e = launch_pdl(attn_kernel<MODE>, dim3(grid), dim3(NTHREADS), Lay<MODE>::SMEM,
                             c.stream, P);
  note_launch(c, KK_ATTN, MODE, flops, bytes);
  return e;
}

thread_local char g_err[256] = "no error";

bn_status check(const bn_attn_desc* d) {
  if (d == nullptr || d->B < 1 || d->L < 1 || d->H < 1 || d->d_head < 1 ||
      (d->causal != 0 && d->causal != 1))
    return BN_ERR_INVALID_ARG;
  if (d->d_head != DH) return BN_ERR_UNSUPPORTED;
  // 32-bit tile indices and TMA coordinates
  const int64_t Lp = bn_attn_lse_stride(d->L);
  if (d->B * d->H * Lp >= (int64_t(1) << 31) || d->L >= (int64_t(1) << 31) ||
      d->H * DH >= (int64_t(1) << 24))
    return BN_ERR_UNSUPPORTED;
  return BN_OK;
}
bool aligned(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// algorithmic FLOPs of the matrix products: 4 B H d_head x (visible (i, j) pairs)
// forward (S and P V), twice that plus the recomputed S in the backward
double visible_pairs(const bn_attn_desc& d) {
  const double L = static_cast<double>(d.L);
  return static_cast<double>(d.B * d.H) * (d.causal ? L * (L + 1) / 2 : L * L);
}


// The launch parameters every mode shares: shapes, tile count, scales, status word.
Params shape_params(const bn_attn_desc& d, int* status) {
  Params P = {};
  P.B = static_cast<int>(d.B);
  P.L = static_cast<int>(d.L);
  P.H = static_cast<int>(d.H);
  P.Lp = static_cast<int>(bn_attn_lse_stride(d.L));
  P.causal = d.causal;
  P.ntiles = static_cast<int>(d.B * d.H * (P.Lp / BR));
  P.scale = 1.f / sqrtf(static_cast<float>(DH));
  P.scale_log2 = P.scale * kLog2e;
  P.status = status;
  return P;
}

// The forward's launch; `unfed` (a test hook) withholds the first query tile.
cudaError_t forward_launch(Ctx& c, const bn_attn_desc& d, const void* q, const void* k,
                           const void* v, void* o, float* lse, int* status, bool unfed) {
  Params P = shape_params(d, status);
  if (!encode3(&P.mx[0], q, d, BR) || !encode3(&P.my[0], k, d, BCF) ||
      !encode3(&P.my[1], v, d, BCF))
    return cudaErrorInvalidValue;
  P.out0 = static_cast<__nv_bfloat16*>(o);
  P.lse = lse;
  P.unfed = unfed ? 1 : 0;
  const double elems = static_cast<double>(d.B * d.L * d.H * DH);
  return launch<FWD>(c, P, unfed ? 0.0 : 4.0 * DH * visible_pairs(d),
                     unfed ? 0.0 : 4.0 * elems * 2 + static_cast<double>(d.B * d.H * P.Lp) * 4);
}

}  // namespace attn

bn_status attn_check(const bn_attn_desc& d) { return attn::check(&d); }
size_t attn_scratch_floats(const bn_attn_desc& d) {
  return static_cast<size_t>(2 * d.B * d.H * bn_attn_lse_stride(d.L));
}

cudaError_t attn_forward(Ctx& c, const bn_attn_desc& d, const void* q, const void* k,
                         const void* v, void* o, float* lse, int* status) {
  return attn::forward_launch(c, d, q, k, v, o, lse, status, false);
}

cudaError_t attn_backward(Ctx& c, const bn_attn_desc& d, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, float* rows_scratch, int* status) {
  using namespace attn;
  const int Lp = static_cast<int>(bn_attn_lse_stride(d.L));
  const int64_t rows = d.B * d.H * Lp;
  float* dd = rows_scratch;
  float* l2 = dd + rows;
  Params P = shape_params(d, status);
  P.l2 = l2;
  P.dd = dd;
  const double elems = static_cast<double>(d.B * d.L * d.H * DH);
  const double pairs = visible_pairs(d);
  // one block per SM, as many warps as two stages of an item (a row's O and dO
  // for up to 16 heads) fit (at most twelve), each warp streaming its items
  const size_t warp_bytes = 4 * static_cast<size_t>(std::min<int64_t>(d.H, 16)) * DH * 2 + 16;
  const int nw = static_cast<int>(std::max<size_t>(
      1, std::min<size_t>(kRowsMaxWarps, (kRowsSmem - 16) / warp_bytes)));
  const size_t rows_smem = warp_bytes * nw + 16;
  static const bool rows_attr = [] {
    cudaFuncSetAttribute(attn_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kRowsSmem));
    return true;
  }();
  (void)rows_attr;
  const int64_t items = static_cast<int64_t>(d.B) * d.L * ((d.H + 15) / 16);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((items + nw - 1) / nw, c.num_sms));
  prof_start(c);
  cudaError_t e = launch_pdl(attn_rows_kernel, dim3(static_cast<unsigned>(blocks)),
                             dim3(nw * 32), rows_smem, c.stream,
                             static_cast<const __nv_bfloat16*>(o),
                             static_cast<const __nv_bfloat16*>(dout), lse, dd, l2, P.B, P.L, P.H,
                             Lp, status);
  note_launch(c, KK_ATTN, 3, 2.0 * elems, 2.0 * elems * 2 + 3.0 * rows * 4);
  if (e != cudaSuccess) return e;
  Params K = P;
  if (!encode3(&K.mx[0], k, d, BR) || !encode3(&K.mx[1], v, d, BR) ||
      !encode3(&K.my[0], q, d, BCF) || !encode3(&K.my[1], dout, d, BCF))
    return cudaErrorInvalidValue;
  K.out0 = static_cast<__nv_bfloat16*>(dv);
  K.out1 = static_cast<__nv_bfloat16*>(dk);
  e = launch<BKV>(c, K, 8.0 * DH * pairs, 6.0 * elems * 2 + 2.0 * rows * 4);
  if (e != cudaSuccess) return e;
  Params Q = P;
  if (!encode3(&Q.mx[0], q, d, BR) || !encode3(&Q.mx[1], dout, d, BR) ||
      !encode3(&Q.my[0], k, d, BCF) || !encode3(&Q.my[1], v, d, BCF))
    return cudaErrorInvalidValue;
  Q.out1 = static_cast<__nv_bfloat16*>(dq);
  return launch<BQ>(c, Q, 6.0 * DH * pairs, 5.0 * elems * 2 + 2.0 * rows * 4);
}

}  // namespace bn

using namespace bn;
using namespace bn::attn;

extern "C" int64_t bn_attn_lse_stride(int64_t L) { return L <= 0 ? 0 : (L + 127) / 128 * 128; }

extern "C" bn_status bn_attn_workspace_size(const bn_attn_desc* d, size_t* lse_bytes,
                                            size_t* scratch_bytes) {
  bn_status s = check(d);
  if (s != BN_OK) return s;
  const size_t rows = static_cast<size_t>(d->B * d->H * bn_attn_lse_stride(d->L));
  if (lse_bytes) *lse_bytes = rows * 4;
  if (scratch_bytes) *scratch_bytes = 256 + 2 * rows * 4;
  return BN_OK;
}

extern "C" bn_status bn_attn_forward(const bn_attn_desc* d, const void* q, const void* k,
                                     const void* v, void* o, float* lse, void* scratch,
                                     bn_stream_t stream) {
  bn_status s = check(d);
  if (s != BN_OK) return s;
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse),
                        static_cast<const void*>(scratch)})
    if (!aligned(p)) return p == nullptr ? BN_ERR_INVALID_ARG : BN_ERR_ALIGNMENT;
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.num_sms = sms();
  const cudaError_t e = attn_forward(c, *d, q, k, v, o, lse, static_cast<int*>(scratch));
  if (e != cudaSuccess) {
    std::snprintf(g_err, sizeof(g_err), "%s", cudaGetErrorString(e));
    return BN_ERR_CUDA;
  }
  return BN_OK;
}

extern "C" bn_status bn_attn_backward(const bn_attn_desc* d, const void* q, const void* k,
                                      const void* v, const void* o, const float* lse,
                                      const void* dout, void* dq, void* dk, void* dv,
                                      void* scratch, bn_stream_t stream) {
  bn_status s = check(d);
  if (s != BN_OK) return s;
  for (const void* p : {q, k, v, o, static_cast<const void*>(lse), dout,
                        static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv), static_cast<const void*>(scratch)})
    if (!aligned(p)) return p == nullptr ? BN_ERR_INVALID_ARG : BN_ERR_ALIGNMENT;
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.num_sms = sms();
  float* rows = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + 256);
  const cudaError_t e = attn_backward(c, *d, q, k, v, o, lse, dout, dq, dk, dv, rows,
                                      static_cast<int*>(scratch));
  if (e != cudaSuccess) {
    std::snprintf(g_err, sizeof(g_err), "%s", cudaGetErrorString(e));
    return BN_ERR_CUDA;
  }
  return BN_OK;
}

// Test hook (include/boostblk_testing.h): the forward with its first stationary
// tile never loaded, so that the MMA thread's bounded wait for it runs out.
extern "C" bn_status bn_testing_attn_forward_unfed(const bn_attn_desc* d, const void* q,
                                                   const void* k, const void* v, void* o,
                                                   float* lse, void* scratch, bn_stream_t stream) {
  bn_status s = check(d);
  if (s != BN_OK) return s;
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse),
                        static_cast<const void*>(scratch)})
    if (!aligned(p)) return p == nullptr ? BN_ERR_INVALID_ARG : BN_ERR_ALIGNMENT;
  Ctx c;
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.num_sms = sms();
  return forward_launch(c, *d, q, k, v, o, lse, static_cast<int*>(scratch), true) == cudaSuccess
             ? BN_OK
             : BN_ERR_CUDA;
}
