// Row-wise kernels of the block: shard statistics of Online RMSNorm, the
// RMSNorm backward, the split-K reduction and small elementwise passes.
// All are HBM-bound: 16-byte vector loads, one warp per row, warp-shuffle
// reductions, and fixed reduction orders (results are bit-reproducible).
#include <algorithm>

#include "common.cuh"
#include "rowops.h"
#include "tc_ptx.cuh"

namespace bn {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// F0: per-row, per-shard sums of squares (one warp per row)
// ---------------------------------------------------------------------------
// 8 elements of T kept packed in registers (16 bytes of bf16, 32 of fp32),
// unpacked element by element where they are used.
template <typename T> struct Pack8;
template <> struct Pack8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    v = *reinterpret_cast<const uint4*>(p);
  }
  __device__ __forceinline__ void zero() { v = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ float operator[](int i) const {
    const uint32_t w = (i < 2) ? v.x : (i < 4) ? v.y : (i < 6) ? v.z : v.w;
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};
template <> struct Pack8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float operator[](int i) const {
    const float4& q = (i < 4) ? a : b;
    const int j = i & 3;
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
  }
};

// Statistics of one row from chunks already in registers: chunk u of a batch
// covers columns base + 256 u + 8 lane .. +7 (zero past d). Shards are whole
// multiples of 8 columns, so a chunk lies in one shard; each shard's sum is
// reduced across the warp once per batch it intersects and added in shard
// order. cur / cur_s / tot carry a shard that continues into the next batch.
template <typename T, int U>
__device__ __forceinline__ void stats_batch(const Pack8<T> (&v)[U], int base, int d, int w,
                                            float* __restrict__ ss_row, int lane, float& cur,
                                            int& cur_s, float& tot) {
  float q[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaf(v[u][i], v[u][i], a);
    q[u] = a;
  }
  const int last = min(d, base + 256 * U) - 1;
  for (int s = base / w; s <= last / w; ++s) {
    const int lo = s * w, hi = lo + w;  // the shard's columns
    float a = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = base + 256 * u + 8 * lane;
      if (c >= lo && c < hi) a += q[u];  // chunks past d are zero and past hi
    }
    a = warp_sum(a);
    if (s != cur_s) {
      if (lane == 0) ss_row[cur_s] = cur;
      cur_s = s;
      cur = 0.f;
    }
    cur += a;
    tot += a;
  }
}

template <typename T, int U>
__device__ __forceinline__ void load_batch(Pack8<T> (&v)[U], const T* __restrict__ xr, int base,
                                           int d, int lane) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = base + 256 * u + 8 * lane;
    if (c < d)
      v[u].load(xr + c);
    else
      v[u].zero();
  }
}

// Rows [warp0, rows) with stride `stride`, one warp each. Rows of at most 2048
// columns are one batch: the next row's loads are issued before this row is
// reduced, so two rows per warp are in flight. Longer rows go batch by batch.
template <typename T>
__device__ __forceinline__ void stats_rows(const T* __restrict__ x, int64_t rows, int d, int S,
                                           float eps, float* __restrict__ ss,
                                           float* __restrict__ rstd, int64_t row0,
                                           int64_t stride, int lane) {
  constexpr int U = 8;
  const int w = d / S;
  if (d <= 256 * U) {
    Pack8<T> v[U], nx[U];
    if (row0 < rows) load_batch<T, U>(v, x + row0 * d, 0, d, lane);
    for (int64_t row = row0; row < rows; row += stride) {
      const int64_t next = row + stride;
      if (next < rows) load_batch<T, U>(nx, x + next * d, 0, d, lane);
      float cur = 0.f, tot = 0.f;
      int cur_s = 0;
      stats_batch<T, U>(v, 0, d, w, ss + row * S, lane, cur, cur_s, tot);
      if (lane == 0) {
        ss[row * S + cur_s] = cur;
        rstd[row] = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = nx[u];
    }
    return;
  }
  for (int64_t row = row0; row < rows; row += stride) {
    const T* xr = x + row * d;
    float cur = 0.f, tot = 0.f;
    int cur_s = 0;
    for (int base = 0; base < d; base += 256 * U) {
      Pack8<T> v[U];
      load_batch<T, U>(v, xr, base, d, lane);
      stats_batch<T, U>(v, base, d, w, ss + row * S, lane, cur, cur_s, tot);
    }
    if (lane == 0) {
      ss[row * S + cur_s] = cur;
      rstd[row] = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
    }
  }
}

// Norm-weight folds (out = A diag(w)) in chunks of up to 1024 columns of one
// row of A, one warp per chunk: fold_chunks counts a job's chunks, fold_chunk
// does chunk k (row k / p, columns from 1024 (k % p), p = chunks per row).
constexpr int kFoldCols = 1024;
template <typename T>
__device__ __forceinline__ int64_t fold_chunks(const FoldJob<T>& f) {
  return f.A == nullptr ? 0 : f.rows * ((f.cols + kFoldCols - 1) / kFoldCols);
}
template <typename T>
__device__ __forceinline__ void fold_chunk(const FoldJob<T>& f, int64_t k, int lane) {
  const int64_t per_row = (f.cols + kFoldCols - 1) / kFoldCols;
  const int64_t r = k / per_row;
  const int64_t c0 = (k - r * per_row) * kFoldCols;
  const int64_t c1 = c0 + kFoldCols < f.cols ? c0 + kFoldCols : f.cols;
  constexpr int U = kFoldCols / 256;
  Pack8<T> a[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {  // every load of the chunk before any store
    const int64_t c = c0 + 256 * u + 8 * lane;
    if (c < c1) a[u].load(f.A + r * f.cols + c);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t c = c0 + 256 * u + 8 * lane;
    if (c < c1) {
      float ww[8], o[8];
      Vec8<T>::load(f.w + c, ww);
#pragma unroll
      for (int k2 = 0; k2 < 8; ++k2) o[k2] = a[u][k2] * ww[k2];
      Vec8<T>::store(f.out + r * f.cols + c, o);
    }
  }
}

// The row statistics, then the norm-weight folds, over one index space of work
// items dealt round robin to the W = 8 gridDim.x warps: items [0, rows) are the
// rows of x, then come the fold chunks of job 0 and of job 1. A chunk moves
// 2 x 1024 elements, a row of x reads d; dealing them together keeps every
// warp's share within one item of the others.
template <typename T>
__global__ void __launch_bounds__(256, sizeof(T) == 2 ? 3 : 1)
    stats_kernel(const T* __restrict__ x, int64_t rows, int d, int S, float eps,
                 float* __restrict__ ss, float* __restrict__ rstd, const FoldJob<T> f0,
                 const FoldJob<T> f1) {
  grid_dependency_sync();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  const int64_t W = static_cast<int64_t>(gridDim.x) * 8;
  stats_rows(x, rows, d, S, eps, ss, rstd, gw, W, lane);
  const int64_t n0 = fold_chunks(f0), n1 = fold_chunks(f1);
  // this warp's first chunk: the item index rows + k is dealt to warp (rows + k) mod W
  for (int64_t k = ((gw - rows) % W + W) % W; k < n0 + n1; k += W) {
    if (k < n0)
      fold_chunk(f0, k, lane);
    else
      fold_chunk(f1, k - n0, lane);
  }
}

template <typename T>
void launch_stats_fold(Ctx& c, const T* x, int64_t rows, int64_t d, int S, float eps, float* ss,
                       float* rstd, const FoldJob<T>& f0, const FoldJob<T>& f1) {
  // three blocks of 8 warps per SM (80 registers a thread for bf16), each warp
  // looping over its rows and then its fold chunks
  const auto chunks = [](const FoldJob<T>& f) -> int64_t {
    return f.A == nullptr ? 0 : f.rows * ((f.cols + kFoldCols - 1) / kFoldCols);
  };
  const int64_t items = rows + chunks(f0) + chunks(f1);
  const unsigned blocks =
      static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((items + 7) / 8, c.num_sms * 3)));
  const double fold_elems = static_cast<double>(f0.A ? f0.rows * f0.cols : 0) +
                            static_cast<double>(f1.A ? f1.rows * f1.cols : 0);
  prof_start(c);
  track(c, launch_pdl(stats_kernel<T>, blocks, 256, 0, c.stream, x, rows, static_cast<int>(d), S,
                      eps, ss, rstd, f0, f1));
  note_launch(c, KK_STATS, -1, 2.0 * rows * d + fold_elems,
              static_cast<double>(rows) * (d * sizeof(T) + 4 * S + 4) +
                  2.0 * fold_elems * sizeof(T));
}

template <typename T>
void launch_stats(Ctx& c, const T* x, int64_t rows, int64_t d, int S, float eps, float* ss,
                  float* rstd) {
  launch_stats_fold<T>(c, x, rows, d, S, eps, ss, rstd, FoldJob<T>{}, FoldJob<T>{});
}

// ---------------------------------------------------------------------------
// B3: RMSNorm backward. Every block writes the dw column sums of its rows to a
// row of `part`; colsum_kernel (or the backward's final launch) adds the rows
// in a fixed order, so dw is bit-reproducible.
// ---------------------------------------------------------------------------
constexpr int kNormBwdUnroll = 4;
constexpr size_t kNormBwdSmemLimit = 200 * 1024;

// Any T and d: one warp per row, two passes over the row (the second one mostly
// from L1/L2), 4 x 16 bytes of every tensor in flight per lane, two blocks of
// 8 warps per SM. Each warp keeps its own dw column sums in shared memory
// (lane-exclusive columns, no atomics).
template <typename T>
__global__ void __launch_bounds__(256, 2)
    norm_bwd_kernel(const T* __restrict__ dn, const T* __restrict__ x, const T* __restrict__ w,
                    const float* __restrict__ rstd, const T* __restrict__ dres, int64_t rows,
                    int d, T* __restrict__ dx, float* __restrict__ part) {
  grid_dependency_sync();
  // [warps][d + d/8] column sums; column c lives at c + c/8, so the 8 columns a
  // lane owns are 9 floats apart from the next lane's: no bank conflicts
  extern __shared__ float acc[];
  const int nw = blockDim.x >> 5;
  const int dp = d + d / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < nw * dp; i += blockDim.x) acc[i] = 0.f;
  __syncthreads();
  float* my = acc + warp * dp;
  const float inv_d = 1.0f / static_cast<float>(d);
  constexpr int U = sizeof(T) == 2 ? kNormBwdUnroll : kNormBwdUnroll / 2;  // same bytes in flight
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * nw + warp; row < rows;
       row += static_cast<int64_t>(gridDim.x) * nw) {
    const T* dnr = dn + row * d;
    const T* xr = x + row * d;
    float s = 0.f;
    for (int base = lane * 8; base < d; base += 256 * U) {
      Pack8<T> a[U], b[U], ww[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * 256;
        if (c < d) {
          a[u].load(dnr + c);
          b[u].load(xr + c);
          ww[u].load(w + c);
        } else {
          a[u].zero();
          b[u].zero();
          ww[u].zero();
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) s = fmaf(a[u][i] * ww[u][i], b[u][i], s);
    }
    s = warp_sum(s);
    const float r = rstd[row];
    const float coef = r * r * s * inv_d;
    const T* dr = dres + row * d;
    T* o = dx + row * d;
    for (int base = lane * 8; base < d; base += 256 * U) {
      Pack8<T> a[U], b[U], ww[U], g[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * 256;
        if (c < d) {
          a[u].load(dnr + c);
          b[u].load(xr + c);
          ww[u].load(w + c);
          g[u].load(dr + c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * 256;
        if (c < d) {
          float out[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            out[i] = g[u][i] + (a[u][i] * ww[u][i] - b[u][i] * coef);
            my[c + c / 8 + i] = fmaf(a[u][i], b[u][i], my[c + c / 8 + i]);
          }
          Vec8<T>::store(o + c, out);
        }
      }
    }
  }
  __syncthreads();
  for (int col = threadIdx.x; col < d; col += blockDim.x) {
    float v = acc[col + col / 8];
    for (int k = 1; k < nw; ++k) v += acc[k * dp + col + col / 8];
    part[static_cast<int64_t>(blockIdx.x) * d + col] = v;
  }
}

// bf16 rows of at most 256 NP columns (NP <= 16), streamed through shared memory. Every
// warp owns a ring of two stages; a stage holds one row of dn', x and dres,
// brought in by three bulk copies that complete on the stage's mbarrier. While
// a warp works on one row, the copies of its next row are in flight, so an SM
// keeps up to 2 x warps rows of reads outstanding without holding them in
// registers. A lane owns the columns 256 u + 8 lane + (0..7), u < NP: their
// norm weight and their dw sums stay in registers for the whole launch. Block
// b takes the contiguous rows [b rows / grid, (b + 1) rows / grid); its warps
// take them round robin. One block per SM. Arithmetic per element, and the
// order of the row sum, as in norm_bwd_kernel. Past 8 chunks a lane the weights
// sit once in shared memory, after the barriers, instead of in registers.
constexpr size_t kNormBwdStreamSmem = 227 * 1024;

// Untiled bulk copy from global memory into this CTA's shared memory,
// completing on `bar`. Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Warps per block: registers bound them up to 8 chunks a lane (8 NP float sums
// and 4 NP registers of weights a lane), shared memory beyond (two stages of 3
// rows, 6 x 2 x 256 NP bytes a warp, and the weights).
template <int NP>
constexpr int norm_bwd_stream_warps() {
  return NP > 12 ? 4 : NP > 8 ? 6 : NP > 4 ? 9 : 16;
}

template <int NP>
__global__ void __launch_bounds__(norm_bwd_stream_warps<NP>() * 32, 1)
    norm_bwd_stream_kernel(const bf16* __restrict__ dn, const bf16* __restrict__ x,
                           const bf16* __restrict__ w, const float* __restrict__ rstd,
                           const bf16* __restrict__ dres, int64_t rows, int d,
                           bf16* __restrict__ dx, float* __restrict__ part, int* status,
                           int unfed) {
  extern __shared__ __align__(128) unsigned char nbs[];
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t row_bytes = static_cast<uint32_t>(d) * 2u;
  const uint32_t stage_bytes = 3u * row_bytes;  // dn' | x | dres
  unsigned char* ring = nbs + static_cast<size_t>(warp) * 2 * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(nbs + static_cast<size_t>(nw) * 2 * stage_bytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * nw);
  const uint32_t bar0 = tc::smem_u32(bars + 2 * warp);
  const uint32_t ring0 = tc::smem_u32(ring);
  if (lane == 0) {
    tc::mbar_init(bar0, 1);
    tc::mbar_init(bar0 + 8, 1);
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  // the norm weight is a parameter: no kernel of the stream writes it
  constexpr bool kSharedW = NP > 8;
  bf16* sw = reinterpret_cast<bf16*>(bars + 2 * nw + 2);
  Pack8<bf16> wv[kSharedW ? 1 : NP];
  float acc[NP][8];
  if constexpr (kSharedW) {
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x)
      *reinterpret_cast<uint4*>(sw + 8 * i) = *reinterpret_cast<const uint4*>(w + 8 * i);
  }
#pragma unroll
  for (int u = 0; u < NP; ++u) {
    if constexpr (!kSharedW) {
      const int c = u * 256 + lane * 8;
      if (c < d)
        wv[u].load(w + c);
      else
        wv[u].zero();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
  }
  // the weights of chunk u (zero past d)
  auto weights = [&](int u) {
    if constexpr (kSharedW) {
      Pack8<bf16> t;
      const int c = u * 256 + lane * 8;
      if (c < d)
        t.load(sw + c);
      else
        t.zero();
      return t;
    } else {
      return wv[u];
    }
  };
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  grid_dependency_sync();

  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * rows / gridDim.x;
  const int64_t first = r0 + warp;
  const int64_t n = first < r1 ? (r1 - first + nw - 1) / nw : 0;  // this warp's rows
  // copies of the warp's row j into stage j & 1 (lane 0)
  auto issue = [&](int64_t j) {
    const int64_t off = (first + j * nw) * d;
    const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(j & 1);
    const uint32_t dst = ring0 + static_cast<uint32_t>(j & 1) * stage_bytes;
    tc::mbar_expect_tx(bar, stage_bytes);
    bulk_load(dst, dn + off, row_bytes, bar);
    bulk_load(dst + row_bytes, x + off, row_bytes, bar);
    bulk_load(dst + 2 * row_bytes, dres + off, row_bytes, bar);
  };
  if (lane == 0) {
    // (test hook) the first warp's first row is never loaded: its wait must run out
    if (n > 0 && !(unfed && blockIdx.x == 0 && warp == 0)) issue(0);
    if (n > 1) issue(1);
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  float r_next = n > 0 ? rstd[first] : 0.f;
  int64_t j = 0;
  for (; j < n; ++j) {
    const int64_t row = first + j * nw;
    const float r = r_next;
    if (j + 1 < n) r_next = rstd[row + nw];  // in flight while this row is worked on
    const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(j & 1);
    // every lane waits (the wait makes the copies visible to it); the warp
    // leaves together if any lane gave up
    const bool landed =
        tc::wait_bar_inline(bar, static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status);
    if (!__all_sync(0xffffffffu, landed)) break;
    const bf16* sdn = reinterpret_cast<const bf16*>(ring + (j & 1) * stage_bytes);
    const bf16* sx = sdn + d;
    const bf16* sg = sdn + 2 * d;
    // dn' and x are read from the stage twice (for the row sum, then for the
    // outputs) rather than held in registers across the warp reduction
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int c = u * 256 + lane * 8;
      Pack8<bf16> a, b;
      if (c < d) {
        a.load(sdn + c);
        b.load(sx + c);
      } else {
        a.zero();
        b.zero();
      }
      const Pack8<bf16> wu = weights(u);
#pragma unroll
      for (int i = 0; i < 8; ++i) s = fmaf(a[i] * wu[i], b[i], s);
    }
    s = warp_sum(s);
    const float coef = r * r * s * inv_d;
    bf16* o = dx + row * d;
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int c = u * 256 + lane * 8;
      if (c < d) {
        Pack8<bf16> a, b, g;
        a.load(sdn + c);
        b.load(sx + c);
        g.load(sg + c);
        const Pack8<bf16> wu = weights(u);
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          out[i] = g[i] + (a[i] * wu[i] - b[i] * coef);
          acc[u][i] = fmaf(a[i], b[i], acc[u][i]);
        }
        Vec8<bf16>::store(o + c, out);
      }
    }
    __syncwarp();  // every lane has read the stage
    if (lane == 0 && j + 2 < n) {
      tc::fence_proxy_async();
      issue(j + 2);
    }
  }
  if (j < n) {
    // a wait gave up: let this warp's copies still in flight (rows j and j + 1)
    // land before the block's shared memory is reused or released
    for (int64_t k = j; k < n && k < j + 2; ++k) {
      const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(k & 1);
      const unsigned long long t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(bar, static_cast<uint32_t>(k >> 1) & 1u) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
  // block sum of the warps' dw columns, in warp order, through shared memory
  __syncthreads();
  float* red = reinterpret_cast<float*>(nbs);  // [nw][d], inside the stages
#pragma unroll
  for (int u = 0; u < NP; ++u) {
    const int c = u * 256 + lane * 8;
    if (c < d) {
      float* p = red + static_cast<size_t>(warp) * d + c;
      *reinterpret_cast<float4*>(p) = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
      *reinterpret_cast<float4*>(p + 4) = make_float4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
    }
  }
  __syncthreads();
  for (int col = threadIdx.x; col < d; col += blockDim.x) {
    float v = red[col];
    for (int k = 1; k < nw; ++k) v += red[static_cast<size_t>(k) * d + col];
    part[static_cast<int64_t>(blockIdx.x) * d + col] = v;
  }
}

// bf16 rows of 4097 to 256 x 2 NPH columns: each row is split between the two
// warps of a pair (warp h of the pair owns chunks h NPH .. h NPH + NPH - 1 of
// 256 columns), so that a row is worked on twice as fast and a pair can keep
// three stages (dn' | x | dres of one row each): two rows of reads in flight
// while it works on a third. The two halves' row sums meet through shared
// memory behind an mbarrier and are added in a fixed order (warp 0's first).
// Stage refills wait on an "empty" mbarrier that both warps arrive on. Every
// wait is bounded; a pair leaves a row together (each warp posts whether its
// stage landed next to its partial sum), drains its copies in flight and joins
// the block's dw reduction.
constexpr int kPairs = 2, kPairStages = 3;
template <int NPH>
__global__ void __launch_bounds__(kPairs * 64, 1)
    norm_bwd_pair_kernel(const bf16* __restrict__ dn, const bf16* __restrict__ x,
                         const bf16* __restrict__ w, const float* __restrict__ rstd,
                         const bf16* __restrict__ dres, int64_t rows, int d,
                         bf16* __restrict__ dx, float* __restrict__ part, int* status, int unfed) {
  extern __shared__ __align__(128) unsigned char nbs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp >> 1, h = warp & 1;
  const uint32_t row_bytes = static_cast<uint32_t>(d) * 2u;
  const uint32_t stage_bytes = 3u * row_bytes;  // dn' | x | dres
  const size_t off_b = static_cast<size_t>(kPairs) * kPairStages * stage_bytes;
  unsigned char* ring = nbs + static_cast<size_t>(pair) * kPairStages * stage_bytes;
  uint64_t* pb = reinterpret_cast<uint64_t*>(nbs + off_b) + pair * 8;  // full[3] empty[3] xch[2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(nbs + off_b + kPairs * 64);
  volatile float* xsum = reinterpret_cast<volatile float*>(nbs + off_b + kPairs * 64 + 16) + pair * 4;
  volatile int* xok = reinterpret_cast<volatile int*>(nbs + off_b + kPairs * 64 + 16 + kPairs * 16) +
                      pair * 4;
  bf16* sw = reinterpret_cast<bf16*>(nbs + off_b + kPairs * 64 + 16 + kPairs * 32);
  const uint32_t full0 = tc::smem_u32(pb), empty0 = full0 + 24, xch0 = full0 + 48;
  const uint32_t ring0 = tc::smem_u32(ring);
  if (h == 0 && lane == 0) {
    for (int i = 0; i < kPairStages; ++i) {
      tc::mbar_init(full0 + 8u * i, 1);
      tc::mbar_init(empty0 + 8u * i, 2);
    }
    tc::mbar_init(xch0, 2);
    tc::mbar_init(xch0 + 8, 2);
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  // the norm weight is a parameter: no kernel of the stream writes it
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x)
    *reinterpret_cast<uint4*>(sw + 8 * i) = *reinterpret_cast<const uint4*>(w + 8 * i);
  float acc[NPH][8];
#pragma unroll
  for (int k = 0; k < NPH; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[k][i] = 0.f;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  grid_dependency_sync();

  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * rows / gridDim.x;
  const int64_t first = r0 + pair;
  const int64_t n = first < r1 ? (r1 - first + kPairs - 1) / kPairs : 0;  // this pair's rows
  const bool issuer = h == 0 && lane == 0;
  int64_t issued = 0;
  // copies of the pair's row j into stage j % 3 (the issuer)
  auto issue = [&](int64_t j) {
    const int64_t off = (first + j * kPairs) * d;
    const uint32_t st = static_cast<uint32_t>(j % kPairStages);
    const uint32_t bar = full0 + 8u * st;
    const uint32_t dst = ring0 + st * stage_bytes;
    tc::mbar_expect_tx(bar, stage_bytes);
    bulk_load(dst, dn + off, row_bytes, bar);
    bulk_load(dst + row_bytes, x + off, row_bytes, bar);
    bulk_load(dst + 2 * row_bytes, dres + off, row_bytes, bar);
  };
  if (issuer) {
    for (int64_t j = 0; j < n && j < kPairStages; ++j) {
      // (test hook) the first pair's first row is never loaded: its waits must run out
      if (!(j == 0 && unfed && blockIdx.x == 0 && pair == 0)) issue(j);
      issued = j + 1;
    }
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  float r_next = n > 0 ? rstd[first] : 0.f;
  int64_t j = 0;
  for (; j < n; ++j) {
    const int64_t row = first + j * kPairs;
    const float r = r_next;
    if (j + 1 < n) r_next = rstd[row + kPairs];
    const uint32_t st = static_cast<uint32_t>(j % kPairStages);
    const uint32_t uph = static_cast<uint32_t>(j / kPairStages) & 1u;
    const bool landed = __all_sync(
        0xffffffffu, tc::wait_bar_inline(full0 + 8u * st, uph, abort_flag, status));
    const bf16* sdn = reinterpret_cast<const bf16*>(ring + st * stage_bytes);
    const bf16* sx = sdn + d;
    const bf16* sg = sdn + 2 * d;
    float s = 0.f;
    if (landed) {
#pragma unroll
      for (int k = 0; k < NPH; ++k) {
        const int c = (h * NPH + k) * 256 + lane * 8;
        if (c < d) {
          Pack8<bf16> a, b, wu;
          a.load(sdn + c);
          b.load(sx + c);
          wu.load(sw + c);
#pragma unroll
          for (int i = 0; i < 8; ++i) s = fmaf(a[i] * wu[i], b[i], s);
        }
      }
      s = warp_sum(s);
    }
    // post this half's sum and whether its stage landed; meet the other half
    const uint32_t xb = xch0 + 8u * static_cast<uint32_t>(j & 1);
    const int slot = static_cast<int>(j & 1) * 2;
    if (lane == 0) {
      xsum[slot + h] = s;
      xok[slot + h] = landed ? 1 : 0;
      tc::mbar_arrive(xb);
    }
    const bool met = __all_sync(0xffffffffu, tc::wait_bar_inline(
                                                  xb, static_cast<uint32_t>(j >> 1) & 1u,
                                                  abort_flag, status));
    if (!met || !xok[slot] || !xok[slot + 1]) break;
    const float total = xsum[slot] + xsum[slot + 1];
    const float coef = r * r * total * inv_d;
    bf16* o = dx + row * d;
#pragma unroll
    for (int k = 0; k < NPH; ++k) {
      const int c = (h * NPH + k) * 256 + lane * 8;
      if (c < d) {
        Pack8<bf16> a, b, g, wu;
        a.load(sdn + c);
        b.load(sx + c);
        g.load(sg + c);
        wu.load(sw + c);
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          out[i] = g[i] + (a[i] * wu[i] - b[i] * coef);
          acc[k][i] = fmaf(a[i], b[i], acc[k][i]);
        }
        Vec8<bf16>::store(o + c, out);
      }
    }
    __syncwarp();  // every lane of this half has read the stage
    if (lane == 0) tc::mbar_arrive(empty0 + 8u * st);
    if (issuer && j + kPairStages < n) {
      // both halves are done with the stage before it is refilled
      if (!tc::wait_bar_inline(empty0 + 8u * st, uph, abort_flag, status)) break;
      tc::fence_proxy_async();
      issue(j + kPairStages);
      issued = j + kPairStages + 1;
    }
    __syncwarp();
  }
  if (issuer && j < n) {
    // the pair left early: let its copies still in flight land before the
    // block's shared memory is reused or released
    for (int64_t k = j; k < issued; ++k) {
      if (k == 0 && unfed && blockIdx.x == 0 && pair == 0) continue;  // never issued
      const uint32_t bar = full0 + 8u * static_cast<uint32_t>(k % kPairStages);
      const uint32_t ph = static_cast<uint32_t>(k / kPairStages) & 1u;
      const unsigned long long t0 = globaltimer_ns();
      while (!tc::mbar_try_wait(bar, ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
  // block sum of the pairs' dw columns, in pair order, through shared memory
  __syncthreads();
  float* red = reinterpret_cast<float*>(nbs);  // [kPairs][d], inside the stages
#pragma unroll
  for (int k = 0; k < NPH; ++k) {
    const int c = (h * NPH + k) * 256 + lane * 8;
    if (c < d) {
      float* q = red + static_cast<size_t>(pair) * d + c;
      *reinterpret_cast<float4*>(q) = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
      *reinterpret_cast<float4*>(q + 4) = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
  }
  __syncthreads();
  for (int col = threadIdx.x; col < d; col += blockDim.x) {
    float v = red[col];
    for (int k = 1; k < kPairs; ++k) v += red[static_cast<size_t>(k) * d + col];
    part[static_cast<int64_t>(blockIdx.x) * d + col] = v;
  }
}

// dw[col] = sum over blocks b of part[b][col] for the 32 columns of block `cb`:
// each of the 8 warps sums a fixed contiguous range of b, the 8 sums are added
// in warp order.
template <typename T>
__device__ __forceinline__ void colsum_block(const float* __restrict__ part, int nblk, int d,
                                             T* __restrict__ out, int cb) {
  __shared__ float red[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = cb * 32 + lane;
  const int per = (nblk + 7) / 8;
  const int b0 = warp * per, b1 = min(nblk, b0 + per);
  float v = 0.f;
  if (col < d) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) v += part[static_cast<int64_t>(b) * d + col];
  }
  red[warp][lane] = v;
  __syncthreads();
  if (warp == 0 && col < d) {
    float t = red[0][lane];
    for (int k = 1; k < 8; ++k) t += red[k][lane];
    out[col] = from_f<T>(t);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) colsum_kernel(const float* __restrict__ part, int nblk, int d,
                                                     T* __restrict__ out) {
  grid_dependency_sync();
  colsum_block(part, nblk, d, out, static_cast<int>(blockIdx.x));
}

int norm_bwd_blocks(int num_sms) { return 2 * num_sms; }

using NormBwdStream = void (*)(const bf16*, const bf16*, const bf16*, const float*, const bf16*,
                               int64_t, int, bf16*, float*, int*, int);
// the instance for rows of np <= 16 chunks: exact up to 8, then 12 or 16 (the
// chunks past d are skipped); longer rows take norm_bwd_pair_kernel
static int norm_bwd_stream_np(int np) { return np <= 8 ? np : np <= 12 ? 12 : 16; }
static NormBwdStream norm_bwd_stream(int np) {
  static const NormBwdStream k[10] = {
      norm_bwd_stream_kernel<1>, norm_bwd_stream_kernel<2>,  norm_bwd_stream_kernel<3>,
      norm_bwd_stream_kernel<4>, norm_bwd_stream_kernel<5>,  norm_bwd_stream_kernel<6>,
      norm_bwd_stream_kernel<7>, norm_bwd_stream_kernel<8>,  norm_bwd_stream_kernel<12>,
      norm_bwd_stream_kernel<16>};
  static const bool attr = [] {
    for (auto f : k)
      cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kNormBwdStreamSmem));
    return true;
  }();
  (void)attr;
  const int q = norm_bwd_stream_np(np);
  return k[q <= 8 ? q - 1 : q == 12 ? 8 : 9];
}
static int norm_bwd_stream_max_warps(int np) {
  const int q = norm_bwd_stream_np(np);
  return q > 12   ? norm_bwd_stream_warps<16>()
         : q > 8  ? norm_bwd_stream_warps<12>()
         : q > 4  ? norm_bwd_stream_warps<8>()
                  : norm_bwd_stream_warps<1>();
}

template <typename T>
int launch_norm_bwd(Ctx& c, const T* dn, const T* x, const T* w, const float* rstd,
                    const T* dres, int64_t rows, int64_t d, T* dx, float* part, int nblk, T* dw,
                    bool colsum, bool unfed) {
  // bf16 rows of up to 5120 columns are streamed through shared memory (one
  // block per SM); anything else takes the two-pass kernel
  constexpr bool kBf16 = sizeof(T) == 2;
  const bool stream = kBf16 && d <= 5120 && d % 8 == 0;
  prof_start(c);
  if (stream) {
    nblk = std::min(nblk, c.num_sms);
    const int np = static_cast<int>((d + 255) / 256);
    if (np > 16) {
      // rows split between the warps of a pair: three stages of three rows per
      // pair, 64 bytes of barriers per pair, the abort flag, the halves' sums and
      // flags (32 bytes per pair) and the weights
      const size_t smem = static_cast<size_t>(kPairs) * kPairStages * 6 * static_cast<size_t>(d) +
                          kPairs * 64 + 16 + kPairs * 32 + 2 * static_cast<size_t>(d);
      static const bool attr = [] {
        cudaFuncSetAttribute(norm_bwd_pair_kernel<10>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kNormBwdStreamSmem));
        return true;
      }();
      (void)attr;
      track(c, launch_pdl(norm_bwd_pair_kernel<10>, nblk, kPairs * 64, smem, c.stream,
                          reinterpret_cast<const bf16*>(dn), reinterpret_cast<const bf16*>(x),
                          reinterpret_cast<const bf16*>(w), rstd,
                          reinterpret_cast<const bf16*>(dres), rows, static_cast<int>(d),
                          reinterpret_cast<bf16*>(dx), part, c.status, unfed ? 1 : 0));
      note_launch(c, KK_NORM_BWD, -1, 8.0 * rows * d,
                  4.0 * rows * d * sizeof(T) + d * sizeof(T) + 4.0 * rows + 4.0 * nblk * d);
      if (!colsum) return nblk;
      prof_start(c);
      track(c, launch_pdl(colsum_kernel<T>, static_cast<unsigned>((d + 31) / 32), 256, 0, c.stream,
                          part, nblk, static_cast<int>(d), dw));
      note_launch(c, KK_COLSUM, -1, 1.0 * nblk * d, 4.0 * nblk * d + d * sizeof(T));
      return nblk;
    }
    // two stages of three rows per warp, then 16 bytes of barriers per warp, the
    // abort flag (16 bytes) and, past 8 chunks a lane, the weights
    const size_t warp_bytes = 12 * static_cast<size_t>(d) + 16;
    const size_t fixed = 16 + (norm_bwd_stream_np(np) > 8 ? 2 * static_cast<size_t>(d) : 0);
    const int nw = static_cast<int>(std::max<size_t>(
        1, std::min<size_t>(norm_bwd_stream_max_warps(np), (kNormBwdStreamSmem - fixed) / warp_bytes)));
    const size_t smem = warp_bytes * nw + fixed;
    track(c, launch_pdl(norm_bwd_stream(np), nblk, nw * 32, smem, c.stream,
                        reinterpret_cast<const bf16*>(dn), reinterpret_cast<const bf16*>(x),
                        reinterpret_cast<const bf16*>(w), rstd, reinterpret_cast<const bf16*>(dres),
                        rows, static_cast<int>(d), reinterpret_cast<bf16*>(dx), part, c.status,
                        unfed ? 1 : 0));
  } else {
    // as many warps as their column sums fit in shared memory
    const size_t row_bytes = sizeof(float) * static_cast<size_t>(d + d / 8);
    const int nw = static_cast<int>(
        std::max<size_t>(1, std::min<size_t>(8, kNormBwdSmemLimit / row_bytes)));
    const size_t smem = row_bytes * nw;
    static const bool attr = [] {
      cudaFuncSetAttribute(norm_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kNormBwdSmemLimit));
      return true;
    }();
    (void)attr;
    track(c, launch_pdl(norm_bwd_kernel<T>, nblk, nw * 32, smem, c.stream, dn, x, w, rstd, dres,
                        rows, static_cast<int>(d), dx, part));
  }
  note_launch(c, KK_NORM_BWD, -1, 8.0 * rows * d,
              4.0 * rows * d * sizeof(T) + d * sizeof(T) + 4.0 * rows + 4.0 * nblk * d);
  if (!colsum) return nblk;  // the caller sums `part` later (launch_finish)
  prof_start(c);
  track(c, launch_pdl(colsum_kernel<T>, static_cast<unsigned>((d + 31) / 32), 256, 0, c.stream,
                      part, nblk, static_cast<int>(d), dw));
  note_launch(c, KK_COLSUM, -1, 1.0 * nblk * d, 4.0 * nblk * d + d * sizeof(T));
  return nblk;
}

// ---------------------------------------------------------------------------
// end of a bf16 backward: reduction of the GEMM's split tiles (fixed order over
// the k-ranges) and the RMSNorm dw column sums, in one launch
// ---------------------------------------------------------------------------
// Split tile rt, slab y of 256 / (BN / 8) rows (one row per BN / 8 threads, 8
// columns per thread).
__device__ __forceinline__ void tile_reduce_block(const TileReduce& r, int rt, int y) {
  const int t = r.full_units + rt;
  int pi = 0;
  while (pi + 1 < r.nprob && t >= r.p[pi + 1].tile_begin) ++pi;
  const TileReduceProb& q = r.p[pi];
  const int tl = t - q.tile_begin;
  const int64_t m0 = static_cast<int64_t>(tl / q.tiles_n) * r.tile_rows;
  const int64_t n0 = static_cast<int64_t>(tl % q.tiles_n) * r.BN;
  const int per_row = r.BN / 8;
  const int c8 = (threadIdx.x % per_row) * 8;
  const int64_t col = n0 + c8;
  if (col >= q.N) return;
  float cv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    cv[k] = (q.colv != nullptr && col + k < q.N) ? __bfloat162float(q.colv[col + k]) : 1.f;
  const int64_t slot_elems = static_cast<int64_t>(r.tile_rows) * r.BN;
  const float* base = r.part + static_cast<int64_t>(rt) * r.rem_split * slot_elems + c8;
  const int rr = y * (256 / per_row) + threadIdx.x / per_row;
  const int64_t row = m0 + rr;
  if (row >= q.M) return;
  const float* src = base + static_cast<int64_t>(rr) * r.BN;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // four k-ranges' loads in flight at a time; the adds keep k order
  for (int s = 0; s < r.rem_split; s += 4) {
    float b[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s + u < r.rem_split) Vec8<float>::load(src + (s + u) * slot_elems, b[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s + u < r.rem_split) {
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] += b[u][k];
      }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] *= cv[k];
  bf16* o = q.out + row * q.ldo + col;
  if (col + 8 <= q.N) {
    Vec8<bf16>::store(o, a);
  } else {
    for (int k = 0; col + k < q.N; ++k) o[k] = __float2bfloat16_rn(a[k]);
  }
}

static int reduce_slabs(const TileReduce& r) { return r.tile_rows / (256 / (r.BN / 8)); }

// blocks [0, rem_tiles x slabs): split tiles; then (d + 31) / 32 blocks per dw job
__global__ void __launch_bounds__(256) finish_kernel(const TileReduce r) {
  grid_dependency_sync();
  int b = static_cast<int>(blockIdx.x);
  const int slabs = r.rem_tiles > 0 ? r.tile_rows / (256 / (r.BN / 8)) : 1;
  const int nred = r.rem_tiles * slabs;
  if (b < nred) {
    tile_reduce_block(r, b / slabs, b % slabs);
    return;
  }
  b -= nred;
  for (int j = 0; j < r.ncol; ++j) {
    const int nb = (r.col[j].d + 31) / 32;
    if (b < nb) {
      colsum_block(r.col[j].part, r.col[j].nblk, r.col[j].d, r.col[j].out, b);
      return;
    }
    b -= nb;
  }
}

// One CTA: lets the next launch start at once, clears `early`, waits for the
// kernel ahead, clears `late`.
__global__ void __launch_bounds__(256) zero_counters_kernel(int* __restrict__ early, int n_early,
                                                            int* __restrict__ late, int n_late) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int i = threadIdx.x; i < n_early; i += blockDim.x) early[i] = 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < n_late; i += blockDim.x) late[i] = 0;
}

void launch_zero_counters(Ctx& c, int* early, int64_t n_early, int* late, int64_t n_late) {
  prof_start(c);
  track(c, launch_pdl(zero_counters_kernel, 1, 256, 0, c.stream, early, static_cast<int>(n_early),
                      late, static_cast<int>(n_late)));
  note_launch(c, KK_ELEMENTWISE, -1, 0.0, 4.0 * static_cast<double>(n_early + n_late));
}

void launch_finish(Ctx& c, const TileReduce& r) {
  int blocks = r.rem_tiles > 0 ? r.rem_tiles * reduce_slabs(r) : 0;
  double flops = 0, bytes = 0;
  if (r.rem_tiles > 0) {
    const double elems = static_cast<double>(r.rem_tiles) * r.tile_rows * r.BN;
    flops += elems * r.rem_split;
    bytes += elems * (4.0 * r.rem_split + 2.0);
  }
  for (int j = 0; j < r.ncol; ++j) {
    blocks += static_cast<int>((r.col[j].d + 31) / 32);
    flops += static_cast<double>(r.col[j].nblk) * r.col[j].d;
    bytes += (4.0 * r.col[j].nblk + 2.0) * r.col[j].d;
  }
  if (blocks == 0) return;
  prof_start(c);
  track(c, launch_pdl(finish_kernel, static_cast<unsigned>(blocks), 256, 0, c.stream, r));
  note_launch(c, r.rem_tiles > 0 ? KK_SPLITK_REDUCE : KK_COLSUM, -1, flops, bytes);
}

// ---------------------------------------------------------------------------
// elementwise passes
// ---------------------------------------------------------------------------
template <typename T, int OP>
__device__ __forceinline__ float ew_op(float a, float b, float rv, int sigma) {
  if (OP == 0) return act_t<T>(a, sigma);
  if (OP == 1) return __fmul_rn(silu_t<T>(a), b);
  return a * rv;
}

// OP 0: h = sigma(z); 1: m = SiLU(G) U; 2: out = in * rowv (in == nullptr: zeros).
// Rows are processed 8 columns (16 bytes of bf16) at a time when every row
// stride is a multiple of 8 elements; the columns past the last whole group of
// 8, and unaligned layouts, go element by element. Both forms evaluate the
// same expression per element, so results do not depend on the form.
template <typename T, int OP>
__global__ void ew_kernel(const T* __restrict__ a, int64_t lda, const T* __restrict__ b,
                          int64_t rows, int64_t cols, const float* __restrict__ rowv, int sigma,
                          T* __restrict__ out, int64_t ldo, int vec) {
  grid_dependency_sync();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t nvec = vec ? cols / 8 : 0;  // whole 8-column groups per row
  for (int64_t i = t0; i < rows * nvec; i += stride) {
    const int64_t r = i / nvec, col = (i - r * nvec) * 8;
    float va[8], vb[8], vo[8];
    const float rv = (OP == 2) ? rowv[r] : 0.f;
    if (OP == 2 && a == nullptr) {
#pragma unroll
      for (int k = 0; k < 8; ++k) va[k] = 0.f;
    } else {
      Vec8<T>::load(a + r * lda + col, va);
    }
    if (OP == 1) Vec8<T>::load(b + r * lda + col, vb);
#pragma unroll
    for (int k = 0; k < 8; ++k) vo[k] = ew_op<T, OP>(va[k], OP == 1 ? vb[k] : 0.f, rv, sigma);
    Vec8<T>::store(out + r * ldo + col, vo);
  }
  const int64_t tail = cols - nvec * 8;  // the remaining columns of every row
  for (int64_t i = t0; i < rows * tail; i += stride) {
    const int64_t r = i / tail, col = nvec * 8 + (i - r * tail);
    const float va = (OP == 2 && a == nullptr) ? 0.f : to_f<T>(a[r * lda + col]);
    const float vb = (OP == 1) ? to_f<T>(b[r * lda + col]) : 0.f;
    out[r * ldo + col] = from_f<T>(ew_op<T, OP>(va, vb, OP == 2 ? rowv[r] : 0.f, sigma));
  }
}

template <typename T, int OP>
static void launch_ew(Ctx& c, const T* a, int64_t lda, const T* b, int64_t rows, int64_t cols,
                      const float* rowv, int sigma, T* out, int64_t ldo) {
  const int64_t n = rows * cols;
  // 16-byte vectors need 16-byte aligned rows in every tensor the kernel touches
  const uintptr_t mis = reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                        reinterpret_cast<uintptr_t>(out);
  const bool vec = (mis & 15) == 0 && (lda * sizeof(T)) % 16 == 0 && (ldo * sizeof(T)) % 16 == 0;
  const int64_t work = vec ? (n + 7) / 8 : n;
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, c.num_sms * 8)));
  prof_start(c);
  track(c, launch_pdl(ew_kernel<T, OP>, grid, 256, 0, c.stream, a, lda, b, rows, cols, rowv, sigma,
                      out, ldo, vec ? 1 : 0));
  note_launch(c, KK_ELEMENTWISE, OP, 4.0 * n, (OP == 1 ? 3.0 : 2.0) * n * sizeof(T));
}

template <typename T>
void launch_sigma(Ctx& c, const T* z, int64_t rows, int64_t cols, int64_t ldz, T* h, int64_t ldh,
                  int sigma) {
  launch_ew<T, 0>(c, z, ldz, nullptr, rows, cols, nullptr, sigma, h, ldh);
}
template <typename T>
void launch_swiglu(Ctx& c, const T* G, const T* U, int64_t rows, int64_t cols, int64_t ld, T* m,
                   int64_t ldm) {
  launch_ew<T, 1>(c, G, ld, U, rows, cols, nullptr, 0, m, ldm);
}
template <typename T>
void launch_rowscale(Ctx& c, const T* in, int64_t ldi, const float* rowv, int64_t rows,
                     int64_t cols, T* out, int64_t ldo) {
  launch_ew<T, 2>(c, in, ldi, nullptr, rows, cols, rowv, 0, out, ldo);
}

#define BN_INSTANTIATE(T)                                                                        \
  template void launch_stats<T>(Ctx&, const T*, int64_t, int64_t, int, float, float*, float*);   \
  template void launch_stats_fold<T>(Ctx&, const T*, int64_t, int64_t, int, float, float*, float*, \
                                     const FoldJob<T>&, const FoldJob<T>&);                    \
  template int launch_norm_bwd<T>(Ctx&, const T*, const T*, const T*, const float*, const T*,   \
                                  int64_t, int64_t, T*, float*, int, T*, bool, bool);                  \
  template void launch_sigma<T>(Ctx&, const T*, int64_t, int64_t, int64_t, T*, int64_t, int);    \
  template void launch_swiglu<T>(Ctx&, const T*, const T*, int64_t, int64_t, int64_t, T*,        \
                                 int64_t);                                                       \
  template void launch_rowscale<T>(Ctx&, const T*, int64_t, const float*, int64_t, int64_t, T*,  \
                                   int64_t);
BN_INSTANTIATE(float)
BN_INSTANTIATE(bf16)

}  // namespace bn
