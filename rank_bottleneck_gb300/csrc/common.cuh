// Device helpers shared by the block library's kernels: element conversion,
// the bottleneck nonlinearities, the device status word and bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace bn {

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation: it may be scheduled while the kernel before it on the stream
// drains, and runs its setup meanwhile. Before it touches global memory (reads
// the predecessor's results, or writes what the predecessor may still read) it
// waits for the predecessor to complete. The wait is unconditional and comes
// before any early exit, so a kernel's completion implies its predecessor's.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Most GEMM problems in one engine launch (the block's weight gradients go out
// together: 11 of them).
constexpr int kMaxProblems = 16;

// Chained launches (tcgen05 engine). A producer launch counts, per row block of
// its tiles (CG x 128 rows), the epilogue warps whose output stores of that
// block have landed (`rows`), and its CTAs once past their grid-dependency wait
// (`entered`). The launch right after it on the stream, the consumer, then
// reads the producer's output as its A operand without waiting for the whole
// producer grid: it waits for `entered` to reach entered_target (so every
// earlier kernel is complete) and, per tile, for its row block's count to reach
// rows_target. Its CTAs start on the SMs the producer's last round leaves idle.
// The producer must not read what the consumer writes. Counters start at zero.
struct ChainLink {
  int* entered = nullptr;
  int* rows = nullptr;
  int entered_target = 0, rows_target = 0;
};

// Device status word bits (first word of the caller's scratch buffer).
constexpr int kStatusTimeout = 1;

// Upper limit of any single wait inside a kernel. Legitimate waits last
// microseconds; after this much wall time the kernel records a timeout,
// unwinds and returns instead of spinning on.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// element conversion
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
// Round a float to the storage precision of T and back.
template <typename T> __device__ __forceinline__ float round_to(float v) {
  return to_f<T>(from_f<T>(v));
}

// ---------------------------------------------------------------------------
// nonlinearities. Written with explicit round-to-nearest intrinsics so that
// every kernel that evaluates them (GEMM epilogues, the recompute kernel of
// checkpoint mode) produces bit-identical results: no FMA contraction can
// differ between call sites.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sigmoid_f(float z) {
  return __frcp_rn(__fadd_rn(1.0f, expf(-z)));
}
__device__ __forceinline__ float silu_f(float z) { return __fmul_rn(z, sigmoid_f(z)); }
// d/dz SiLU(z) = s (1 + z (1 - s)), s = sigmoid(z)
__device__ __forceinline__ float silu_grad_f(float z) {
  float s = sigmoid_f(z);
  return __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(z, __fsub_rn(1.0f, s))));
}
// sigma: 0 = identity, 1 = SiLU (bn_sigma)
__device__ __forceinline__ float act_f(float z, int sigma) { return sigma ? silu_f(z) : z; }
__device__ __forceinline__ float act_grad_f(float z, int sigma) {
  return sigma ? silu_grad_f(z) : 1.0f;
}

// Compact forms for bf16 data, whose results are rounded to 8 significant
// bits: sigmoid(z) = 1 / (1 + 2^(-z log2 e)) from the hardware's approximate
// base-2 exponential and reciprocal (relative error near 2^-22, far below
// bf16's 2^-9). Every bf16 kernel uses these same instruction sequences, so
// the forward epilogues and the checkpoint recompute stay bit-identical.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_fast(float z) {
  return rcp_approx(__fadd_rn(1.0f, ex2_approx(__fmul_rn(z, -1.4426950408889634f))));
}
__device__ __forceinline__ float silu_fast(float z) { return __fmul_rn(z, sigmoid_fast(z)); }
__device__ __forceinline__ float silu_grad_fast(float z) {
  const float s = sigmoid_fast(z);
  return __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(z, __fsub_rn(1.0f, s))));
}
__device__ __forceinline__ float act_fast(float z, int sigma) { return sigma ? silu_fast(z) : z; }
__device__ __forceinline__ float act_grad_fast(float z, int sigma) {
  return sigma ? silu_grad_fast(z) : 1.0f;
}
// The nonlinearities for element type T: compact for bf16, accurate for fp32.
template <typename T> __device__ __forceinline__ float act_t(float z, int sigma);
template <> __device__ __forceinline__ float act_t<float>(float z, int sigma) { return act_f(z, sigma); }
template <> __device__ __forceinline__ float act_t<__nv_bfloat16>(float z, int sigma) {
  return act_fast(z, sigma);
}
template <typename T> __device__ __forceinline__ float silu_t(float z);
template <> __device__ __forceinline__ float silu_t<float>(float z) { return silu_f(z); }
template <> __device__ __forceinline__ float silu_t<__nv_bfloat16>(float z) { return silu_fast(z); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// 8-element vectors (16 bytes of bf16, 32 bytes of fp32)
// ---------------------------------------------------------------------------
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* f) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* f) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};
template <> struct Vec8<float> {
  __device__ __forceinline__ static void load(const float* p, float* f) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
};

}  // namespace bn
