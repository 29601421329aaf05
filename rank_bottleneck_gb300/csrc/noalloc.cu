// bn_weight_grad_noalloc: the split-K weight-gradient GEMM of the backward
// pass, with its scratch in a fixed device array owned by this library instead
// of a buffer from the caller.
//
// Who needs it: code that must not allocate GPU memory at all, e.g. a caller
// whose memory is fully reserved up front by its own pool, or code that runs
// where a cudaMalloc would synchronise the device or is forbidden. Those callers
// still own and pass every input and output; only the fp32 partial tiles of
// the K split (and the device status word) live here.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/boostblk.h"
#include "gemm.h"

namespace bn {
namespace {

// Fixed scratch: 256 bytes of status word, then the fp32 partial tiles (at most
// one 128 x 256 tile per SM, whatever the problem's size). Every GPU that loads
// this library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr size_t kStatusBytes = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per
// device with that device current. In host code `g_noalloc_scratch` names a host
// stand-in, never the device memory, so kernels must get this address instead.
bn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BN_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return BN_OK;
}

}  // namespace
}  // namespace bn

using namespace bn;

extern "C" bn_status bn_weight_grad_noalloc(int64_t M, int64_t N, int64_t T, const void* A,
                                            int64_t lda, const void* B, int64_t ldb,
                                            const void* colscale, void* dW, int64_t ldw,
                                            bn_stream_t stream) {
  if (M < 1 || N < 1 || T < 1 || !A || !B || !dW || lda < M || ldb < N || ldw < N)
    return BN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                        reinterpret_cast<uintptr_t>(dW) | reinterpret_cast<uintptr_t>(colscale);
  if ((mis & 15) || (lda % 8) || (ldb % 8) || (ldw % 8)) return BN_ERR_ALIGNMENT;

  void* scratch = nullptr;
  bn_status st = scratch_address(&scratch);
  if (st != BN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the partial tiles are fully overwritten
  if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess) return BN_ERR_CUDA;

  GemmLaunch g;
  g.epi = EPI_STORE;
  g.allow_split = true;
  g.nprob = 1;
  GemmProblem& p = g.p[0];
  p.M = M;
  p.N = N;
  p.K = T;
  p.a[0].ptr = A;
  p.a[0].ld = lda;
  p.a[0].mn_major = true;
  p.b[0].ptr = B;
  p.b[0].ld = ldb;
  p.b[0].mn_major = true;
  p.out[0] = dW;
  p.ldo[0] = ldw;
  p.colv = colscale;

  Ctx c;
  c.stream = s;
  c.status = static_cast<int*>(scratch);
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && nsm > 0)
    c.num_sms = nsm;
  c.partial = reinterpret_cast<float*>(static_cast<char*>(scratch) + kStatusBytes);
  c.partial_bytes = kNoAllocScratchBytes - kStatusBytes;
  if (c.partial_bytes < gemm_tc_partial_bytes(c.num_sms)) return BN_ERR_UNSUPPORTED;
  gemm_tc(c, g);
  if (c.bad) return BN_ERR_UNSUPPORTED;
  if (c.err != cudaSuccess) return BN_ERR_CUDA;
  return BN_OK;
}
