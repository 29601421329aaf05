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
#include "../../include/boostblk_testing.h"
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

bn_status cuda_failed(cudaError_t e) { return static_cast<bn_status>(record_cuda_error(e)); }

// Device address of the scratch array on the current device, looked up once per
// device with that device current. In host code `g_noalloc_scratch` names a host
// stand-in, never the device memory, so kernels must get this address instead.
bn_status scratch_address(void** out, int* device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failed(e);
  if (dev < 0 || dev >= kMaxDevices) return BN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_failed(e);
    if (p == nullptr) return BN_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  *device = dev;
  return BN_OK;
}

// The weight-gradient launch on the fixed array. `unfed` (tests only) makes the
// launch a chained consumer of an upstream launch that never comes, so that its
// bounded wait runs out.
bn_status weight_grad(int64_t M, int64_t N, int64_t T, const void* A, int64_t lda, const void* B,
                      int64_t ldb, const void* colscale, void* dW, int64_t ldw,
                      bn_stream_t stream, int* unfed) {
  if (M < 1 || N < 1 || T < 1 || !A || !B || !dW || lda < M || ldb < N || ldw < N)
    return BN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                        reinterpret_cast<uintptr_t>(dW) | reinterpret_cast<uintptr_t>(colscale);
  if ((mis & 15) || (lda % 8) || (ldb % 8) || (ldw % 8)) return BN_ERR_ALIGNMENT;

  void* scratch = nullptr;
  int dev = 0;
  bn_status st = scratch_address(&scratch, &dev);
  if (st != BN_OK) return st;
  int nsm = 0;
  cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_failed(e);
  if (nsm < 1) return BN_ERR_UNSUPPORTED;
  const size_t partial_bytes = kNoAllocScratchBytes - kStatusBytes;
  if (partial_bytes < gemm_tc_partial_bytes(nsm)) return BN_ERR_UNSUPPORTED;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the partial tiles are fully overwritten
  e = cudaMemsetAsync(scratch, 0, kStatusBytes, s);
  if (e != cudaSuccess) return cuda_failed(e);

  GemmLaunch g;
  g.epi = EPI_STORE;
  g.allow_split = unfed == nullptr;
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
  c.num_sms = nsm;
  c.partial = reinterpret_cast<float*>(static_cast<char*>(scratch) + kStatusBytes);
  c.partial_bytes = partial_bytes;
  if (unfed != nullptr) {
    c.chain_in.entered = unfed;
    c.chain_in.rows = unfed + 1;
    c.chain_in.entered_target = 1;
    c.chain_in.rows_target = 1;
  }
  gemm_tc(c, g);
  if (c.bad) return BN_ERR_UNSUPPORTED;
  if (c.err != cudaSuccess) return cuda_failed(c.err);
  return BN_OK;
}

}  // namespace
}  // namespace bn

using namespace bn;

extern "C" bn_status bn_weight_grad_noalloc(int64_t M, int64_t N, int64_t T, const void* A,
                                            int64_t lda, const void* B, int64_t ldb,
                                            const void* colscale, void* dW, int64_t ldw,
                                            bn_stream_t stream) {
  return weight_grad(M, N, T, A, lda, B, ldb, colscale, dW, ldw, stream, nullptr);
}

extern "C" bn_status bn_weight_grad_noalloc_status(bn_stream_t stream) {
  void* scratch = nullptr;
  int dev = 0;
  bn_status st = scratch_address(&scratch, &dev);
  if (st != BN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(scratch, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_failed(e);
  return (word & kStatusTimeout) ? BN_ERR_TIMEOUT : BN_OK;
}

extern "C" bn_status bn_testing_weight_grad_noalloc_unfed(int64_t M, int64_t N, int64_t T,
                                                          const void* A, int64_t lda,
                                                          const void* B, int64_t ldb, void* dW,
                                                          int64_t ldw, int* counters,
                                                          bn_stream_t stream) {
  if (counters == nullptr || M > 256) return BN_ERR_INVALID_ARG;
  return weight_grad(M, N, T, A, lda, B, ldb, nullptr, dW, ldw, stream, counters);
}
