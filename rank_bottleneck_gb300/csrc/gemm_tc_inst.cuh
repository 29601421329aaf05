// Instantiations of the tcgen05 GEMM kernel for one tile width (GEMM_BN) and
// one CTA grouping (GEMM_CG); included by the gemm_tc_bn*_cg*.cu units.
#include <mutex>

#include "gemm_tc_launch.h"

namespace bn {
namespace tc {
namespace {

template <int EK, bool AMN, bool BMN>
int go(const Params& P, int units, int num_sms, cudaStream_t s) {
  constexpr int BN = GEMM_BN, CG = GEMM_CG;
  auto k = gemm_kernel<BN, EK, AMN, BMN, CG>;
  constexpr int SMEM = Cfg<BN, EK, CG>::SMEM_BYTES;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(kernel_threads<EK>(), 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  if (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // persistent grid: as many CTAs (pairs) as can be resident at once
  static int max_groups = 0;
  static bool usable = true;
  static std::once_flag once;
  std::call_once(once, [&] {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (is_fold<EK>()) {
      // its warpgroups trade registers (setmaxnreg) on the assumption that every
      // thread is launched with kNormRegsLaunch of them: with fewer the trade
      // could not complete, so the kernel is not launched at all
      cudaFuncAttributes fa;
      usable = cudaFuncGetAttributes(&fa, k) == cudaSuccess && fa.numRegs == kNormRegsLaunch;
      cudaGetLastError();
    }
    int n = 0;
    if (CG == 2) {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * num_sms, 1, 1);
      if (cudaOccupancyMaxActiveClusters(&n, k, &q) != cudaSuccess || n <= 0) n = num_sms / 2;
      cudaGetLastError();
    } else {
      n = num_sms;
    }
    max_groups = n;
  });
  if (!usable) return 0;
  const int groups = units < max_groups ? units : max_groups;
  cfg.gridDim = dim3(groups * CG, 1, 1);
  // programmatic dependent launch (see grid_dependency_sync)
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs += 1;
  cudaLaunchKernelEx(&cfg, k, P);
  return groups * CG;
}

}  // namespace

#define BN_CAT2(a, b, c) a##b##c
#define BN_CAT(a, b, c) BN_CAT2(a, b, c)
int BN_CAT(launch_bn, GEMM_BN, BN_CAT(_cg, GEMM_CG, ))(int ek, bool a_mn, bool b_mn,
                                                        const Params& P, int units, int num_sms,
                                                        cudaStream_t s) {
  const int key = ek * 4 + (a_mn ? 2 : 0) + (b_mn ? 1 : 0);
  switch (key) {
    case K_STORE * 4 + 0: return go<K_STORE, false, false>(P, units, num_sms, s);
    case K_STORE * 4 + 1: return go<K_STORE, false, true>(P, units, num_sms, s);
    case K_STORE * 4 + 3: return go<K_STORE, true, true>(P, units, num_sms, s);
    case K_SIGMA * 4 + 0: return go<K_SIGMA, false, false>(P, units, num_sms, s);
    case K_RESID * 4 + 0: return go<K_RESID, false, false>(P, units, num_sms, s);
    case K_DSIGMA * 4 + 1: return go<K_DSIGMA, false, true>(P, units, num_sms, s);
    case K_DSWIGLU * 4 + 1: return go<K_DSWIGLU, false, true>(P, units, num_sms, s);
    case K_CHAIN * 4 + 1: return go<K_CHAIN, false, true>(P, units, num_sms, s);
    case K_NORM * 4 + 0: return go<K_NORM, false, false>(P, units, num_sms, s);
    case K_SDSIGMA * 4 + 1: return go<K_SDSIGMA, false, true>(P, units, num_sms, s);
    case K_SWIGLU * 4 + 0: return go<K_SWIGLU, false, false>(P, units, num_sms, s);
    default: return 0;
  }
}

}  // namespace tc
}  // namespace bn
