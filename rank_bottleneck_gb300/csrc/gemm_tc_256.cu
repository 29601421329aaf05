// tcgen05 GEMM instantiations with 256-column tiles.
#include "gemm_tc_launch.h"

namespace bn {
namespace tc {

template <int EK, bool AMN, bool BMN>
static void go(const Params& P, int grid, cudaStream_t s) {
  auto k = gemm_kernel<256, EK, AMN, BMN>;
  static const bool attr_set = [&]() {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<256, EK>::SMEM_BYTES);
    return true;
  }();
  (void)attr_set;
  k<<<grid, NUM_THREADS, Cfg<256, EK>::SMEM_BYTES, s>>>(P);
}

bool launch_bn256(int ek, bool a_mn, bool b_mn, const Params& P, int grid, cudaStream_t s) {
  const int key = ek * 4 + (a_mn ? 2 : 0) + (b_mn ? 1 : 0);
  switch (key) {
    case K_STORE * 4 + 0: go<K_STORE, false, false>(P, grid, s); return true;
    case K_STORE * 4 + 1: go<K_STORE, false, true>(P, grid, s); return true;
    case K_STORE * 4 + 3: go<K_STORE, true, true>(P, grid, s); return true;
    case K_PART * 4 + 3: go<K_PART, true, true>(P, grid, s); return true;
    case K_SIGMA * 4 + 0: go<K_SIGMA, false, false>(P, grid, s); return true;
    case K_RESID * 4 + 0: go<K_RESID, false, false>(P, grid, s); return true;
    case K_DSIGMA * 4 + 1: go<K_DSIGMA, false, true>(P, grid, s); return true;
    case K_DSWIGLU * 4 + 1: go<K_DSWIGLU, false, true>(P, grid, s); return true;
    case K_CHAIN * 4 + 1: go<K_CHAIN, false, true>(P, grid, s); return true;
    default: return false;
  }
}

}  // namespace tc
}  // namespace bn
