// Launchers of the tcgen05 GEMM kernel instantiations (one translation unit
// per tile width so they compile in parallel).
#pragma once
#include <cuda_runtime.h>
#include "gemm_tc_kernel.cuh"

namespace bn {
namespace tc {
// Returns false if (ek, a_mn, b_mn) has no instantiation at this tile width.
bool launch_bn128(int ek, bool a_mn, bool b_mn, const Params& P, int grid, cudaStream_t s);
bool launch_bn256(int ek, bool a_mn, bool b_mn, const Params& P, int grid, cudaStream_t s);
}  // namespace tc
}  // namespace bn
