// Launchers of the tcgen05 GEMM kernel instantiations (one translation unit
// per tile width and CTA grouping so they compile in parallel).
#pragma once
#include <cuda_runtime.h>
#include "gemm_tc_kernel.cuh"

namespace bn {
namespace tc {
// Launch kind `ek` with operand majorness (a_mn, b_mn) over `units` work units.
// Returns the CTAs launched, 0 if there is no such instantiation (or it cannot
// run). CG = 2 launches clusters of two CTAs (one 256-row tile per pair).
int launch_bn128_cg1(int ek, bool a_mn, bool b_mn, const Params& P, int units, int num_sms,
                     cudaStream_t s);
int launch_bn256_cg1(int ek, bool a_mn, bool b_mn, const Params& P, int units, int num_sms,
                     cudaStream_t s);
int launch_bn128_cg2(int ek, bool a_mn, bool b_mn, const Params& P, int units, int num_sms,
                     cudaStream_t s);
int launch_bn256_cg2(int ek, bool a_mn, bool b_mn, const Params& P, int units, int num_sms,
                     cudaStream_t s);
}  // namespace tc
}  // namespace bn
