// tcgen05 GEMM instantiations: 128-column tiles, CTA group of 1.
#define GEMM_BN 128
#define GEMM_CG 1
#include "gemm_tc_inst.cuh"
