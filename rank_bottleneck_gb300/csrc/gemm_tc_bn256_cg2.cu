// tcgen05 GEMM instantiations: 256-column tiles, CTA group of 2.
#define GEMM_BN 256
#define GEMM_CG 2
#include "gemm_tc_inst.cuh"
