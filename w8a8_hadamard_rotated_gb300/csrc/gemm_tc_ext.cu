// The tcgen05 GEMM kernels with the extended epilogue (bias, bf16 output,
// bf16 LoRA up weight): the same kernel source as gemm_tc.cu, instantiated
// here for kExt = true so that the two sets of instantiations compile in
// parallel.
#define CONVROT_GEMM_EXT_TU 1
#include "gemm_tc.cu"
