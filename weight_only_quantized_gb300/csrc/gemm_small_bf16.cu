// The small-M GEMM kernels for bf16 layers: the source of gemm_small.cu, built as a second
// translation unit so that the fp16 and bf16 instantiations compile in parallel.
#define GPTQ_SMALL_BF16_UNIT 1
#include "gemm_small.cu"
