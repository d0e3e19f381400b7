// bf16 matmuls on the tcgen05 tensor cores.  (Placeholder until the kernel lands:
// every entry reports GPT2_EUNSUPPORTED and the FMA kernel runs.)
#include "gemm_tc.h"
#include "../../include/gpt2.h"

int gemm_tc_available() { return 0; }
size_t gemm_tc_scratch_floats(size_t, size_t) { return 0; }
int gemm_tc_forward(cudaStream_t, __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
                    const __nv_bfloat16*, int, int, int, int, __nv_bfloat16*) {
    return GPT2_EUNSUPPORTED;
}
int gemm_tc_backward_dx(cudaStream_t, __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, int, int,
                        int, int, const __nv_bfloat16*) {
    return GPT2_EUNSUPPORTED;
}
int gemm_tc_backward_dw(cudaStream_t, float*, const __nv_bfloat16*, const __nv_bfloat16*, int, int, int,
                        float*, size_t) {
    return GPT2_EUNSUPPORTED;
}
