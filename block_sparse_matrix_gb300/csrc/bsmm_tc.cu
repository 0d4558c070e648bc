// tcgen05 tensor-core kernels (16-bit inputs, float32 accumulation in TMEM).
#include "bsmm_internal.cuh"

bool tc_supported(bsmm_ctx *, bsmm_dtype) { return false; }
bsmm_status tc_fprop(bsmm_ctx *, const void *, const void *, void *, int, bsmm_dtype, cudaStream_t)
{
    return BSMM_ERR_UNSUPPORTED;
}
bsmm_status tc_bprop(bsmm_ctx *, const void *, const void *, void *, int, bsmm_dtype, cudaStream_t)
{
    return BSMM_ERR_UNSUPPORTED;
}
bsmm_status tc_updat(bsmm_ctx *, const GroupPtrs &, float *, int, bsmm_dtype, int, cudaStream_t)
{
    return BSMM_ERR_UNSUPPORTED;
}
void tc_release(bsmm_ctx *) {}
