// attn_tc_split.cu -- the tensor-core attention kernel's layer-path variant: split schedule with
// every row written a second time as the bf16 hi/lo pair that o_proj's bf16x3 product reads (page
// "inferencelayer 0.2.3, src/diffusion_gemma_gpu.rs", item DG_ATTN followed by the output
// projection).  Head sizes 128 and 256 (those the projections take).  Compiled on its own so that
// the default instantiations in attn_tc.cu are unaffected by it.
#include "attn_tc_kernel.cuh"

namespace dg {

cudaError_t attn_tc_split_prepare(int hd)
{
    switch (hd) {
    case 128:
        return cudaFuncSetAttribute(attn_tc_kernel<128, false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<128>::SMEM_BYTES);
    case 256:
        return cudaFuncSetAttribute(attn_tc_kernel<256, false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<256>::SMEM_BYTES);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn_tc_split(const cudaLaunchConfig_t &cfg, const TcMaps &maps,
                                 const AttnTcParams &p, int hd)
{
    switch (hd) {
    case 128: return cudaLaunchKernelEx(&cfg, attn_tc_kernel<128, false, true>, maps, p);
    case 256: return cudaLaunchKernelEx(&cfg, attn_tc_kernel<256, false, true>, maps, p);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
