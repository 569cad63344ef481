// attn_tc.cu -- launch, schedule-side queries and one-time setup of the tensor-core attention
// kernel (attn_tc_kernel.cuh) for its default instantiations: the split schedule writing fp32
// rows and the stream-K schedule.  The variant that also writes the bf16 hi/lo operand split for
// o_proj is compiled in attn_tc_split.cu: kept out of this module, the default kernels' code
// stays exactly as it is without that variant.
#include "attn_tc_kernel.cuh"

namespace dg {
namespace {

template <int HD>
cudaError_t launch_hd(const AttnTcParams &p, const TcMaps &maps, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = p.sk_ctas ? dim3(p.sk_ctas) : dim3((p.rows + kTileM - 1) / kTileM, p.nkv, p.splits);
    cfg.blockDim = dim3(Layout<HD>::THREADS);
    cfg.dynamicSmemBytes = Layout<HD>::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0] = pdl_attribute();
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = p.splits;
    cfg.attrs = attr;
    cfg.numAttrs = p.cluster_combine ? 2 : 1;
    if (p.sk_ctas) return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, true>, maps, p);
    if (p.out_hi) return launch_attn_tc_split(cfg, maps, p, HD);
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, false>, maps, p);
}

template <int HD>
int max_clusters_hd(int splits, int qtiles, int nkv)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(qtiles, nkv, splits);
    cfg.blockDim = dim3(Layout<HD>::THREADS);
    cfg.dynamicSmemBytes = Layout<HD>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = splits;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<HD, false>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int HD>
cudaError_t prepare_hd()
{
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<HD>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_tc_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<HD>::SMEM_BYTES);
}

}  // namespace

TcGeom tc_geometry(int hd)
{
    switch (hd) {
    case 64: return {Cfg<64>::NK, Cfg<64>::VK, Cfg<64>::QL_TMEM};
    case 128: return {Cfg<128>::NK, Cfg<128>::VK, Cfg<128>::QL_TMEM};
    case 256: return {Cfg<256>::NK, Cfg<256>::VK, Cfg<256>::QL_TMEM};
    default: return {0, 0, false};
    }
}

size_t attn_tc_smem_bytes(int hd)
{
    switch (hd) {
    case 64: return Layout<64>::SMEM_BYTES;
    case 128: return Layout<128>::SMEM_BYTES;
    case 256: return Layout<256>::SMEM_BYTES;
    default: return 0;
    }
}

cudaError_t attn_tc_prepare(int hd)
{
    switch (hd) {
    case 64: return prepare_hd<64>();
    case 128: return prepare_hd<128>();
    case 256: return prepare_hd<256>();
    default: return cudaErrorInvalidValue;
    }
}

int attn_tc_max_clusters(int hd, int splits, int qtiles, int nkv)
{
    if (splits < 2 || splits > kMaxClusterSplits) return 0;
    switch (hd) {
    case 64: return max_clusters_hd<64>(splits, qtiles, nkv);
    case 128: return max_clusters_hd<128>(splits, qtiles, nkv);
    case 256: return max_clusters_hd<256>(splits, qtiles, nkv);
    default: return 0;
    }
}

cudaError_t launch_attn_tc(const AttnTcParams &p, const TcMaps &maps, int hd, cudaStream_t s)
{
    switch (hd) {
    case 64: return launch_hd<64>(p, maps, s);
    case 128: return launch_hd<128>(p, maps, s);
    case 256: return launch_hd<256>(p, maps, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
