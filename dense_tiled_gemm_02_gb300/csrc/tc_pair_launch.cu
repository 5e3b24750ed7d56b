// tc_pair_launch.cu -- instantiations and cluster launches of the CTA-pair
// (cta_group::2) GEMM kernel.
#include <cuda_runtime.h>

#include "tc_gemm2.cuh"
#include "tc_launch.h"

namespace gb300 {

namespace {
template <int BN, int STAGES, int KSUB, bool I8X>
cudaLaunchConfig_t pair_config(int grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(PairCfg<BN, KSUB, I8X>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes<BN, STAGES, KSUB, I8X>();
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel in the stream finishes (pdl_wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int BN, int STAGES, int KSUB, bool I8X>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                        const CUtensorMap& c, const KParams& p, int grid, cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<BN, STAGES, KSUB, I8X>(grid, st, attr);
  return cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<BN, STAGES, KSUB, I8X>, a, b, d, c, p);
}

template <int BN, int STAGES, int KSUB, bool I8X>
cudaError_t prepare_pair() {
  return cudaFuncSetAttribute(tc_gemm_pair_kernel<BN, STAGES, KSUB, I8X>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              pair_smem_bytes<BN, STAGES, KSUB, I8X>());
}

template <int BN, int STAGES, int KSUB, bool I8X>
int max_clusters_pair() {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<BN, STAGES, KSUB, I8X>(2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<BN, STAGES, KSUB, I8X>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}
}  // namespace

#define GB_PAIR(BN_, ST_, KS_, I8_)                                                 \
  PairVariant{BN_, ST_, KS_, I8_, pair_smem_bytes<BN_, ST_, KS_, I8_>(),            \
              &launch_pair<BN_, ST_, KS_, I8_>, &prepare_pair<BN_, ST_, KS_, I8_>, \
              &max_clusters_pair<BN_, ST_, KS_, I8_>}

const PairVariant kPairVariants[] = {GB_PAIR(256, 6, 1, false), GB_PAIR(256, 3, 2, false),
                                     GB_PAIR(224, 6, 1, false), GB_PAIR(128, 8, 1, false),
                                     GB_PAIR(128, 4, 2, false), GB_PAIR(256, 5, 1, true)};
const int kNumPairVariants = 6;

}  // namespace gb300
