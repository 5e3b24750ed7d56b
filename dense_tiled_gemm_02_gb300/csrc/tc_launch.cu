// tc_launch.cu -- instantiations and launchers of the tcgen05 GEMM kernel.
// Compiled once per tile width (TC_BN) so that the instantiations build in
// parallel.
#include <cuda_runtime.h>

#include "tc_gemm.cuh"
#include "tc_launch.h"

#ifndef TC_BN
#error "TC_BN must be defined"
#endif

namespace gb300 {

namespace {
// CS > 1 with p.csk > 1: clusters of p.csk CTAs (cluster split-K).
template <int BN, int STAGES, bool I8X, int PW, int CS>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b, const KParams& p, int grid,
                        cudaStream_t st) {
  constexpr uint32_t smem = smem_bytes<BN, STAGES, PW, CS>();
  auto kernel = tc_gemm_kernel<BN, STAGES, I8X, PW, CS>;
  if (CS == 1 || p.csk <= 1)
    return launch_pdl(kernel, dim3(grid), dim3(NUM_THREADS + 32 * PW), smem, st, a, b, p);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NUM_THREADS + 32 * PW);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.csk);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a, b, p);
}

template <int BN, int STAGES, bool I8X, int PW, int CS>
cudaError_t prepare_impl() {
  constexpr uint32_t smem = smem_bytes<BN, STAGES, PW, CS>();
  return cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, I8X, PW, CS>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}
}  // namespace

#define GB_VARIANT(BN_, ST_, I8_, PW_, CS_)                                           \
  TcVariant{BN_, ST_, I8_, PW_, CS_, smem_bytes<BN_, ST_, PW_, CS_>(),                \
            &launch_impl<BN_, ST_, I8_, PW_, CS_>, &prepare_impl<BN_, ST_, I8_, PW_, CS_>}

// Cluster split-K variants give up ring stages for the landing slots.
#if TC_BN == 256
const TcVariant kVariantsBN256[] = {GB_VARIANT(256, 4, false, 0, 1),
                                    GB_VARIANT(256, 4, false, 4, 1)};
const int kNumVariantsBN256 = 2;
#elif TC_BN == 128
const TcVariant kVariantsBN128[] = {GB_VARIANT(128, 7, false, 0, 1), GB_VARIANT(128, 6, true, 0, 1),
                                    GB_VARIANT(128, 6, false, 4, 1),
                                    GB_VARIANT(128, 5, false, 0, 2)};
const int kNumVariantsBN128 = 4;
#elif TC_BN == 64
const TcVariant kVariantsBN64[] = {GB_VARIANT(64, 9, false, 0, 1), GB_VARIANT(64, 8, false, 0, 2),
                                   GB_VARIANT(64, 5, false, 0, 4)};
const int kNumVariantsBN64 = 3;
#endif

}  // namespace gb300
