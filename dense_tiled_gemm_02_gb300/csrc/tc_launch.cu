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
template <int BN, int STAGES, bool I8X, int PW>
cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b, const KParams& p, int grid,
                        cudaStream_t st) {
  constexpr uint32_t smem = smem_bytes<BN, STAGES, PW>();
  return launch_pdl(tc_gemm_kernel<BN, STAGES, I8X, PW>, dim3(grid), dim3(NUM_THREADS + 32 * PW),
                    smem, st, a, b, p);
}

template <int BN, int STAGES, bool I8X, int PW>
cudaError_t prepare_impl() {
  constexpr uint32_t smem = smem_bytes<BN, STAGES, PW>();
  return cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, I8X, PW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}
}  // namespace

#define GB_VARIANT(BN_, ST_, I8_, PW_)                                                          \
  TcVariant{BN_, ST_, I8_, PW_, smem_bytes<BN_, ST_, PW_>(), &launch_impl<BN_, ST_, I8_, PW_>, \
            &prepare_impl<BN_, ST_, I8_, PW_>}

#if TC_BN == 256
const TcVariant kVariantsBN256[] = {GB_VARIANT(256, 4, false, 0), GB_VARIANT(256, 4, false, 4)};
const int kNumVariantsBN256 = 2;
#elif TC_BN == 128
const TcVariant kVariantsBN128[] = {GB_VARIANT(128, 7, false, 0), GB_VARIANT(128, 6, true, 0),
                                    GB_VARIANT(128, 6, false, 4)};
const int kNumVariantsBN128 = 3;
#elif TC_BN == 64
const TcVariant kVariantsBN64[] = {GB_VARIANT(64, 9, false, 0)};
const int kNumVariantsBN64 = 1;
#endif

}  // namespace gb300
