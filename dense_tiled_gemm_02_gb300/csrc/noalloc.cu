// noalloc.cu -- split-K GEMM entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc/cudaFree at the point where they need
// a GEMM: code running under a framework whose caching allocator owns every
// byte of device memory (a side allocation escapes its accounting and can
// fail once the pool has reserved the device), and latency-critical paths
// where cudaFree's implicit device-wide synchronisation, or a slow
// cudaMalloc, is not acceptable.  gemm_create serves everyone else: it
// allocates the split-K workspace and a status word per handle.
//
// This entry point instead keeps its scratch (the device status word and the
// fp32 partial sums of the K splits) in one file-scope __device__ array of
// GEMM_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
// until the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a stand-in object), so the first call on each
// device looks the address up with cudaGetSymbolAddress while that device is
// current and caches it; later calls reuse it.  All calls share the array:
// the status word is cleared at the start of each call and every partial sum
// is rewritten before it is read, and calls whose kernels overlap on the GPU
// race on the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.h"
#include "gemm.h"
#include "plan_table.h"
#include "tc_launch.h"

using namespace gb300;

namespace {

static_assert(GEMM_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// [0, 256): status word; [256, end): split-K partial sums.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

constexpr size_t kPartialOffset = 256;
constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 16;

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns nullptr on failure.
void* scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// Tensor map of a 16-bit operand read in place: K-major storage has dims
// {K, rows} and box {BK, box_rows}; MN-major storage dims {MN, K}, box
// {64, BK}; 128-byte swizzle, zero fill outside the tensor.
bool encode(CUtensorMap* tm, const void* base, int64_t ld, bool k_major, int64_t mn, int64_t K,
            int box_rows) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {k_major ? (cuuint64_t)K : (cuuint64_t)mn,
                        k_major ? (cuuint64_t)mn : (cuuint64_t)K};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {k_major ? (cuuint32_t)BK : 64u,
                       k_major ? (cuuint32_t)box_rows : (cuuint32_t)BK};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

const TcVariant* variant_for(int bn) {
  const TcVariant* tabs[3] = {kVariantsBN256, kVariantsBN128, kVariantsBN64};
  const int counts[3] = {kNumVariantsBN256, kNumVariantsBN128, kNumVariantsBN64};
  for (int t = 0; t < 3; ++t)
    for (int i = 0; i < counts[t]; ++i)
      if (tabs[t][i].bn == bn && !tabs[t][i].i8x && tabs[t][i].pw == 0) return &tabs[t][i];
  return nullptr;
}

bool half_type(int t) { return t == T_F16 || t == T_BF16; }
int esize(int t) { return t == T_F32 || t == T_I32 ? 4 : (t == T_I8 ? 1 : 2); }
int64_t packed(int layout, int64_t rows, int64_t cols) {
  return layout == GEMM_ROW_MAJOR ? cols : rows;
}

}  // namespace

extern "C" GEMM_API int gemm_run_splitk_noalloc(const gemm_desc_t* desc, int splits,
                                                const void* A, const void* B, const void* C,
                                                void* D, gemm_stream_t stream) {
  if (!desc || !A || !B || !D || splits < 1 || splits > kMaxSplits) return GEMM_ERR_INVALID_ARG;
  gemm_desc_t d = *desc;
  if (d.M <= 0 || d.N <= 0 || d.K <= 0) return GEMM_ERR_INVALID_ARG;
  if (d.M > INT32_MAX / 2 || d.N > INT32_MAX / 2 || d.K > INT32_MAX / 2) return GEMM_ERR_INVALID_ARG;
  for (int l : {d.layout_a, d.layout_b, d.layout_c, d.layout_d})
    if (l != GEMM_ROW_MAJOR && l != GEMM_COL_MAJOR) return GEMM_ERR_INVALID_ARG;
  if (!half_type(d.ab_type)) return GEMM_ERR_UNSUPPORTED;
  if (!(half_type(d.d_type) || static_cast<int>(d.d_type) == T_F32)) return GEMM_ERR_UNSUPPORTED;
  if (C && !(half_type(d.c_type) || static_cast<int>(d.c_type) == T_F32))
    return GEMM_ERR_UNSUPPORTED;
  if (d.lda == 0) d.lda = packed(d.layout_a, d.M, d.K);
  if (d.ldb == 0) d.ldb = packed(d.layout_b, d.K, d.N);
  if (d.ldc == 0) d.ldc = packed(d.layout_c, d.M, d.N);
  if (d.ldd == 0) d.ldd = packed(d.layout_d, d.M, d.N);
  if (d.lda < packed(d.layout_a, d.M, d.K) || d.ldb < packed(d.layout_b, d.K, d.N) ||
      d.ldd < packed(d.layout_d, d.M, d.N) || (C && d.ldc < packed(d.layout_c, d.M, d.N)))
    return GEMM_ERR_INVALID_ARG;
  // A and B are read in place by the TMA unit: 16-byte aligned rows only.
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(A, 16) || mis(B, 16) || (d.lda * 2) % 16 != 0 || (d.ldb * 2) % 16 != 0)
    return GEMM_ERR_MISALIGNED;
  if (mis(D, esize(d.d_type)) || (C && mis(C, esize(d.c_type)))) return GEMM_ERR_MISALIGNED;

  const int bn = d.N <= 64 ? 64 : (d.N <= 128 ? 128 : 256);
  KParams kp{};
  kp.M = (int)d.M;
  kp.N = (int)d.N;
  kp.K = (int)d.K;
  kp.tiles_m = (int)((d.M + BM - 1) / BM);
  kp.tiles_n = (int)((d.N + bn - 1) / bn);
  kp.group_m = kp.tiles_m < 8 ? kp.tiles_m : 8;
  kp.num_kb = (int)((d.K + BK - 1) / BK);
  const int s_req = splits < kp.num_kb ? splits : kp.num_kb;
  kp.kb_per_split = (kp.num_kb + s_req - 1) / s_req;
  kp.splits = (kp.num_kb + kp.kb_per_split - 1) / kp.kb_per_split;
  kp.kb_per_chunk = kp.num_kb;
  kp.kgroup = 1;
  kp.a_mn = d.layout_a == GEMM_COL_MAJOR ? 1 : 0;
  kp.b_mn = d.layout_b == GEMM_ROW_MAJOR ? 1 : 0;
  const uint32_t bf16 = static_cast<int>(d.ab_type) == T_BF16 ? 1u : 0u;
  kp.idesc = idesc_f16(bf16, (uint32_t)kp.a_mn, (uint32_t)kp.b_mn, BM, (uint32_t)bn);
  const bool row_d = d.layout_d == GEMM_ROW_MAJOR;
  // Reject problems whose partial sums do not fit in the scratch array.
  const uint64_t need = (uint64_t)kp.splits * (uint64_t)d.M * (uint64_t)d.N * 4u;
  if (kp.splits > 1 && need > GEMM_NOALLOC_SCRATCH_BYTES - kPartialOffset)
    return GEMM_ERR_INVALID_ARG;

  int dev = -1, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
  char* scratch = static_cast<char*>(scratch_address(dev));
  if (!scratch) return GEMM_ERR_CUDA;
  const TcVariant* v = variant_for(bn);
  if (!v || v->prepare() != cudaSuccess) return GEMM_ERR_CUDA;

  kp.C = C;
  kp.c_type = d.c_type;
  kp.c_rs = d.layout_c == GEMM_ROW_MAJOR ? d.ldc : 1;
  kp.c_cs = d.layout_c == GEMM_ROW_MAJOR ? 1 : d.ldc;
  kp.D = D;
  kp.d_type = d.d_type;
  kp.d_rs = row_d ? d.ldd : 1;
  kp.d_cs = row_d ? 1 : d.ldd;
  kp.c_vec = (C && kp.c_cs == 1 && !mis(C, 16) && (kp.c_rs * esize(d.c_type)) % 16 == 0) ? 1 : 0;
  kp.d_vec = (kp.d_cs == 1 && !mis(D, 16) && (kp.d_rs * esize(d.d_type)) % 16 == 0) ? 1 : 0;
  kp.ws = reinterpret_cast<float*>(scratch + kPartialOffset);
  kp.ws_rs = row_d ? d.N : 1;
  kp.ws_cs = row_d ? 1 : d.M;
  kp.ws_split = d.M * d.N;
  kp.status = reinterpret_cast<uint32_t*>(scratch);
  kp.timeout_ns = 2000000000ull;
  kp.debug_flags = 0;

  CUtensorMap tma, tmb;
  if (!encode(&tma, A, d.lda, kp.a_mn == 0, d.M, d.K, BM) ||
      !encode(&tmb, B, d.ldb, kp.b_mn == 0, d.N, d.K, bn))
    return GEMM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(kp.status, 0, sizeof(uint32_t), st) != cudaSuccess) return GEMM_ERR_CUDA;
  int64_t units = (int64_t)kp.tiles_m * kp.tiles_n * kp.splits;
  const int grid = (int)(units < sms ? units : sms);
  if (v->launch(tma, tmb, kp, grid, st) != cudaSuccess) return GEMM_ERR_CUDA;
  if (kp.splits > 1 && launch_reduce(kp, row_d ? 1 : 0, sms, st) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

// The status word lives at the start of the same static array; reading it
// back allocates nothing (a 4-byte copy into the caller's stack).
extern "C" GEMM_API int gemm_noalloc_status(gemm_stream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_NO_DEVICE;
  const uint32_t* word = static_cast<const uint32_t*>(scratch_address(dev));
  if (!word) return GEMM_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GEMM_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  return (v & STATUS_TIMEOUT) ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}
