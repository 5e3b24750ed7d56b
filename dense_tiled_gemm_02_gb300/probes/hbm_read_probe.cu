// hbm_read_probe.cu -- HBM read ceilings of the access patterns the GEMM
// kernels use, without any arithmetic: how fast 8192 x 4096 bf16 (67 MB) can
// be streamed into shared memory by plain 16-byte loads and by TMA boxes of
// several shapes, and how fast 4096 rows of 8 KB (33.5 MB) move by 1-D bulk
// copies (the decode kernel's form).  Not part of the library.
// Four copies of each buffer rotate, so that consecutive launches miss L2;
// each figure is the mean of 40 back-to-back launches (CUDA events).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//       -o hbm_read_probe dense_tiled_gemm_02_gb300/probes/hbm_read_probe.cu && ./hbm_read_probe
//
// Every wait is bounded (200 ms); every TMA box lies inside its tensor.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "../csrc/ptx.cuh"
using namespace gb300;

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e)); exit(1);} } while (0)

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeFn enc() {
  static EncodeFn f = nullptr;
  if (!f) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
    f = (EncodeFn)p;
  }
  return f;
}

constexpr int ROWS = 8192, COLS = 4096;  // bf16 elements
constexpr uint64_t TMO = 200000000ull;   // 200 ms bound on every wait

struct TP {
  int rows_per_cta;   // row block height (box rows), rows = cta * rows_per_cta
  int share;          // CTAs reading the same row block (1 or 2)
  int box_inner;      // elements per box row (64 with swizzle, up to 256 without)
  int boxes_per_stage;  // consecutive K boxes per stage
  int stages;
  uint32_t* status;
};

__global__ void __launch_bounds__(64, 1) tma_read(const __grid_constant__ CUtensorMap tm, TP p) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t box_bytes = p.rows_per_cta * p.box_inner * 2;
  const uint32_t stage_bytes = box_bytes * p.boxes_per_stage;
  uint64_t* bars = (uint64_t*)(sm + p.stages * stage_bytes);
  __shared__ int abort_flag;
  const uint32_t b0 = smem_u32(bars);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) { mbar_init(b0 + 8 * s, 1); mbar_init(b0 + 8 * (p.stages + s), 1); }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int block = blockIdx.x / p.share;
  const int row0 = block * p.rows_per_cta;
  const int nk = COLS / (p.box_inner * p.boxes_per_stage);  // stages to fill
  if (threadIdx.x == 0) {
    int s = 0; uint32_t ph = 0;
    for (int i = 0; i < nk; ++i) {
      if (!bounded_wait(b0 + 8 * (p.stages + s), ph ^ 1u, &abort_flag, p.status, 1u, TMO)) break;
      mbar_arrive_expect_tx(b0 + 8 * s, stage_bytes);
      for (int j = 0; j < p.boxes_per_stage; ++j)
        tma_load_2d(smem_u32(sm + s * stage_bytes + j * box_bytes), &tm,
                    (i * p.boxes_per_stage + j) * p.box_inner, row0, b0 + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1u; }
    }
  } else if (threadIdx.x == 32) {
    int s = 0; uint32_t ph = 0;
    for (int i = 0; i < nk; ++i) {
      if (!bounded_wait(b0 + 8 * s, ph, &abort_flag, p.status, 2u, TMO)) break;
      mbar_arrive(b0 + 8 * (p.stages + s));
      if (++s == p.stages) { s = 0; ph ^= 1u; }
    }
  }
  __syncthreads();
  // drain: the last fills of each stage must land before exit
  if (threadIdx.x == 0) {
    for (int i = (nk > p.stages ? nk - p.stages : 0); i < nk; ++i)
      drain_wait(b0 + 8 * (i % p.stages), (i / p.stages) & 1, TMO);
  }
}

// plain streaming read with 16-byte loads
__global__ void ld_read(const uint4* __restrict__ a, size_t n16, uint32_t* out) {
  uint32_t x = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v0 = __ldg(a + i), v1 = __ldg(a + i + stride), v2 = __ldg(a + i + 2 * stride), v3 = __ldg(a + i + 3 * stride);
    x ^= v0.x ^ v1.y ^ v2.z ^ v3.w;
  }
  for (; i < n16; i += stride) { uint4 v = __ldg(a + i); x ^= v.x; }
  if (x == 0x12345678u) out[0] = x;
}

struct BP { int rows; int row_bytes; int cpb; int stages_cols; uint32_t* status; };
// decode-like: block b bulk-copies rows [b*cpb, b*cpb+cpb) of 8 KB, `stages_cols` at once
__global__ void __launch_bounds__(32) bulk_read(const uint8_t* B, BP p) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) { mbar_init(b, 1); abort_flag = 0; fence_mbar_init(); }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const int r0 = blockIdx.x * p.cpb;
  const int n = min(p.cpb, p.rows - r0);
  uint32_t ph = 0;
  for (int c0 = 0; c0 < n; c0 += p.stages_cols) {
    const int m = min(p.stages_cols, n - c0);
    mbar_arrive_expect_tx(b, m * p.row_bytes);
    for (int c = 0; c < m; ++c)
      bulk_load_1d(smem_u32(sm + c * p.row_bytes), B + (size_t)(r0 + c0 + c) * p.row_bytes, p.row_bytes, b);
    if (!bounded_wait(b, ph, &abort_flag, p.status, 4u, TMO)) return;
    ph ^= 1u;
  }
}

int main(int argc, char** argv) {
  const int NBUF = 4;
  const size_t bytes = (size_t)ROWS * COLS * 2;
  std::vector<void*> buf(NBUF);
  for (auto& b : buf) { CK(cudaMalloc(&b, bytes)); CK(cudaMemset(b, 1, bytes)); }
  uint32_t* status; CK(cudaMalloc(&status, 64)); CK(cudaMemset(status, 0, 64));
  cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  const int iters = 40;
  int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));

  auto timeit = [&](auto launch) {
    for (int i = 0; i < 4; ++i) launch(i);
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(e0));
    for (int i = 0; i < iters; ++i) launch(i);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
    CK(cudaGetLastError());
    uint32_t st; CK(cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost));
    if (st) printf("  status %u (a wait timed out)\n", st);
    return ms * 1000.f / iters;  // us per launch
  };

  // plain loads: whole 67 MB and first half (33.5 MB)
  for (size_t part : {bytes, bytes / 2}) {
    for (int bpsm : {2, 4, 8}) {
      float us = timeit([&](int i) { ld_read<<<sms * bpsm, 512>>>((const uint4*)buf[i % NBUF], part / 16, status); });
      printf("ld_read %5.1f MB grid %d x512: %7.2f us  %7.1f GB/s\n", part / 1e6, sms * bpsm, us, part / us / 1e3);
    }
  }

  // TMA patterns
  struct Cfg { const char* name; int rows_per_cta, share, box_inner, bps, stages; bool swz; };
  std::vector<Cfg> cfgs = {
      {"128 rows, 2 CTAs share (128x64 tiles of N = 128)", 128, 2, 64, 1, 8, true},
      {"128 rows, 64 CTAs", 128, 1, 64, 1, 12, true},
      {"64 rows, 128 CTAs", 64, 1, 64, 1, 16, true},
      {"64 rows, 128 CTAs, 2 boxes/stage (256 B)", 64, 1, 64, 2, 8, true},
      {"64 rows, 128 CTAs, 4 boxes/stage (512 B)", 64, 1, 64, 4, 4, true},
      {"32 rows, 256 CTAs", 32, 1, 64, 1, 16, true},
      {"64 rows, 128 CTAs, no swizzle 256-el box (512 B)", 64, 1, 256, 1, 4, false},
      {"32 rows, 256 CTAs, no swizzle 256-el box (512 B)", 32, 1, 256, 1, 8, false},
      {"128 rows, 64 CTAs, no swizzle 256-el box (512 B)", 128, 1, 256, 1, 3, false},
  };
  for (auto& c : cfgs) {
    std::vector<CUtensorMap> tms(NBUF);
    for (int b = 0; b < NBUF; ++b) {
      cuuint64_t dims[2] = {(cuuint64_t)COLS, (cuuint64_t)ROWS};
      cuuint64_t strides[1] = {(cuuint64_t)COLS * 2};
      cuuint32_t box[2] = {(cuuint32_t)c.box_inner, (cuuint32_t)c.rows_per_cta};
      cuuint32_t es[2] = {1, 1};
      CUresult r = enc()(&tms[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf[b], dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         c.swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) { printf("encode failed %d for %s\n", (int)r, c.name); exit(1); }
    }
    TP p{c.rows_per_cta, c.share, c.box_inner, c.bps, c.stages, status};
    const int grid = ROWS / c.rows_per_cta * c.share;
    const size_t smem = (size_t)c.stages * c.rows_per_cta * c.box_inner * 2 * c.bps + 16 * c.stages + 1024;
    if (smem > 227 * 1024 || COLS % (c.box_inner * c.bps) != 0) { printf("bad cfg %s\n", c.name); continue; }
    CK(cudaFuncSetAttribute(tma_read, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    float us = timeit([&](int i) { tma_read<<<grid, 64, smem>>>(tms[i % NBUF], p); });
    printf("tma %-50s grid %4d smem %6zu: %7.2f us  %7.1f GB/s (DRAM bytes %.1f MB)\n", c.name, grid, smem, us,
           bytes / us / 1e3, bytes / 1e6);
  }

  // decode-like bulk copies over the first 33.5 MB as 4096 rows of 8 KB
  for (int cpb : {27, 14, 7, 4}) {
    for (int sc : {27, 9, 3}) {
      if (sc > cpb) continue;
      BP p{4096, 8192, cpb, sc, status};
      const int grid = (4096 + cpb - 1) / cpb;
      const size_t smem = (size_t)sc * 8192;
      CK(cudaFuncSetAttribute(bulk_read, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
      float us = timeit([&](int i) { bulk_read<<<grid, 32, smem>>>((const uint8_t*)buf[i % NBUF], p); });
      printf("bulk 8KB rows: %2d rows/block, %2d in flight, grid %4d: %7.2f us  %7.1f GB/s\n", cpb, sc, grid, us,
             4096 * 8192 / us / 1e3);
    }
  }
  CK(cudaDeviceSynchronize());
  printf("done\n");
  return 0;
}
