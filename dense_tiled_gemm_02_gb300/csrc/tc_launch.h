// tc_launch.h -- host-side view of the compiled tcgen05 kernel variants.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.h"

namespace gb300 {

// Launch with programmatic stream serialisation allowed: the kernel may be
// scheduled while the previous kernel in the stream finishes, and waits for
// it in pdl_wait() before touching global memory (hides launch latency
// between the kernels of one GEMM call).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}


struct TcVariant {
  int bn;
  int stages;
  bool i8x;
  int pw;  // producer warps beside the TMA unit (in-kernel loads of unaligned rows)
  int cs;  // largest cluster for split-K through shared memory (1: none)
  uint32_t smem;
  cudaError_t (*launch)(const CUtensorMap&, const CUtensorMap&, const KParams&, int grid,
                        cudaStream_t);
  cudaError_t (*prepare)();  // sets the dynamic shared-memory limit on the current device
};

extern const TcVariant kVariantsBN256[];
extern const int kNumVariantsBN256;
extern const TcVariant kVariantsBN128[];
extern const int kNumVariantsBN128;
extern const TcVariant kVariantsBN64[];
extern const int kNumVariantsBN64;

// CTA-pair variants (clusters of 2, tile 256 x bn).  max_clusters() is the
// number of 2-CTA clusters that can be resident at once on the current
// device (0 on failure); call prepare() first.
struct PairVariant {
  int bn;
  int stages;
  int ksub;  // 64-wide K slices per ring stage
  bool i8x;  // exact int8 (bf16-widened operands, chunked int32 sums)
  uint32_t smem;
  // tensor maps of A, B and, when KParams::d_tma, D and (exact int8) C
  cudaError_t (*launch)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                        const CUtensorMap&, const KParams&, int grid, cudaStream_t);
  cudaError_t (*prepare)();
  int (*max_clusters)();
};

extern const PairVariant kPairVariants[];
extern const int kNumPairVariants;

cudaError_t launch_reduce(const KParams& p, int row_order, int num_sms, cudaStream_t st);
// E8M0 scales S (R rows of nsb 32-element K blocks, row-major) packed into
// 512-byte cells per (128-row tile, group of four blocks): byte 16 j + 4 c + k
// of cell (t, g) = S[128 t + 32 c + j][4 g + k], 127 (2^0) outside S.
cudaError_t launch_pack_scales(const uint8_t* S, int R, int nsb, int nsb4, int tiles,
                               uint8_t* dst, cudaStream_t st);

// Native int8 GEMM (i8_mma.cu): A and B K-contiguous (element (m, k) of A at
// A[m * lda + k], element (k, n) of B at B[n * ldb + k]; rows and bases
// 16-byte aligned), int32 C (may be null) and D with element strides; 128 x
// 128 tiles in the grouped order, one block each.  vec: C (when present)
// and D have unit column strides, even row strides and 8-byte aligned bases.
struct I8Params {
  int M, N, K;
  int tiles_m, tiles_n, group_m;
  const int8_t* A;
  long long lda;
  const int8_t* B;
  long long ldb;
  const int32_t* C;
  long long c_rs, c_cs;
  int32_t* D;
  long long d_rs, d_cs;
  int vec;
};
cudaError_t prepare_i8_mma();
cudaError_t launch_i8_mma(const I8Params& p, cudaStream_t st);
// dst[r * ld_dst + k] = src[r * rs + k * ks] (int8, r < rows, k < cols).
cudaError_t launch_to_kmajor_i8(const int8_t* src, long long rs, long long ks, long long rows,
                                long long cols, int8_t* dst, long long ld_dst, cudaStream_t st);
cudaError_t launch_repack(const void* src, int src_type, long long ld_src, uint16_t* dst,
                          long long ld_dst, long long rows, long long cols, int num_sms,
                          cudaStream_t st);
// Decode regime (decode.cu): M <= kDecodeMaxRows rows, B K-contiguous (element (k, n)
// at B[n * ldb + k]), K a multiple of 8 (16-byte loads when B is 16-byte
// aligned and ldb a multiple of 8, else 2-byte loads).  Each block writes
// the fp32 partial sums of its K slice (kc elements) to ws (slice s at
// ws + s * ws_split, element (m, n) at m * ws_rs + n * ws_cs); the last of a
// column block's `splits` blocks adds them in slice order, adds C and
// stores D.  counters: one per block of decode_columns_per_block()
// columns, zero between calls.
constexpr int kDecodeMaxRows = 4;
struct DecodeArgs {
  const uint16_t* A;
  long long a_rs, a_cs;
  const uint16_t* B;
  long long ldb;
  int M, N, K, kc, splits;
  bool bf16;
  float* ws;
  long long ws_split, ws_rs, ws_cs;
  unsigned* counters;
  const void* C;  // may be null
  int c_type;
  long long c_rs, c_cs;
  void* D;
  int d_type;
  long long d_rs, d_cs;
  // Bulk-copy form (bulk = true): blocks of cpb whole columns over all of K;
  // A's rows copied once, B's columns streamed through a ring of `stages`
  // stages of cps whole columns (from decode_bulk_ring); the bound and
  // status word of its waits, test hooks.
  bool bulk = false;
  int cpb = 0, stages = 0, cps = 0;
  uint32_t* status = nullptr;
  unsigned long long timeout_ns = 0;
  int debug_flags = 0;
  // Tensor-core form (decode_mma.cu, mma = true): M <= kDecodeMmaMaxRows,
  // B K-contiguous (b_kcontig, K a multiple of 8) or N-contiguous (element
  // (k, n) at B[k * ldb + n]); blocks of decode_mma_cols(b_kcontig) columns
  // and K slices of kc (a multiple of decode_mma_kstep(b_kcontig)); the
  // same partials, counters and finish as the split-K form.
  bool mma = false;
  bool b_kcontig = true;
};
cudaError_t launch_decode(const DecodeArgs& d, cudaStream_t st);
constexpr int kDecodeMmaMaxRows = 16;
cudaError_t launch_decode_mma(const DecodeArgs& d, cudaStream_t st);
int decode_mma_cols(bool b_kcontig);
int decode_mma_kstep(bool b_kcontig);
size_t decode_mma_smem(int M, int kc, bool b_kcontig);
// Ring of the bulk-copy form for M rows of K elements and cpb columns per
// block, in the shared memory it may use beside A: when all cpb columns fit,
// a slot for each (stages * *cps >= cpb, one round trip, no stage reused);
// otherwise stages of *cps = 8 columns.  Returns the stage count (the form
// needs every column to fit, or at least two stages).
int decode_bulk_ring(int M, long long K, int cpb, int* cps);
// Dynamic shared memory of one block of the bulk-copy form.
long long decode_bulk_smem(int M, long long K, int stages, int cps);
int decode_columns_per_block();
// Resident blocks of the decode kernel per SM for M rows and slices of kc.
int decode_blocks_per_sm(int M, int kc);

// Copies of 16-bit rows between buffers of any 2-byte alignment (rows x
// cols elements, row strides in elements); up to kMaxCopyJobs in one
// launch.  Jobs with no elements are skipped.
constexpr int kMaxCopyJobs = 3;
struct CopyJob16 {
  const uint16_t* src;
  long long ld_src;
  uint16_t* dst;
  long long ld_dst;
  long long rows, cols;
};
struct CopyJobs16 {
  CopyJob16 job[kMaxCopyJobs];
};
cudaError_t launch_copy16(const CopyJob16* jobs, int n, int num_sms, cudaStream_t st);

// 16-bit rows from a 16-byte aligned workspace (ld_src a multiple of 8
// elements) to a destination of any 2-byte alignment.
cudaError_t launch_copy_out16(const uint16_t* src, long long ld_src, uint16_t* dst,
                              long long ld_dst, long long rows, long long cols, int num_sms,
                              cudaStream_t st);

}  // namespace gb300
