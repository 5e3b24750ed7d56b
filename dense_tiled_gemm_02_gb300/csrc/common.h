// common.h -- structures shared by the host planner and the device kernels.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GB_HD __host__ __device__ __forceinline__
#else
#define GB_HD inline
#endif

namespace gb300 {

// Element type codes (the values of gemm_dtype_t).
enum : int { T_F16 = 1, T_BF16 = 2, T_F32 = 3, T_I8 = 4, T_I32 = 5 };

// Tile geometry of the tcgen05 kernels: one CTA owns a BM x BN output tile
// and walks K in BK-wide slices (BK 16-bit elements = one 128-byte row).
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;  // warp 0: TMA loads, warp 1: MMA issue, warps 2-5: epilogue

// Device status word bits.
constexpr uint32_t STATUS_TIMEOUT = 1u;

// Debug flags (test hooks).
constexpr int DBG_SKIP_FIRST_FILL = 1;

// Kernel parameters (passed by value).  Coordinates are those of the
// internal problem, which may be the transposed problem D^T = B^T A^T.
struct KParams {
  int M, N, K;                   // internal problem
  int tiles_m, tiles_n, group_m; // output tile grid and raster group
  int splits, kb_per_split, num_kb;
  int kb_per_chunk;              // k-blocks accumulated in one TMEM pass (exact-int8 mode)
  int a_mn, b_mn;                // operand majors: 0 = K-major, 1 = MN-major
  uint32_t idesc;                // tcgen05 instruction descriptor
  // epilogue (internal coordinates: row r < M, column c < N)
  const void* C;
  int c_type;
  long long c_rs, c_cs;          // element strides of C
  void* D;
  int d_type;
  long long d_rs, d_cs;
  int d_vec;                     // D rows contiguous and 16-byte aligned
  int d_tma;                     // 16-bit D stored through shared memory by TMA (pair kernel)
  int c_vec;                     // C rows contiguous and 16-byte aligned
  float* ws;                     // split-K partial sums (fp32), or null
  long long ws_rs, ws_cs, ws_split;
  uint32_t* status;              // device status word
  unsigned long long timeout_ns; // bound of every device-side wait
  int debug_flags;
  // Last-wave split (pair kernel): tiles from tail_start on (in raster
  // order) are each computed as two K halves by two clusters; the second
  // half leaves its fp32 partial in tail_ws and raises tail_flags to
  // epoch, the first half adds it and finishes the tile.
  int tail_start;                // first split tile (= number of whole tiles)
  int tail_parts;                // 1 = no split, 2 = split in two K halves
  float* tail_ws;                // [split tile][CTA half][128 rows][BN] fp32
  uint32_t* tail_flags;          // [split tile][CTA half]
  uint32_t epoch;                // value the flags take during this run
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator
// (bits 4-5 = 1), A/B element type (bits 7-9, 10-12: 0 fp16, 1 bf16),
// operand majors (bit 15 A, bit 16 B: 0 K-major, 1 MN-major), N/8 in bits
// 17-22 and M/16 in bits 24-28.
GB_HD constexpr uint32_t idesc_f16(uint32_t bf16, uint32_t a_mn, uint32_t b_mn,
                                                 uint32_t m, uint32_t n) {
  return (1u << 4) | (bf16 << 7) | (bf16 << 10) | (a_mn << 15) | (b_mn << 16) |
         ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Grouped tile order (FlagGems "Hygon optimization", "Grouped scheduling"):
// tiles are numbered so that GROUP_M consecutive tile rows walk the tile
// columns together; the last group holds the tile rows that remain.
GB_HD void raster_tile(int64_t t, int64_t num_pid_m, int64_t num_pid_n, int64_t group_m,
                       int64_t& pid_m, int64_t& pid_n) {
  const int64_t in_group = group_m * num_pid_n;
  const int64_t group_id = t / in_group;
  const int64_t first_m = group_id * group_m;
  const int64_t rem = num_pid_m - first_m;
  const int64_t size_m = rem < group_m ? rem : group_m;
  pid_m = first_m + (t % in_group) % size_m;
  pid_n = (t % in_group) / size_m;
}

}  // namespace gb300
