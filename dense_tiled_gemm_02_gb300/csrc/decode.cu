// decode.cu -- the decode regime: D = A*B + C with M <= 4 rows and B's K
// dimension contiguous (a weight stored N x K).  Two forms: the split-K
// kernel described here, for any alignment and for few columns, and the
// bulk-copy form further down, for 16-byte aligned rows and N of at least
// four columns per SM.
//
// At M <= 4 the multiply is bound by reading B once (2*N*K bytes), not by
// arithmetic, so this kernel streams B with 16-byte loads on the CUDA cores
// instead of padding the rows up to a tensor-core tile.  (At 16 rows the
// CUDA-core arithmetic per B element is no longer small: that case was
// measured 3x slower here than on the tensor-core path, which it keeps.)  Block (x, y) takes
// 32 columns of D and the y-th slice of K:
//   * the slice of A (M rows x kc) is staged in shared memory as 16-bit
//     values (the same for every column);
//   * warp w takes columns 4w .. 4w+3 of the block; lane l reads K elements
//     8l + 256j of each column's row of B (one 512-byte segment per column
//     and step for the warp) and multiplies them with the matching A
//     elements of every row, so one A load from shared memory serves four
//     columns;
//   * each lane's fp32 sums are added across the warp by a fixed butterfly,
//     and lane 0 writes the slice's partial sums to the workspace;
//   * the block that finishes last among the K slices of its columns (a
//     per-column-block counter) adds the slices' partials in slice order,
//     adds C, converts and stores D, and resets the counter.  The sum's
//     order does not depend on which block is last: deterministic, and no
//     second kernel.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.h"
#include "ptx.cuh"
#include "tc_launch.h"

namespace gb300 {

namespace {

constexpr int DEC_THREADS = 256;
constexpr int DEC_NC = 4;                          // columns per warp
constexpr int DEC_COLS = DEC_NC * DEC_THREADS / 32;  // columns per block

__device__ __forceinline__ float dec_load(const void* base, int t, long long off) {
  if (t == T_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[off]);
  if (t == T_F16) return __half2float(static_cast<const __half*>(base)[off]);
  return static_cast<const float*>(base)[off];
}

__device__ __forceinline__ void dec_store(void* base, int t, long long off, float v) {
  if (t == T_BF16)
    static_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(v);
  else if (t == T_F16)
    static_cast<__half*>(base)[off] = __float2half_rn(v);
  else
    static_cast<float*>(base)[off] = v;
}

template <bool BF16>
__device__ __forceinline__ void widen8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 x = __half22float2(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

// MM: rows the registers are sized for (M <= MM).  kc: K elements of a
// slice, a multiple of 8; the slice of block y is [y*kc, min(K, y*kc + kc)).
// VEC: B's rows start on 16-byte boundaries (16-byte loads), else 2-byte
// loads of the same elements.
template <int MM, bool BF16, bool VEC>
__global__ void __launch_bounds__(DEC_THREADS)
    decode_kn_kernel(const DecodeArgs d) {
  const uint16_t* __restrict__ A = d.A;
  const uint16_t* __restrict__ B = d.B;
  const long long a_rs = d.a_rs, a_cs = d.a_cs, ldb = d.ldb;
  const int M = d.M, N = d.N, K = d.K, kc = d.kc;
  extern __shared__ __align__(16) uint16_t sA[];  // [MM][kc]
  pdl_wait();
  pdl_trigger();
  const int k0 = blockIdx.y * kc;
  const int kn = min(kc, K - k0);  // a multiple of 8 (K is)
  // Stage A's slice (rows M .. MM-1 are zero).
  for (int i = threadIdx.x; i < MM * kc; i += DEC_THREADS) {
    const int m = i / kc, kk = i - m * kc;
    sA[i] = (m < M && kk < kn) ? A[m * a_rs + static_cast<long long>(k0 + kk) * a_cs]
                               : uint16_t(0);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * DEC_COLS + warp * DEC_NC;
  float acc[MM][DEC_NC];
#pragma unroll
  for (int m = 0; m < MM; ++m)
#pragma unroll
    for (int c = 0; c < DEC_NC; ++c) acc[m][c] = 0.f;
  const uint16_t* brow[DEC_NC];
#pragma unroll
  for (int c = 0; c < DEC_NC; ++c)
    brow[c] = B + static_cast<long long>(min(n0 + c, N - 1)) * ldb + k0;

  // Four 256-element steps at a time, all their B loads issued before the
  // first use: one memory round trip per four steps, not per step.
  constexpr int U = 4;
  for (int kb = 8 * lane; kb < kn; kb += 256 * U) {
    uint4 raw[U][DEC_NC];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = kb + 256 * u;
#pragma unroll
      for (int c = 0; c < DEC_NC; ++c) {
        if (kk >= kn) {
          raw[u][c] = make_uint4(0u, 0u, 0u, 0u);
        } else if (VEC) {
          raw[u][c] = ld_global_v4_pinned(brow[c] + kk);
        } else {
          uint16_t e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) e[i] = brow[c][kk + i];
          raw[u][c] = make_uint4(e[0] | (uint32_t(e[1]) << 16), e[2] | (uint32_t(e[3]) << 16),
                                 e[4] | (uint32_t(e[5]) << 16), e[6] | (uint32_t(e[7]) << 16));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = kb + 256 * u;
      if (kk >= kn) break;
      float b[DEC_NC][8];
#pragma unroll
      for (int c = 0; c < DEC_NC; ++c) widen8<BF16>(raw[u][c], b[c]);
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        float a[8];
        widen8<BF16>(*reinterpret_cast<const uint4*>(sA + m * kc + kk), a);
#pragma unroll
        for (int c = 0; c < DEC_NC; ++c) {
          float s = acc[m][c];
#pragma unroll
          for (int e = 0; e < 8; ++e) s = fmaf(a[e], b[c][e], s);
          acc[m][c] = s;
        }
      }
    }
  }
  // Sum over the warp (fixed butterfly), then lane 0 writes the partials.
#pragma unroll
  for (int m = 0; m < MM; ++m)
#pragma unroll
    for (int c = 0; c < DEC_NC; ++c) {
      float v = acc[m][c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[m][c] = v;
    }
  if (lane == 0) {
    float* out = d.ws + blockIdx.y * d.ws_split;
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
      for (int c = 0; c < DEC_NC; ++c)
        if (m < M && n0 + c < N)
          out[m * d.ws_rs + static_cast<long long>(n0 + c) * d.ws_cs] = acc[m][c];
  }
  // The last block of this column block's K slices finishes the columns.
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(d.counters + blockIdx.x, 1u);
    last = old == static_cast<unsigned>(d.splits) - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int nb = blockIdx.x * DEC_COLS;
  for (int i = threadIdx.x; i < M * DEC_COLS; i += DEC_THREADS) {
    const int m = i / DEC_COLS, n = nb + (i - m * DEC_COLS);
    if (n >= N) continue;
    float v = 0.f;
    for (int sl = 0; sl < d.splits; ++sl)
      v += d.ws[sl * d.ws_split + m * d.ws_rs + static_cast<long long>(n) * d.ws_cs];
    if (d.C) v += dec_load(d.C, d.c_type, m * d.c_rs + static_cast<long long>(n) * d.c_cs);
    dec_store(d.D, d.d_type, m * d.d_rs + static_cast<long long>(n) * d.d_cs, v);
  }
  if (threadIdx.x == 0) d.counters[blockIdx.x] = 0u;  // ready for the next call
}

// ---------------------------------------------------------------- bulk-copy form
// Block b owns columns [b*cpb, min(N, b*cpb + cpb)) of D over all of K, cpb
// chosen so that the grid is whole waves of one block per SM; there is no
// split-K tail.  Warp 8, lane 0, copies A's M rows into shared memory once
// and then streams the block's columns of B (column n's K elements are
// contiguous) through a ring of stages of cps whole columns, one 1-D bulk
// copy of 2K bytes per column; warp w of 0-7 takes the block's columns w,
// w + 8, ..., adds its K products (lane l: elements 8l + 256i) with a fixed
// butterfly, adds C and stores D.  Either every column has a stage slot of
// its own (stages * cps >= cpb: all copies in flight at once, no stage
// reused) or cps = 8, so that a warp waits on every fill of every stage in
// turn and its parity waits cannot run a phase ahead.  Full and empty barriers hand the stages
// over; every wait is bounded, and on a timeout the producer still waits
// (bounded) for the copies it issued before the block exits.
constexpr int DB_CWARPS = 8;                       // consumer warps = columns per stage
constexpr int DB_THREADS = 32 * (DB_CWARPS + 1);
constexpr int DB_BAR_BYTES = 256;  // full[12], empty[12], A's barrier, abort flag at the end
constexpr int DB_MAX_STAGES = 12;
constexpr int DB_SMEM_BUDGET = 227 * 1024;

template <int MM, bool BF16>
__global__ void __launch_bounds__(DB_THREADS) decode_bulk_kernel(const DecodeArgs d) {
  extern __shared__ __align__(128) unsigned char dsm[];
  const int S = d.stages, cpb = d.cpb, cps = d.cps;
  const int M = d.M, N = d.N, K = d.K;
  const int n0 = blockIdx.x * cpb;
  const int ncols = min(cpb, N - n0);
  const int ngroups = (ncols + cps - 1) / cps;
  const uint32_t row_bytes = static_cast<uint32_t>(K) * 2u;
  const uint32_t bars = smem_u32(dsm);  // full[0, S), empty[S, 2S), A at 2 * DB_MAX_STAGES
  const uint32_t a_bar = bars + 8 * (2 * DB_MAX_STAGES);
  const uint32_t a_smem = bars + DB_BAR_BYTES;
  const uint32_t ring = a_smem + MM * row_bytes;
  const uint32_t stage_bytes = cps * row_bytes;
  volatile int* abort = reinterpret_cast<volatile int*>(dsm + DB_BAR_BYTES - 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (S + i), cps);  // one arrival per column of a full stage
    }
    mbar_init(a_bar, 1);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const bool skip_first = (d.debug_flags & DBG_SKIP_FIRST_FILL) != 0;

  if (warp == DB_CWARPS) {  // producer
    if (lane != 0) return;
    mbar_arrive_expect_tx(a_bar, static_cast<uint32_t>(M) * row_bytes);
    for (int m = 0; m < M; ++m)
      bulk_load_1d(a_smem + m * row_bytes, d.A + static_cast<long long>(m) * d.a_rs, row_bytes,
                   a_bar);
    int issued = 0;
    for (int j = 0; j < ngroups; ++j) {
      const int s = j % S;
      const uint32_t full = bars + 8 * s;
      if (j >= S && !bounded_wait(bars + 8 * (S + s), (j / S - 1) & 1, abort, d.status,
                                  STATUS_TIMEOUT, d.timeout_ns))
        break;
      issued = j + 1;
      if (j == 0 && skip_first) continue;  // test hook: a stage never filled
      const int ng = min(cps, ncols - j * cps);
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(ng) * row_bytes);
      const uint32_t st = ring + s * stage_bytes;
      for (int c = 0; c < ng; ++c)
        bulk_load_1d(st + c * row_bytes, d.B + static_cast<long long>(n0 + j * cps + c) * d.ldb,
                     row_bytes, full);
    }
    // The block's shared memory must outlive every copy issued into it: wait
    // for A and for the last fill of each stage (no later phase was armed).
    drain_wait(a_bar, 0, d.timeout_ns);
    for (int j = max(0, issued - S); j < issued; ++j)
      if (!(j == 0 && skip_first)) drain_wait(bars + 8 * (j % S), (j / S) & 1, d.timeout_ns);
    return;
  }

  // consumers: warp w takes the block's columns w, w + 8, ...; a column's
  // stage is freed once each of its cps columns has been read.
  if (!bounded_wait(a_bar, 0, abort, d.status, STATUS_TIMEOUT, d.timeout_ns)) return;
  const uint16_t* sA = reinterpret_cast<const uint16_t*>(dsm + DB_BAR_BYTES);
  for (int col = warp; col < ncols; col += DB_CWARPS) {
    const int j = col / cps, s = j % S;
    if (!bounded_wait(bars + 8 * s, (j / S) & 1, abort, d.status, STATUS_TIMEOUT, d.timeout_ns))
      return;
    const uint16_t* sB = reinterpret_cast<const uint16_t*>(
        dsm + DB_BAR_BYTES + MM * static_cast<size_t>(row_bytes) +
        static_cast<size_t>(s) * stage_bytes + static_cast<size_t>(col - j * cps) * row_bytes);
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.f;
    for (int kk = 8 * lane; kk < K; kk += 256) {
      float b[8];
      widen8<BF16>(*reinterpret_cast<const uint4*>(sB + kk), b);
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        if (m < M) {
          float a[8];
          widen8<BF16>(*reinterpret_cast<const uint4*>(sA + m * K + kk), a);
          float v = acc[m];
#pragma unroll
          for (int e = 0; e < 8; ++e) v = fmaf(a[e], b[e], v);
          acc[m] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));  // the column has been read
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
    if (lane == 0) {
      const long long n = n0 + col;
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        if (m >= M) continue;
        float v = acc[m];
        if (d.C) v += dec_load(d.C, d.c_type, m * d.c_rs + n * d.c_cs);
        dec_store(d.D, d.d_type, m * d.d_rs + n * d.d_cs, v);
      }
    }
  }
}

template <int MM, bool BF16>
cudaError_t launch_bulk_mm(const DecodeArgs& d, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(decode_bulk_smem(d.M, d.K, d.stages, d.cps));
  auto kernel = decode_bulk_kernel<MM, BF16>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return cudaGetLastError();
  const dim3 grid(static_cast<unsigned>((d.N + d.cpb - 1) / d.cpb));
  return launch_pdl(kernel, grid, dim3(DB_THREADS), smem, st, d);
}

template <bool BF16>
cudaError_t launch_bulk(const DecodeArgs& d, cudaStream_t st) {
  if (d.M <= 1) return launch_bulk_mm<1, BF16>(d, st);
  if (d.M <= 2) return launch_bulk_mm<2, BF16>(d, st);
  return launch_bulk_mm<4, BF16>(d, st);
}

template <int MM, bool BF16, bool VEC>
cudaError_t launch_mm(const DecodeArgs& d, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(MM) * d.kc * sizeof(uint16_t);
  auto kernel = decode_kn_kernel<MM, BF16, VEC>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return cudaGetLastError();
  const dim3 grid(static_cast<unsigned>((d.N + DEC_COLS - 1) / DEC_COLS),
                  static_cast<unsigned>(d.splits));
  return launch_pdl(kernel, grid, dim3(DEC_THREADS), smem, st, d);
}

template <bool BF16, bool VEC>
cudaError_t launch_type(const DecodeArgs& d, cudaStream_t st) {
  if (d.M <= 1) return launch_mm<1, BF16, VEC>(d, st);
  if (d.M <= 2) return launch_mm<2, BF16, VEC>(d, st);
  return launch_mm<4, BF16, VEC>(d, st);
}

}  // namespace

int decode_columns_per_block() { return DEC_COLS; }

int decode_blocks_per_sm(int M, int kc) {
  const size_t smem = static_cast<size_t>(M <= 1 ? 1 : M <= 2 ? 2 : 4) * kc * sizeof(uint16_t);
  int n = 0;
  const auto k = M <= 1 ? decode_kn_kernel<1, true, true>
                        : M <= 2 ? decode_kn_kernel<2, true, true> : decode_kn_kernel<4, true, true>;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, DEC_THREADS, smem) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

long long decode_bulk_smem(int M, long long K, int stages, int cps) {
  const long long mm = M <= 1 ? 1 : M <= 2 ? 2 : 4;  // A rows the kernel is sized for
  const long long row = K * static_cast<long long>(sizeof(uint16_t));
  return DB_BAR_BYTES + mm * row + static_cast<long long>(stages) * cps * row;
}

int decode_bulk_ring(int M, long long K, int cpb, int* cps) {
  const long long mm = M <= 1 ? 1 : M <= 2 ? 2 : 4;
  const long long row = K * static_cast<long long>(sizeof(uint16_t));
  const long long left = DB_SMEM_BUDGET - DB_BAR_BYTES - mm * row;
  *cps = DB_CWARPS;
  if (row <= 0 || left <= 0 || cpb < 1) return 0;
  const long long fit = left / row;  // whole columns of B beside A
  const int c = (cpb + DB_MAX_STAGES - 1) / DB_MAX_STAGES;
  const int st = (cpb + c - 1) / c;
  if (static_cast<long long>(st) * c <= fit) {  // a slot for every column: one round trip
    *cps = c;
    return st;
  }
  return static_cast<int>(std::min<long long>(DB_MAX_STAGES, fit / DB_CWARPS));
}

cudaError_t launch_decode(const DecodeArgs& d, cudaStream_t st) {
  if (d.M < 1 || d.M > kDecodeMaxRows || d.K % 8 != 0) return cudaErrorInvalidValue;
  if (d.bulk) {
    // Every bulk copy starts on a 16-byte boundary and moves a multiple of
    // 16 bytes: A and B 16-byte aligned, their row strides and kch
    // multiples of 8 elements (K is).
    const bool aligned = reinterpret_cast<uintptr_t>(d.B) % 16 == 0 && d.ldb % 8 == 0 &&
                         reinterpret_cast<uintptr_t>(d.A) % 16 == 0 &&
                         d.a_cs == 1 && (d.M == 1 || d.a_rs % 8 == 0);
    int cps = 0;
    const int stages = decode_bulk_ring(d.M, d.K, d.cpb, &cps);
    if (!aligned || d.K <= 0 || d.cpb < 1 || d.cpb > 4 * DB_CWARPS || d.stages < 1 ||
        d.stages != stages || d.cps != cps || (d.stages * d.cps < d.cpb && d.stages < 2) ||
        d.status == nullptr)
      return cudaErrorInvalidValue;
    return d.bf16 ? launch_bulk<true>(d, st) : launch_bulk<false>(d, st);
  }
  if (d.kc % 8 != 0) return cudaErrorInvalidValue;
  const bool vec = reinterpret_cast<uintptr_t>(d.B) % 16 == 0 && d.ldb % 8 == 0;
  if (d.bf16) return vec ? launch_type<true, true>(d, st) : launch_type<true, false>(d, st);
  return vec ? launch_type<false, true>(d, st) : launch_type<false, false>(d, st);
}

}  // namespace gb300
