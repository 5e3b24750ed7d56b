// aux_kernels.cu -- the bandwidth-bound helpers around the tensor-core kernel.
//
//  * splitk_reduce_kernel: sums the fp32 partial tiles of a split-K run in a
//    fixed order (split 0, 1, ...), adds C in fp32 and stores D with one
//    conversion.  With zero splits it computes D = C (the K = 0 case).
//  * copy_rows16_kernel: copies 16-bit rows between buffers of any 2-byte
//    alignment: operands whose rows the TMA unit cannot read in place into a
//    padded workspace, and C / D rows that are not 16-byte aligned into and
//    out of aligned workspace rows.
//  * widen_i8_x16_kernel / widen_i8_x4_kernel / repack_kernel: int8
//    operands widened to bf16 in the workspace (exact: |v| <= 128 needs 8
//    bits), sixteen or four elements a thread when rows allow it, else one.
//
// All of them put consecutive threads on consecutive addresses and are
// launched with programmatic stream serialisation (pdl_wait first).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.h"
#include "ptx.cuh"
#include "tc_launch.h"

namespace gb300 {

__device__ __forceinline__ float ld_f(const void* base, int t, long long off) {
  if (t == T_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[off]);
  if (t == T_F16) return __half2float(static_cast<const __half*>(base)[off]);
  return static_cast<const float*>(base)[off];
}

__device__ __forceinline__ void st_f(void* base, int t, long long off, float v) {
  if (t == T_BF16)
    static_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(v);
  else if (t == T_F16)
    static_cast<__half*>(base)[off] = __float2half_rn(v);
  else
    static_cast<float*>(base)[off] = v;
}

// row_order = 1: element index walks D row by row (D rows contiguous),
// otherwise column by column.
__global__ void splitk_reduce_kernel(const KParams p, int row_order) {
  pdl_wait();
  pdl_trigger();
  // D walked along its contiguous dimension: `inner` is N for row-major D
  // and M otherwise.  Thread t of block x takes inner indices
  // base + k * 256 + t (k < EPT) of the outer lines strided over block y, so
  // every warp access covers consecutive addresses and all loads of a split
  // are in flight together.  Two elements a thread: a D of a few long lines
  // (M = 1 .. 64) still spreads over many blocks.
  constexpr int EPT = 2;
  const long long outer = row_order ? p.M : p.N;
  const long long inner = row_order ? p.N : p.M;
  const long long base = static_cast<long long>(blockIdx.x) * blockDim.x * EPT + threadIdx.x;
  if (base >= inner) return;
  for (long long o = blockIdx.y; o < outer; o += gridDim.y) {
    auto rc = [&](int k, long long& r, long long& c) {
      const long long i = base + static_cast<long long>(k) * blockDim.x;
      r = row_order ? o : i;
      c = row_order ? i : o;
    };
    if (p.d_type == T_I32) {  // K = 0 with int32 C: D = C
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        long long r, c;
        rc(k, r, c);
        if ((row_order ? c : r) >= inner) continue;
        static_cast<int*>(p.D)[r * p.d_rs + c * p.d_cs] =
            p.C ? static_cast<const int*>(p.C)[r * p.c_rs + c * p.c_cs] : 0;
      }
      continue;
    }
    // C and up to four splits' partials are all requested before the first
    // add (the sum itself still runs split 0, 1, ... in order).
    float cv[EPT], acc[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      long long r, c;
      rc(k, r, c);
      cv[k] = (p.C && (row_order ? c : r) < inner) ? ld_f(p.C, p.c_type, r * p.c_rs + c * p.c_cs)
                                                   : 0.f;
      acc[k] = 0.f;
    }
    for (int s0 = 0; s0 < p.splits; s0 += 4) {
      float v[4][EPT];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
          long long r, c;
          rc(k, r, c);
          v[q][k] = (s0 + q < p.splits && (row_order ? c : r) < inner)
                        ? p.ws[(s0 + q) * p.ws_split + r * p.ws_rs + c * p.ws_cs]
                        : 0.f;
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (s0 + q < p.splits)  // (no +0.0 for absent splits: it would turn -0.0 into +0.0)
#pragma unroll
          for (int k = 0; k < EPT; ++k) acc[k] += v[q][k];
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      long long r, c;
      rc(k, r, c);
      if ((row_order ? c : r) >= inner) continue;
      st_f(p.D, p.d_type, r * p.d_rs + c * p.d_cs, p.C ? acc[k] + cv[k] : acc[k]);
    }
  }
}

// Copy rows x cols elements (storage order) from src (leading dimension
// ld_src) to the 16-bit dst (leading dimension ld_dst).  src_type T_I8
// widens to bf16 (exact); 16-bit types are copied bit for bit.  Block x
// covers 256 consecutive columns of one row band; rows are strided over
// block y, so neighbouring threads touch neighbouring addresses and no
// thread divides.
__global__ void repack_kernel(const void* __restrict__ src, int src_type, long long ld_src,
                              uint16_t* __restrict__ dst, long long ld_dst, long long rows,
                              long long cols) {
  pdl_wait();
  pdl_trigger();
  const long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  // Four rows per step: their loads are independent, so four are in flight.
  constexpr int R = 4;
  const long long step = static_cast<long long>(gridDim.y) * R;
  for (long long r0 = static_cast<long long>(blockIdx.y) * R; r0 < rows; r0 += step) {
    uint16_t v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = r0 + i;
      if (r >= rows) break;
      if (src_type == T_I8) {
        const __nv_bfloat16 b = __float2bfloat16_rn(
            static_cast<float>(static_cast<const int8_t*>(src)[r * ld_src + c]));
        v[i] = *reinterpret_cast<const uint16_t*>(&b);
      } else {
        v[i] = static_cast<const uint16_t*>(src)[r * ld_src + c];
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (r0 + i >= rows) break;
      dst[(r0 + i) * ld_dst + c] = v[i];
    }
  }
}

// 16-bit rows copied between buffers of any 2-byte alignment (into or out
// of the aligned workspace).  Consecutive lanes take consecutive elements,
// so every warp access covers 64 contiguous bytes on both sides (2 bytes per
// lane at a wider stride would touch a sector per lane).  Block x covers
// 256 * 8 columns of a row band, element k of thread t at column
// base + k * 256 + t; rows are strided over block y.  (Sixteen elements a
// thread, with half the blocks, measured slower.)
constexpr int kCopyEpt = 8;  // elements of a row per thread

// Up to kMaxCopyJobs copies in one launch, job blockIdx.z: the operand
// copies and the C staging of a call overlap instead of each waiting for
// the tail of the one before.
__global__ void copy_rows16_kernel(const CopyJobs16 jobs) {
  pdl_wait();
  pdl_trigger();
  const CopyJob16 j = jobs.job[blockIdx.z];
  constexpr int EPT = kCopyEpt;
  const long long base = static_cast<long long>(blockIdx.x) * blockDim.x * EPT + threadIdx.x;
  if (base >= j.cols) return;
  for (long long r = blockIdx.y; r < j.rows; r += gridDim.y) {
    uint16_t v[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const long long c = base + static_cast<long long>(k) * blockDim.x;
      if (c < j.cols) v[k] = j.src[r * j.ld_src + c];
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const long long c = base + static_cast<long long>(k) * blockDim.x;
      if (c < j.cols) j.dst[r * j.ld_dst + c] = v[k];
    }
  }
}

// 8-bit rows (8-bit float operands) copied into the aligned workspace, the
// 16-bit kernel's pattern with bytes.
__global__ void copy_rows8_kernel(const uint8_t* __restrict__ src, long long ld_src,
                                  uint8_t* __restrict__ dst, long long ld_dst, long long rows,
                                  long long cols) {
  pdl_wait();
  pdl_trigger();
  constexpr int EPT = 2 * kCopyEpt;
  const long long base = static_cast<long long>(blockIdx.x) * blockDim.x * EPT + threadIdx.x;
  if (base >= cols) return;
  for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
    uint8_t v[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const long long c = base + static_cast<long long>(k) * blockDim.x;
      if (c < cols) v[k] = src[r * ld_src + c];
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const long long c = base + static_cast<long long>(k) * blockDim.x;
      if (c < cols) dst[r * ld_dst + c] = v[k];
    }
  }
}

// int8 -> bf16 widening, 4 elements per thread (rows whose starts and
// lengths are multiples of 4 elements), four rows per step.
__global__ void widen_i8_x4_kernel(const char4* __restrict__ src, long long ld_src4,
                                   uint2* __restrict__ dst, long long ld_dst4, long long rows,
                                   long long cols4) {
  pdl_wait();
  pdl_trigger();
  const long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols4) return;
  constexpr int R = 4;
  const long long step = static_cast<long long>(gridDim.y) * R;
  for (long long r0 = static_cast<long long>(blockIdx.y) * R; r0 < rows; r0 += step) {
    char4 x[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (r0 + i < rows) x[i] = src[(r0 + i) * ld_src4 + c];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (r0 + i >= rows) break;
      const __nv_bfloat162 lo =
          __floats2bfloat162_rn(static_cast<float>(x[i].x), static_cast<float>(x[i].y));
      const __nv_bfloat162 hi =
          __floats2bfloat162_rn(static_cast<float>(x[i].z), static_cast<float>(x[i].w));
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&lo);
      o.y = *reinterpret_cast<const uint32_t*>(&hi);
      dst[(r0 + i) * ld_dst4 + c] = o;
    }
  }
}

// int8 -> bf16 widening, 16 elements per thread (rows whose starts and
// lengths are multiples of 16 elements): one 16-byte load and two 16-byte
// stores per row, so a warp moves 512 contiguous bytes in and 1 KB out per
// access; two rows per step.
__global__ void widen_i8_x16_kernel(const uint4* __restrict__ src, long long ld_src16,
                                    uint4* __restrict__ dst, long long ld_dst8, long long rows,
                                    long long cols16) {
  pdl_wait();
  pdl_trigger();
  const long long c = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols16) return;
  constexpr int R = 2;
  const long long step = static_cast<long long>(gridDim.y) * R;
  for (long long r0 = static_cast<long long>(blockIdx.y) * R; r0 < rows; r0 += step) {
    uint4 x[R];
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (r0 + i < rows) x[i] = src[(r0 + i) * ld_src16 + c];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (r0 + i >= rows) break;
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // bytes of w[k], low to high: elements 4k .. 4k + 3 (signed)
        const float e0 = static_cast<float>(static_cast<int8_t>(w[k] & 0xFFu));
        const float e1 = static_cast<float>(static_cast<int8_t>((w[k] >> 8) & 0xFFu));
        const float e2 = static_cast<float>(static_cast<int8_t>((w[k] >> 16) & 0xFFu));
        const float e3 = static_cast<float>(static_cast<int8_t>(w[k] >> 24));
        const __nv_bfloat162 lo = __floats2bfloat162_rn(e0, e1);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(e2, e3);
        o[2 * k] = *reinterpret_cast<const uint32_t*>(&lo);
        o[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
      uint4* const d = dst + (r0 + i) * ld_dst8 + 2 * c;
      d[0] = make_uint4(o[0], o[1], o[2], o[3]);
      d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

namespace {
// copy_rows16_kernel: 2048 columns per block, rows strided over block y.
dim3 copy_rows_grid(long long rows, long long cols, int num_sms, int njobs) {
  const unsigned gx = static_cast<unsigned>((cols + 256 * kCopyEpt - 1) / (256 * kCopyEpt));
  long long gy = (static_cast<long long>(num_sms) * 16 + gx - 1) / gx;
  if (gy > rows) gy = rows;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  return dim3(gx, static_cast<unsigned>(gy), static_cast<unsigned>(njobs));
}

dim3 copy_grid(long long chunks, long long rows, int num_sms) {
  const unsigned gx = static_cast<unsigned>((chunks + 255) / 256);
  long long gy = (static_cast<long long>(num_sms) * 16 + gx - 1) / gx;
  const long long row_steps = (rows + 3) / 4;  // the copy kernels take four rows a step
  if (gy > row_steps) gy = row_steps;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  return dim3(gx, static_cast<unsigned>(gy));
}
}  // namespace

cudaError_t launch_reduce(const KParams& p, int row_order, int num_sms, cudaStream_t st) {
  if (static_cast<long long>(p.M) * p.N == 0) return cudaSuccess;
  const long long outer = row_order ? p.M : p.N;
  const long long inner = row_order ? p.N : p.M;
  const unsigned gx = static_cast<unsigned>((inner + 511) / 512);  // 256 threads x 2 elements
  long long gy = (static_cast<long long>(num_sms) * 16 + gx - 1) / gx;
  if (gy > outer) gy = outer;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  return launch_pdl(splitk_reduce_kernel, dim3(gx, static_cast<unsigned>(gy)), dim3(256), 0, st,
                    p, row_order);
}


cudaError_t launch_repack(const void* src, int src_type, long long ld_src, uint16_t* dst,
                          long long ld_dst, long long rows, long long cols, int num_sms,
                          cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const bool x16 = src_type == T_I8 && cols % 16 == 0 && ld_src % 16 == 0 && ld_dst % 8 == 0 &&
                   reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 16 == 0;
  if (x16)
    return launch_pdl(widen_i8_x16_kernel, copy_grid(cols / 16, rows, num_sms), dim3(256), 0, st,
                      static_cast<const uint4*>(src), ld_src / 16, reinterpret_cast<uint4*>(dst),
                      ld_dst / 8, rows, cols / 16);
  const bool x4 = src_type == T_I8 && cols % 4 == 0 && ld_src % 4 == 0 && ld_dst % 4 == 0 &&
                  reinterpret_cast<uintptr_t>(src) % 4 == 0;
  if (x4)
    return launch_pdl(widen_i8_x4_kernel, copy_grid(cols / 4, rows, num_sms), dim3(256), 0, st,
                      static_cast<const char4*>(src), ld_src / 4, reinterpret_cast<uint2*>(dst),
                      ld_dst / 4, rows, cols / 4);
  if (src_type == T_E4M3 || src_type == T_E5M2 || src_type == T_MXE4M3 ||
      src_type == T_MXE5M2) {  // bytes into a byte workspace
    const dim3 g = copy_rows_grid(rows, (cols + 1) / 2, num_sms, 1);
    return launch_pdl(copy_rows8_kernel, g, dim3(256), 0, st, static_cast<const uint8_t*>(src),
                      ld_src, reinterpret_cast<uint8_t*>(dst), ld_dst, rows, cols);
  }
  if (src_type != T_I8) {
    const CopyJob16 j{static_cast<const uint16_t*>(src), ld_src, dst, ld_dst, rows, cols};
    return launch_copy16(&j, 1, num_sms, st);
  }
  return launch_pdl(repack_kernel, copy_grid(cols, rows, num_sms), dim3(256), 0, st, src,
                    src_type, ld_src, dst, ld_dst, rows, cols);
}

// One 32-bit word (four exponents of one row: K blocks 4 g .. 4 g + 3) per
// thread; consecutive threads write consecutive words of a cell.
__global__ void pack_scales_kernel(const uint8_t* __restrict__ S, int R, int nsb, int nsb4,
                                   long long words, uint32_t* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; w < words;
       w += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long cell = w >> 7;           // (tile, group): 128 words each
    const int within = static_cast<int>(w & 127);
    const long long t = cell / nsb4;
    const int g = static_cast<int>(cell - t * nsb4);
    const int j = within >> 2, c = within & 3;
    const long long row = 128 * t + 32 * c + j;
    uint32_t v = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = 4 * g + k;
      const uint32_t e = (row < R && b < nsb) ? S[row * nsb + b] : 127u;
      v |= e << (8 * k);
    }
    dst[w] = v;
  }
}

cudaError_t launch_pack_scales(const uint8_t* S, int R, int nsb, int nsb4, int tiles,
                               uint8_t* dst, cudaStream_t st) {
  const long long words = static_cast<long long>(tiles) * nsb4 * 128;
  const int grid = static_cast<int>(std::min<long long>((words + 255) / 256, 65535));
  return launch_pdl(pack_scales_kernel, dim3(grid), dim3(256), 0, st, S, R, nsb, nsb4, words,
                    reinterpret_cast<uint32_t*>(dst));
}

cudaError_t launch_copy16(const CopyJob16* jobs, int n, int num_sms, cudaStream_t st) {
  if (n < 1 || n > kMaxCopyJobs) return cudaErrorInvalidValue;
  CopyJobs16 js{};
  long long rows = 0, cols = 0;
  int m = 0;
  for (int i = 0; i < n; ++i) {
    if (jobs[i].rows == 0 || jobs[i].cols == 0) continue;
    js.job[m++] = jobs[i];
    rows = jobs[i].rows > rows ? jobs[i].rows : rows;
    cols = jobs[i].cols > cols ? jobs[i].cols : cols;
  }
  if (m == 0) return cudaSuccess;
  return launch_pdl(copy_rows16_kernel, copy_rows_grid(rows, cols, num_sms, m), dim3(256), 0, st,
                    js);
}

cudaError_t launch_copy_out16(const uint16_t* src, long long ld_src, uint16_t* dst,
                              long long ld_dst, long long rows, long long cols, int num_sms,
                              cudaStream_t st) {
  const CopyJob16 j{src, ld_src, dst, ld_dst, rows, cols};
  return launch_copy16(&j, 1, num_sms, st);
}

}  // namespace gb300
