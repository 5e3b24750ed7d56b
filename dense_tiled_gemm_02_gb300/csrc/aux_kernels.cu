// aux_kernels.cu -- the bandwidth-bound helpers around the tensor-core kernel.
//
//  * splitk_reduce_kernel: sums the fp32 partial tiles of a split-K run in a
//    fixed order (split 0, 1, ...), adds C in fp32 and stores D with one
//    conversion.  With zero splits it computes D = C (the K = 0 case).
//  * repack_kernel: copies an operand whose rows are not 16-byte aligned into
//    a padded workspace that the TMA unit can read; for int8 operands it
//    also widens every value to bf16 (exact: |v| <= 128 needs 8 bits).
//
// Both walk their arrays in storage order with consecutive threads on
// consecutive addresses, in grid-stride loops sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

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
  const long long total = static_cast<long long>(p.M) * p.N;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    long long r, c;
    if (row_order) {
      r = idx / p.N;
      c = idx - r * p.N;
    } else {
      c = idx / p.M;
      r = idx - c * p.M;
    }
    if (p.d_type == T_I32) {
      int v = 0;
      if (p.C) v = static_cast<const int*>(p.C)[r * p.c_rs + c * p.c_cs];
      static_cast<int*>(p.D)[r * p.d_rs + c * p.d_cs] = v;
      continue;
    }
    float acc = 0.f;
    for (int s = 0; s < p.splits; ++s) acc += p.ws[s * p.ws_split + r * p.ws_rs + c * p.ws_cs];
    if (p.C) acc += ld_f(p.C, p.c_type, r * p.c_rs + c * p.c_cs);
    st_f(p.D, p.d_type, r * p.d_rs + c * p.d_cs, acc);
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

// 16-bit rows copied between a side whose rows start on 16-byte boundaries
// (a workspace with its leading dimension rounded up to 8 elements) and a
// side with arbitrary 2-byte alignment.  A thread moves 8 consecutive
// elements: one 16-byte access on the aligned side, eight 2-byte accesses on
// the other (consecutive threads cover consecutive bytes, so a warp access
// still spans 512 contiguous bytes).  TO_ALIGNED: src arbitrary -> dst
// aligned; otherwise src aligned -> dst arbitrary.  Elements of the aligned
// side's last chunk beyond `cols` are written as zeros or not read.
template <bool TO_ALIGNED>
__global__ void copy16_kernel(const uint16_t* __restrict__ src, long long ld_src,
                              uint16_t* __restrict__ dst, long long ld_dst, long long rows,
                              long long cols) {
  pdl_wait();
  pdl_trigger();
  const long long c8 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c8 * 8 >= cols) return;
  const long long c0 = c8 * 8;
  const int nv = cols - c0 < 8 ? static_cast<int>(cols - c0) : 8;
  constexpr int R = 4;
  const long long step = static_cast<long long>(gridDim.y) * R;
  for (long long r0 = static_cast<long long>(blockIdx.y) * R; r0 < rows; r0 += step) {
    uint4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = r0 + i;
      if (r >= rows) break;
      if (TO_ALIGNED) {
        uint16_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = k < nv ? src[r * ld_src + c0 + k] : uint16_t(0);
        v[i].x = e[0] | (uint32_t(e[1]) << 16);
        v[i].y = e[2] | (uint32_t(e[3]) << 16);
        v[i].z = e[4] | (uint32_t(e[5]) << 16);
        v[i].w = e[6] | (uint32_t(e[7]) << 16);
      } else {
        v[i] = *reinterpret_cast<const uint4*>(src + r * ld_src + c0);
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = r0 + i;
      if (r >= rows) break;
      if (TO_ALIGNED) {
        *reinterpret_cast<uint4*>(dst + r * ld_dst + c0) = v[i];
      } else {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < nv) dst[r * ld_dst + c0 + k] = static_cast<uint16_t>(w[k / 2] >> (16 * (k & 1)));
      }
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

cudaError_t launch_reduce(const KParams& p, int row_order, int num_sms, cudaStream_t st) {
  const long long total = static_cast<long long>(p.M) * p.N;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                    p, row_order);
}

namespace {
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

cudaError_t launch_repack(const void* src, int src_type, long long ld_src, uint16_t* dst,
                          long long ld_dst, long long rows, long long cols, int num_sms,
                          cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const bool x4 = src_type == T_I8 && cols % 4 == 0 && ld_src % 4 == 0 && ld_dst % 4 == 0 &&
                  reinterpret_cast<uintptr_t>(src) % 4 == 0;
  if (x4)
    return launch_pdl(widen_i8_x4_kernel, copy_grid(cols / 4, rows, num_sms), dim3(256), 0, st,
                      static_cast<const char4*>(src), ld_src / 4, reinterpret_cast<uint2*>(dst),
                      ld_dst / 4, rows, cols / 4);
  if (src_type != T_I8 && ld_dst % 8 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0)
    return launch_pdl(copy16_kernel<true>, copy_grid((cols + 7) / 8, rows, num_sms), dim3(256), 0,
                      st, static_cast<const uint16_t*>(src), ld_src, dst, ld_dst, rows, cols);
  return launch_pdl(repack_kernel, copy_grid(cols, rows, num_sms), dim3(256), 0, st, src,
                    src_type, ld_src, dst, ld_dst, rows, cols);
}

cudaError_t launch_copy_out16(const uint16_t* src, long long ld_src, uint16_t* dst,
                              long long ld_dst, long long rows, long long cols, int num_sms,
                              cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  return launch_pdl(copy16_kernel<false>, copy_grid((cols + 7) / 8, rows, num_sms), dim3(256), 0,
                    st, src, ld_src, dst, ld_dst, rows, cols);
}

}  // namespace gb300
