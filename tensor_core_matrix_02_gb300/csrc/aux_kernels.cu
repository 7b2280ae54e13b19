// aux_kernels.cu -- bandwidth-bound helpers of the GEMM paths: the fixed-order
// split-K reduction (D = C + sum of K-slice partials) and the exact 8-bit integer
// -> bf16 widening that lets integer products run on the bf16 tensor-core path.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace mma42 {

namespace {

// D[4i .. 4i+3] = C[4i .. 4i+3] + acc for C and D of type OUT (0 f32, 1 f16, 2 bf16;
// a half result is the f32 sum rounded to nearest even).
template <int OUT>
__device__ __forceinline__ void add_c_store4(const void* __restrict__ C, void* __restrict__ D, int64_t i,
                                             float4 acc) {
  if constexpr (OUT == 0) {
    const float4 c = static_cast<const float4*>(C)[i];
    static_cast<float4*>(D)[i] = make_float4(c.x + acc.x, c.y + acc.y, c.z + acc.z, c.w + acc.w);
  } else {
    const uint2 c = static_cast<const uint2*>(C)[i];
    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
    const uint32_t cw[4] = {c.x & 0xffffu, c.x >> 16, c.y & 0xffffu, c.y >> 16};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if constexpr (OUT == 1)
        o[e] = __half_as_ushort(__float2half_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(cw[e]))) + a[e]));
      else
        o[e] = __bfloat16_as_ushort(
            __float2bfloat16_rn(__bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(cw[e]))) + a[e]));
    }
    static_cast<uint2*>(D)[i] = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
  }
}

// OUT: 0 f32, 1 f16, 2 bf16 (C and D); four outputs per step.
template <int OUT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4* __restrict__ P, int ksplit,
                                                            int64_t n4, const void* __restrict__ C,
                                                            void* __restrict__ D) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 acc = P[i];
#pragma unroll 4
    for (int s = 1; s < ksplit; ++s) {   // slices in order: the result does not depend on timing
      const float4 p = P[s * n4 + i];
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
    add_c_store4<OUT>(C, D, i, acc);
  }
}

// The tail split's reduction (see launch_tail_reduce).  Block (x, y): rows
// [4x, 4x + 4) of tail tile y, whose place in D the GEMM's raster gives once per
// block; each thread adds four consecutive outputs of one row.
// OUT 0..2 as above with f32 partials summed in slice order; 3: i32, wrapping.
template <int OUT>
__global__ void __launch_bounds__(256) tail_reduce_kernel(TailReduce r, GemmArgs g) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  const int pt = static_cast<int>(blockIdx.y);
  int mt, nt;
  tile_coords(g.tail_from + pt, g, mt, nt);
  const int c4s = r.tile_cols / 4;
  const int tr = static_cast<int>(blockIdx.x) * (blockDim.x / c4s) + static_cast<int>(threadIdx.x) / c4s;
  const int tc = (static_cast<int>(threadIdx.x) % c4s) * 4;
  if (tr >= r.tile_rows) return;
  const int64_t row = static_cast<int64_t>(mt) * r.tile_rows + tr;
  const int64_t col = static_cast<int64_t>(nt) * r.tile_cols + tc;
  if (row >= r.M || col >= r.N) return;   // N % 4 == 0: the four are all in or all out
  const int64_t slice4 = static_cast<int64_t>(r.T) * r.tile_rows * c4s;   // four-element groups per K slice
  const int64_t i = (static_cast<int64_t>(pt) * r.tile_rows + tr) * c4s + tc / 4;
  const int64_t o4 = (row * r.N + col) / 4;
  if constexpr (OUT == 3) {
    const int4* P = static_cast<const int4*>(r.P);
    const int4 c = static_cast<const int4*>(r.C)[o4];
    uint32_t acc[4] = {static_cast<uint32_t>(c.x), static_cast<uint32_t>(c.y), static_cast<uint32_t>(c.z),
                       static_cast<uint32_t>(c.w)};
    if (r.alpha != 0 || r.beta != 0) {
      const int64_t rf = static_cast<int64_t>(r.alpha) * r.beta * r.K +
                         (r.beta != 0 ? static_cast<int64_t>(r.beta) * r.rowsum[row] : 0);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc[e] += static_cast<uint32_t>(static_cast<uint64_t>(
            rf + (r.alpha != 0 ? static_cast<int64_t>(r.alpha) * r.colsum[col + e] : 0)));
    }
#pragma unroll 4
    for (int s = 0; s < r.S; ++s) {
      const int4 p = P[s * slice4 + i];
      acc[0] += static_cast<uint32_t>(p.x);
      acc[1] += static_cast<uint32_t>(p.y);
      acc[2] += static_cast<uint32_t>(p.z);
      acc[3] += static_cast<uint32_t>(p.w);
    }
    static_cast<int4*>(r.D)[o4] = make_int4(static_cast<int>(acc[0]), static_cast<int>(acc[1]),
                                            static_cast<int>(acc[2]), static_cast<int>(acc[3]));
  } else {
    const float4* P = static_cast<const float4*>(r.P);
    float4 acc = P[i];
#pragma unroll 4
    for (int s = 1; s < r.S; ++s) {   // slices in order, then C, as in splitk_reduce_kernel
      const float4 p = P[s * slice4 + i];
      acc.x += p.x;
      acc.y += p.y;
      acc.z += p.z;
      acc.w += p.w;
    }
    add_c_store4<OUT>(r.C, r.D, o4, acc);
  }
}

// D = C + sum_s P[s] for i32 partials, summed exactly in 64 bits in slice order;
// clamp: saturate to the i32 range, else wrap modulo 2^32.
// fix: the corrections of unsigned operands run as signed ones (see GemmArgs).
struct IntFix {
  const int32_t* rowsum;
  const int32_t* colsum;
  int alpha, beta;
  int64_t K, N;
};

__global__ void __launch_bounds__(256) splitk_reduce_i32_kernel(const int4* __restrict__ P, int ksplit, int64_t n4,
                                                                const int4* __restrict__ C, int4* __restrict__ D,
                                                                int clamp, IntFix fix) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int4 c = C[i];
    int64_t acc[4] = {c.x, c.y, c.z, c.w};
    if (fix.alpha != 0 || fix.beta != 0) {
      const int64_t row = (4 * i) / fix.N, col = 4 * i - row * fix.N;   // N % 4 == 0: one row per step
      const int64_t rf = static_cast<int64_t>(fix.alpha) * fix.beta * fix.K +
                         (fix.beta != 0 ? static_cast<int64_t>(fix.beta) * fix.rowsum[row] : 0);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc[e] += rf + (fix.alpha != 0 ? static_cast<int64_t>(fix.alpha) * fix.colsum[col + e] : 0);
    }
#pragma unroll 4
    for (int s = 0; s < ksplit; ++s) {
      const int4 p = P[s * n4 + i];
      acc[0] += p.x;
      acc[1] += p.y;
      acc[2] += p.z;
      acc[3] += p.w;
    }
    int32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (clamp) o[e] = static_cast<int32_t>(acc[e] > INT32_MAX ? INT32_MAX : (acc[e] < INT32_MIN ? INT32_MIN : acc[e]));
      else o[e] = static_cast<int32_t>(static_cast<uint32_t>(static_cast<uint64_t>(acc[e])));
    }
    D[i] = make_int4(o[0], o[1], o[2], o[3]);
  }
}

// Every 8-bit integer (signed -128..127 or unsigned 0..255) has at most 8
// significant bits and so is exact in bf16.  Its f32 value comes from integer
// arithmetic: for |v| < 2^22 the f32 with bits 0x4B400000 + v is 1.5 * 2^23 + v
// exactly, and subtracting 1.5 * 2^23 leaves v exactly; the bf16 pattern is then
// the top half of the f32 (its low 16 bits are zero).
// `offset` is subtracted first (128 moves an unsigned operand into the signed range).
template <bool UNSIGNED>
__device__ __forceinline__ uint32_t int8_to_f32_bits(uint32_t word, int byte, int offset) {
  const int v = (UNSIGNED ? static_cast<int>((word >> (8 * byte)) & 0xffu)
                          : static_cast<int>(static_cast<int8_t>(word >> (8 * byte)))) - offset;
  return __float_as_uint(__int_as_float(0x4B400000 + v) - 12582912.0f);
}

// Eight values: bf16 patterns of bytes 0..3 of `lo` and of `hi`, in order.
template <bool UNSIGNED>
__device__ __forceinline__ uint4 widen8(uint2 w, int offset) {
  uint4 o;
  o.x = __byte_perm(int8_to_f32_bits<UNSIGNED>(w.x, 0, offset), int8_to_f32_bits<UNSIGNED>(w.x, 1, offset), 0x7632);
  o.y = __byte_perm(int8_to_f32_bits<UNSIGNED>(w.x, 2, offset), int8_to_f32_bits<UNSIGNED>(w.x, 3, offset), 0x7632);
  o.z = __byte_perm(int8_to_f32_bits<UNSIGNED>(w.y, 0, offset), int8_to_f32_bits<UNSIGNED>(w.y, 1, offset), 0x7632);
  o.w = __byte_perm(int8_to_f32_bits<UNSIGNED>(w.y, 2, offset), int8_to_f32_bits<UNSIGNED>(w.y, 3, offset), 0x7632);
  return o;
}

// A and B in one launch: groups [0, na8) of A, then [0, nb8) of B, 8 values each;
// a_unsigned / b_unsigned pick the reading of each operand, a_offset / b_offset are
// subtracted.  A thread reads 8 bytes and writes 16, so each warp-wide load and
// store covers one contiguous run; each thread keeps WIDEN_UNROLL groups in flight.
constexpr int WIDEN_UNROLL = 4;

__global__ void __launch_bounds__(256) i8_to_bf16_kernel(const uint2* __restrict__ a, uint4* __restrict__ a16,
                                                         int64_t na8, const uint2* __restrict__ b,
                                                         uint4* __restrict__ b16, int64_t nb8, int a_unsigned,
                                                         int b_unsigned, int a_offset, int b_offset) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  const int64_t n = na8 + nb8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i0 < n;
       i0 += stride * WIDEN_UNROLL) {
    uint2 w[WIDEN_UNROLL];
#pragma unroll
    for (int u = 0; u < WIDEN_UNROLL; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n) w[u] = __ldcs(i < na8 ? a + i : b + (i - na8));   // read once
    }
#pragma unroll
    for (int u = 0; u < WIDEN_UNROLL; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= n) continue;
      const bool in_a = i < na8;
      uint4* dst = in_a ? a16 + i : b16 + (i - na8);
      const int off = in_a ? a_offset : b_offset;
      *dst = (in_a ? a_unsigned : b_unsigned) ? widen8<true>(w[u], off) : widen8<false>(w[u], off);
    }
  }
}

// Row sums of A' = A - offset (M x K 8-bit, K % 16 == 0): one warp per row, 16-byte
// loads; exact in i32 (|sum| <= 128 K).
template <bool UNSIGNED>
__global__ void __launch_bounds__(256) int8_rowsum_kernel(const int4* __restrict__ A, int64_t M, int64_t K16,
                                                          int offset, int32_t* __restrict__ r) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < M; row += warps) {
    int acc = 0;
    for (int64_t v = lane; v < K16; v += 32) {
      const int4 w = A[row * K16 + v];
      const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        acc = UNSIGNED ? static_cast<int>(__dp4a(static_cast<unsigned>(words[k]), 0x01010101u, static_cast<unsigned>(acc)))
                       : __dp4a(words[k], 0x01010101, acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) r[row] = acc - static_cast<int>(K16 * 16) * offset;
  }
}

// Column sums of B' = B - offset (K x N 8-bit, N % 16 == 0): a thread sums 4 columns
// over a band of COLSUM_ROWS rows and adds them to c (zeroed first) atomically.
constexpr int COLSUM_ROWS = 64;
template <bool UNSIGNED>
__global__ void __launch_bounds__(256) int8_colsum_kernel(const uint32_t* __restrict__ B, int64_t K, int64_t N4,
                                                          int offset, int32_t* __restrict__ c) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  const int64_t bands = (K + COLSUM_ROWS - 1) / COLSUM_ROWS;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < bands * N4;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t band = t / N4, j4 = t - band * N4;
    const int64_t k0 = band * COLSUM_ROWS, k1 = min(K, k0 + COLSUM_ROWS);
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    for (int64_t k = k0; k < k1; ++k) {
      const uint32_t w = B[k * N4 + j4];
      if (UNSIGNED) {
        s0 += static_cast<int>(w & 0xffu);
        s1 += static_cast<int>((w >> 8) & 0xffu);
        s2 += static_cast<int>((w >> 16) & 0xffu);
        s3 += static_cast<int>(w >> 24);
      } else {
        s0 += static_cast<int8_t>(w);
        s1 += static_cast<int8_t>(w >> 8);
        s2 += static_cast<int8_t>(w >> 16);
        s3 += static_cast<int8_t>(w >> 24);
      }
    }
    const int n = static_cast<int>(k1 - k0) * offset;
    atomicAdd(c + 4 * j4 + 0, s0 - n);
    atomicAdd(c + 4 * j4 + 1, s1 - n);
    atomicAdd(c + 4 * j4 + 2, s2 - n);
    atomicAdd(c + 4 * j4 + 3, s3 - n);
  }
}

// See launch_meta_native.  Both layouts are built from 8-byte chunks of the row-major
// index: chunk (r, z) is bytes [8z, 8z + 8) of row r (K/8 bytes a row), the index of
// one 64-element K slice (f16: two 32-K MMAs; FP8: one 64-K MMA).  A block loads a
// 32-row x 32-chunk tile with loads along the rows, then writes the tensor-core layout
// with stores along r.  kind::f16 (one entry per stage): word kk of the entry of lane r
// holds the 16-bit halves h = (r >> 3) & 1 of word kk of the chunks of rows (r & ~8) and
// (r | 8), the lower row in the low half.  FP8 (one entry per MMA): the row's own chunk.
// Rows past M and slots past the index's (z >= slots, up to slots_out) read as
// 0x44444444 (position pair {0,1} in every group).  `rows` (a multiple of 16 at
// least M: a lane past M can still carry half of a real row's index) rows are
// written per slot, 8 bytes each.
constexpr int kMetaTile = 32;

__global__ void __launch_bounds__(256) meta_native_kernel(const uint2* __restrict__ idx, uint2* __restrict__ native,
                                                          int64_t M, int64_t rows, int64_t slots, int64_t slots_out,
                                                          int f16) {
  griddep_launch_dependents();
  griddep_wait();   // launched with programmatic dependent launch
  __shared__ uint2 tile[kMetaTile][kMetaTile + 1];
  const int64_t tiles_z = (slots_out + kMetaTile - 1) / kMetaTile;
  const int64_t tiles = tiles_z * ((rows + kMetaTile - 1) / kMetaTile);
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_z) * kMetaTile;
    const int64_t z0 = (t % tiles_z) * kMetaTile;
    __syncthreads();   // the previous tile's reads of `tile` are done
    for (int i = threadIdx.x; i < kMetaTile * kMetaTile; i += blockDim.x) {
      const int rr = i / kMetaTile, zz = i % kMetaTile;
      const int64_t r = r0 + rr, z = z0 + zz;
      tile[rr][zz] = (r < M && z < slots) ? idx[r * slots + z] : make_uint2(0x44444444u, 0x44444444u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kMetaTile * kMetaTile; i += blockDim.x) {
      const int zz = i / kMetaTile, rr = i % kMetaTile;
      const int64_t r = r0 + rr, z = z0 + zz;
      if (r >= rows || z >= slots_out) continue;
      uint2 v;
      if (f16) {
        const uint32_t sh = 16u * ((rr >> 3) & 1);
        const uint2 a = tile[rr & ~8][zz], b = tile[rr | 8][zz];
        v.x = ((a.x >> sh) & 0xffffu) | (((b.x >> sh) & 0xffffu) << 16);
        v.y = ((a.y >> sh) & 0xffffu) | (((b.y >> sh) & 0xffffu) << 16);
      } else {
        const uint2 a = tile[rr][zz];
        v.x = a.x;
        v.y = a.y;
      }
      native[z * rows + r] = v;
    }
  }
}

int grid_for(int64_t work, int num_sms) {
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* P, int ksplit, const void* C, void* D, int64_t MN, int out,
                                 int num_sms, cudaStream_t stream) {
  const int64_t n4 = MN / 4;
  const float4* p = reinterpret_cast<const float4*>(P);
  if (out == 1) return launch_pdl(splitk_reduce_kernel<1>, grid_for(n4, num_sms), 256, 0, stream, p, ksplit, n4, C, D);
  if (out == 2) return launch_pdl(splitk_reduce_kernel<2>, grid_for(n4, num_sms), 256, 0, stream, p, ksplit, n4, C, D);
  return launch_pdl(splitk_reduce_kernel<0>, grid_for(n4, num_sms), 256, 0, stream, p, ksplit, n4, C, D);
}

cudaError_t launch_tail_reduce(const TailReduce& r, const GemmArgs& g, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (r.T == 0) return cudaSuccess;
  const int threads = 256, rows_per_block = threads / (r.tile_cols / 4);   // 4 rows of 256 columns
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((r.tile_rows + rows_per_block - 1) / rows_per_block),
                     static_cast<unsigned>(r.T), 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (r.out) {
    case 0: return cudaLaunchKernelEx(&cfg, tail_reduce_kernel<0>, r, g);
    case 1: return cudaLaunchKernelEx(&cfg, tail_reduce_kernel<1>, r, g);
    case 2: return cudaLaunchKernelEx(&cfg, tail_reduce_kernel<2>, r, g);
    default: return cudaLaunchKernelEx(&cfg, tail_reduce_kernel<3>, r, g);
  }
}

cudaError_t launch_splitk_reduce_i32(const int32_t* P, int ksplit, const int32_t* C, int32_t* D, int64_t MN,
                                     bool clamp, const int32_t* rowsum, const int32_t* colsum, int alpha, int beta,
                                     int64_t K, int64_t N, int num_sms, cudaStream_t stream) {
  const int64_t n4 = MN / 4;
  const IntFix fix{rowsum, colsum, alpha, beta, K, N};
  return launch_pdl(splitk_reduce_i32_kernel, grid_for(n4, num_sms), 256, 0, stream, reinterpret_cast<const int4*>(P),
                    ksplit, n4, reinterpret_cast<const int4*>(C), reinterpret_cast<int4*>(D), clamp ? 1 : 0, fix);
}

cudaError_t launch_meta_native(const uint8_t* idx, void* native, int64_t M, int64_t K, bool f16, int64_t rows,
                               int64_t slots_out, int num_sms, cudaStream_t stream) {
  const int64_t slots = K / 64;   // 8 index bytes per row each
  const int64_t tiles = ((slots_out + kMetaTile - 1) / kMetaTile) * ((rows + kMetaTile - 1) / kMetaTile);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(tiles, int64_t(num_sms) * 8))), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, meta_native_kernel, reinterpret_cast<const uint2*>(idx), static_cast<uint2*>(native),
                            M, rows, slots, slots_out, f16 ? 1 : 0);
}

cudaError_t launch_i8_to_bf16(const void* a, bool a_unsigned, int a_offset, uint16_t* a16, int64_t na, const void* b,
                              bool b_unsigned, int b_offset, uint16_t* b16, int64_t nb, int num_sms,
                              cudaStream_t stream) {
  const int64_t na8 = na / 8, nb8 = nb / 8;
  return launch_pdl(i8_to_bf16_kernel, grid_for((na8 + nb8 + WIDEN_UNROLL - 1) / WIDEN_UNROLL, num_sms), 256, 0,
                    stream, static_cast<const uint2*>(a), reinterpret_cast<uint4*>(a16), na8,
                    static_cast<const uint2*>(b), reinterpret_cast<uint4*>(b16), nb8, a_unsigned ? 1 : 0,
                    b_unsigned ? 1 : 0, a_offset, b_offset);
}

cudaError_t launch_int8_rowsum(const void* A, bool is_unsigned, int offset, int64_t M, int64_t K, int32_t* r,
                               int num_sms, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((M + 7) / 8, static_cast<int64_t>(num_sms) * 8);
  if (is_unsigned)
    return launch_pdl(int8_rowsum_kernel<true>, static_cast<int>(blocks), 256, 0, stream,
                      static_cast<const int4*>(A), M, K / 16, offset, r);
  return launch_pdl(int8_rowsum_kernel<false>, static_cast<int>(blocks), 256, 0, stream, static_cast<const int4*>(A),
                    M, K / 16, offset, r);
}

cudaError_t launch_int8_colsum(const void* B, bool is_unsigned, int offset, int64_t K, int64_t N, int32_t* c,
                               int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(c, 0, static_cast<size_t>(N) * sizeof(int32_t), stream);
  if (e != cudaSuccess || K == 0 || N == 0) return e;
  const int64_t N4 = N / 4, work = ((K + COLSUM_ROWS - 1) / COLSUM_ROWS) * N4;
  if (is_unsigned)
    return launch_pdl(int8_colsum_kernel<true>, grid_for(work, num_sms), 256, 0, stream,
                      static_cast<const uint32_t*>(B), K, N4, offset, c);
  return launch_pdl(int8_colsum_kernel<false>, grid_for(work, num_sms), 256, 0, stream,
                    static_cast<const uint32_t*>(B), K, N4, offset, c);
}

}  // namespace mma42
