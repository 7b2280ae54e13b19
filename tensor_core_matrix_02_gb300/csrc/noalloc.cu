// noalloc.cu -- mma_gemm_splitk_noalloc: the K-split dense GEMM with its scratch in
// a fixed device array, for callers that cannot allocate device memory.
//
// Who needs it: some callers may not call the CUDA allocator at the point where
// they want a product.  Examples: a process whose device memory is owned by
// another framework's caching allocator, so a cudaMalloc of ours would fail or
// fragment it; a latency-critical loop, where cudaMalloc/cudaFree may block on
// device-wide synchronisation; a runtime whose policy allows no allocation after
// start-up.  mma_gemm takes its split-K partials from a pool the library grows on
// demand; this entry point instead keeps them in g_splitk_scratch below, a
// file-scope device array that the CUDA module creates on every device that loads
// the library and that lives until the process exits.  The call allocates nothing
// and frees nothing.
//
// Contract (also in include/mma42.h):
//  * ksplit * M * N * 4 bytes must fit in kScratchBytes (32 MiB); larger requests,
//    ksplit outside [2, 16] and ksplit above the number of K blocks (so also
//    K == 0) are rejected with MMA_ERR_SHAPE before anything is launched.
//  * A, B, C, D and the stream belong to the current device; a D that is not
//    device memory of the current device is rejected with MMA_ERR_INVALID_ARG.
//  * Every call on a device uses the same array and it keeps the last call's
//    contents.  Nothing in it needs to start at zero: each call writes every
//    partial element it later reads.  Calls whose work overlaps on the GPU (two
//    streams, or two host threads) race on the array and give wrong results.
//  * The first call on each device does a one-time set-up (it looks up the
//    array's device address with cudaGetSymbolAddress, with that device current).
//    Make that first call before any stream capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/mma42.h"
#include "host_util.h"
#include "launch.h"

namespace {

constexpr int64_t kScratchFloats = int64_t(8) << 20;   // 8 Mi floats
constexpr int64_t kScratchBytes = kScratchFloats * 4;  // 32 MiB
static_assert(kScratchBytes == (int64_t(32) << 20), "the header documents a 32 MiB array");

// The split-K partials: ksplit slices of M x N f32.  In host code this name is
// only a stand-in for the device array; kernels get its device address, which
// the set-up below reads with cudaGetSymbolAddress.
static __device__ __align__(256) float g_splitk_scratch[kScratchFloats];

struct NoAllocDevice {
  bool ready = false;
  float* scratch = nullptr;   // device address of g_splitk_scratch on this device
  int* err = nullptr;         // device error word
  int num_sms = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_na_mutex;
NoAllocDevice g_na[kMaxDevices];

// One-time set-up per device, with that device current.  Allocates nothing.
mma_status_t noalloc_device(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MMA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& s = g_na[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitk_scratch) != cudaSuccess || !p) return MMA_ERR_CUDA;
    s.scratch = static_cast<float*>(p);
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MMA_ERR_CUDA;
    s.err = mma42::host::error_word();
    if (!s.err || !mma42::host::ensure_encoder()) return MMA_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return MMA_OK;
}

// p is device memory of the current device (a query; allocates nothing)
bool on_current_device(const void* p) {
  int dev = 0;
  cudaPointerAttributes at;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();   // clear a sticky query error
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

bool float_types(const mma_dtypes_t& t) {
  if (t.acc != MMA_F32) return false;
  if (t.a == MMA_F16 && t.b == MMA_F16) return true;
  if (t.a == MMA_BF16 && t.b == MMA_BF16) return true;
  return mma42::host::fp8_type(t.a) && mma42::host::fp8_type(t.b);
}

}  // namespace

extern "C" mma_status_t mma_gemm_splitk_noalloc(const void* A, const void* B, const void* C, void* D, int64_t M,
                                                int64_t N, int64_t K, mma_dtypes_t t, int32_t ksplit,
                                                void* stream) {
  using namespace mma42;
  if (!float_types(t)) return MMA_ERR_UNSUPPORTED;
  const int ea = host::elem_size(t.a), eb = host::elem_size(t.b);
  mma_status_t st = host::check_gemm_args(A, K * ea, M * K * ea, B, C, D, M, N, K, eb, 4);
  if (st != MMA_OK || M == 0 || N == 0) return st;
  const bool f8 = host::fp8_type(t.a);
  // outputs at most 128 wide take 128-column blocks, as in mma_gemm: no MMA, B
  // staging or epilogue work on columns past N
  const Variant v = N <= 128 ? (f8 ? V_DENSE_F8_N128 : V_DENSE_F16_N128) : (f8 ? V_DENSE_F8 : V_DENSE_F16);
  const VariantInfo vi = variant_info(v);
  const int64_t kblocks = (K + vi.bkl - 1) / vi.bkl;
  if (ksplit < 2 || ksplit > 16 || ksplit > kblocks) return MMA_ERR_SHAPE;
  if (M * N > kScratchFloats / ksplit) return MMA_ERR_SHAPE;   // ksplit * M * N floats must fit

  NoAllocDevice* dev = nullptr;
  if ((st = noalloc_device(&dev)) != MMA_OK) return st;
  // the array lives on the current device: an output on another device would have
  // the kernel read and write the wrong GPU's memory
  if (!on_current_device(D)) return MMA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + vi.bm - 1) / vi.bm);
  a.tiles_n = static_cast<int>((N + vi.bn - 1) / vi.bn);
  a.kblocks = static_cast<int>(kblocks);
  a.ksplit = ksplit;
  a.chunk_kb = 0;
  a.group_m = 16;
  a.idesc = host::instr_desc(host::format_code(t.a), host::format_code(t.b), vi.bn, false);
  a.err = dev->err;
  a.wait_ns = host::wait_limit_ns();
  a.inject = 0;
  const int64_t units = static_cast<int64_t>(a.tiles_m) * a.tiles_n * ksplit;
  const int grid = static_cast<int>(std::min<int64_t>(units, dev->num_sms));

  TensorMaps m;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(K) * ea};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.bka), static_cast<uint32_t>(vi.bm)};
    if (!host::encode_map(&m.a, host::map_type(ea), 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MMA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * eb};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.b_atom_n), static_cast<uint32_t>(vi.bkl)};
    if (!host::encode_map(&m.b, host::map_type(eb), 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MMA_ERR_CUDA;
  }
  m.meta = m.a;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * 4};
    const uint32_t box[2] = {32u, 32u};
    if (!host::encode_map(&m.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !host::encode_map(&m.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MMA_ERR_CUDA;
  }
  {
    // partial slice s of the scratch holds rows x columns of the M x N output
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M), static_cast<uint64_t>(ksplit)};
    const uint64_t str[2] = {static_cast<uint64_t>(N) * 4, static_cast<uint64_t>(M) * N * 4};
    const uint32_t box[3] = {32u, 32u, 1u};
    if (!host::encode_map(&m.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dev->scratch, dims, str, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
      return MMA_ERR_CUDA;
  }
  cudaError_t e = launch_gemm(v, m, a, grid, s);
  if (e == cudaSuccess) {
    host::count_launches(1);
    e = launch_splitk_reduce(dev->scratch, ksplit, C, D, M * N, 0,
                             dev->num_sms, s);
    if (e == cudaSuccess) host::count_launches(1);
  }
  return e == cudaSuccess ? MMA_OK : MMA_ERR_CUDA;
}
