// tc_peak.cu -- the throughput ceiling of tcgen05.mma on the running GPU, measured.
//
// Every SM pair (a cluster of two CTAs) allocates TMEM, fills one pipeline stage of
// operands in shared memory -- the same tile layouts, descriptors and instruction
// shapes as the CTA-pair GEMM kernels (M = 256, N = 256 per instruction) -- and one
// thread issues that stage's MMAs over and over, with no TMA traffic and no
// epilogue.  So the rate is what the tensor cores sustain on operands already in
// shared memory: the ceiling the GEMMs' pipelines feed towards.
//
// Kinds (ops counted as 2 per multiply-add, logical K for the 4:2-sparse forms):
//   0  kind::f16 dense, bf16 x bf16 -> f32            K 16 per instruction
//   1  kind::f8f6f4 dense, E4M3 x E4M3 -> f32          K 32
//   2  kind::f16 4:2-sparse, bf16 -> f32               K 32 (logical)
//   3  kind::f8f6f4 4:2-sparse, E4M3 -> f32            K 64 (logical)
// The index of the sparse kinds names positions {0, 1} of every group of four.
//
// The issuing thread counts SM clock cycles from its first MMA to the completion
// of its last (clock64), so the ops per clock per SM come out independent of the
// clock the power limit allows; the host times the launch for ops per second.
#include <cstdint>

#include "gemm_pair_kernel.cuh"
#include "gemm_sparse_pair_kernel.cuh"
#include "launch.h"

namespace mma42 {

namespace {

constexpr int kPeakCtaThreads = 128;
// enough dynamic shared memory that no two CTAs share an SM (each allocates all of
// its SM's TMEM)
constexpr int kPeakSmemBytes = 160 * 1024;

__device__ __forceinline__ uint32_t peak_mix(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Shapes of one stage, taken from the GEMM kernels' own configurations.
template <int KIND, bool SPARSE>
struct PeakShape;
template <int KIND>
struct PeakShape<KIND, false> {
  using Cfg = PairCfg<KIND, false>;
  static constexpr int A_BYTES = Cfg::A_BYTES;
  static constexpr int B_BYTES = Cfg::B_BYTES;
  static constexpr int META_BYTES = 0;
  static constexpr int MMAS = Cfg::MMAS;
  static constexpr int K_PER_MMA = Cfg::UMMA_K;
};
template <int KIND>
struct PeakShape<KIND, true> {
  using Cfg = SparsePairCfg<KIND>;
  static constexpr int A_BYTES = Cfg::A_BYTES;
  static constexpr int B_BYTES = Cfg::B_BYTES;
  static constexpr int META_BYTES = Cfg::META_BYTES;
  static constexpr int MMAS = Cfg::MMAS;
  static constexpr int K_PER_MMA = Cfg::UMMA_KL;
};

template <int KIND, bool SPARSE>
__global__ void __launch_bounds__(kPeakCtaThreads, 1)
    tc_peak_kernel(int64_t iters, uint32_t idesc, uint64_t wait_ns, unsigned long long* __restrict__ cycles,
                   int* __restrict__ err) {
  using Sh = PeakShape<KIND, SPARSE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sa = smem_addr(smem);
  const uint32_t sb = sa + Sh::A_BYTES;
  const uint32_t sm = sb + Sh::B_BYTES;
  uint8_t* misc = smem + Sh::A_BYTES + Sh::B_BYTES + Sh::META_BYTES;
  const uint32_t done_bar = smem_addr(misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8);
  (void)sm;   // the index tiles (sparse kinds only)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_id_x());

  // operands: pseudo-random finite values of magnitude [0.5, 1) and either sign
  // (bf16: exponent 126; E4M3: exponent field 6), so the data toggles as in a GEMM
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  const uint32_t seed = static_cast<uint32_t>(blockIdx.x) << 20;
  for (int i = threadIdx.x; i < (Sh::A_BYTES + Sh::B_BYTES) / 4; i += blockDim.x) {
    const uint32_t h = peak_mix(seed ^ static_cast<uint32_t>(i));
    words[i] = (KIND == KIND_F16) ? ((h & 0x807f807fu) | 0x3f003f00u) : ((h & 0x87878787u) | 0x30303030u);
  }
  for (int i = threadIdx.x; i < Sh::META_BYTES / 4; i += blockDim.x)
    words[(Sh::A_BYTES + Sh::B_BYTES) / 4 + i] = 0x44444444u;   // positions {0, 1} in every group
  fence_proxy_async_smem();   // the generic-proxy writes above are read by the tensor cores
  if (threadIdx.x == 0) {
    mbar_init(done_bar, 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 1 && lane == 0) {
    if (rank == 0) {
      const uint32_t meta = tmem_base + 256;   // after the 256 accumulator columns
      if constexpr (SPARSE) {
        using Cfg = typename Sh::Cfg;
#pragma unroll
        for (int sl = 0; sl < Cfg::META_SLOTS; ++sl)
          tmem_cp_pair_128x128b(meta + sl * Cfg::META_SLOT_COLS,
                                smem_desc(sm + sl * Cfg::META_SLOT_BYTES, Cfg::META_SLOT_BYTES, 128, LAYOUT_NONE));
      }
      const long long t0 = clock64();
      for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < Sh::MMAS; ++kk) {
          using Cfg = typename Sh::Cfg;
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          if constexpr (SPARSE) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
            const uint32_t mslot = meta + (kk / Cfg::MMAS_PER_SLOT) * Cfg::META_SLOT_COLS;
            const uint32_t id = idesc | static_cast<uint32_t>(kk % Cfg::MMAS_PER_SLOT);
            umma_sp_pair<KIND>(tmem_base, ad, bd, mslot, id, acc);
          } else {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
            umma_pair<KIND>(tmem_base, ad, bd, idesc, acc);
          }
        }
      }
      umma_commit_pair_mc(done_bar, 3);
      bool ok = mbar_try_wait(done_bar, 0);
      const uint64_t w0 = global_timer_ns();
      while (!ok && global_timer_ns() - w0 <= wait_ns) ok = mbar_try_wait(done_bar, 0);
      const long long t1 = clock64();
      if (!ok) atomicOr(err, 1);
      cycles[cid] = static_cast<unsigned long long>(t1 - t0);
    } else {
      // the commit arrives on both CTAs' barriers: the pair's MMAs, which write this
      // CTA's TMEM, are done before it is freed
      bool ok = mbar_try_wait(done_bar, 0);
      const uint64_t w0 = global_timer_ns();
      while (!ok && global_timer_ns() - w0 <= wait_ns) ok = mbar_try_wait(done_bar, 0);
      if (!ok) atomicOr(err, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <int KIND, bool SPARSE>
cudaError_t launch_peak_kind(int64_t iters, uint32_t idesc, uint64_t wait_ns, unsigned long long* cycles, int* err,
                             int clusters, cudaStream_t stream) {
  auto kernel = tc_peak_kernel<KIND, SPARSE>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kPeakCtaThreads, 1, 1);
  cfg.dynamicSmemBytes = kPeakSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, iters, idesc, wait_ns, cycles, err);
}

template <int KIND, bool SPARSE>
int max_clusters_kind() {
  auto kernel = tc_peak_kernel<KIND, SPARSE>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmemBytes) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(kPeakCtaThreads, 1, 1);
  cfg.dynamicSmemBytes = kPeakSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void*>(kernel), &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace

double tc_peak_ops_per_cluster_iter(int kind) {
  switch (kind) {
    case 0: return 2.0 * 256 * 256 * PeakShape<KIND_F16, false>::K_PER_MMA * PeakShape<KIND_F16, false>::MMAS;
    case 1: return 2.0 * 256 * 256 * PeakShape<KIND_F8, false>::K_PER_MMA * PeakShape<KIND_F8, false>::MMAS;
    case 2: return 2.0 * 256 * 256 * PeakShape<KIND_F16, true>::K_PER_MMA * PeakShape<KIND_F16, true>::MMAS;
    case 3: return 2.0 * 256 * 256 * PeakShape<KIND_F8, true>::K_PER_MMA * PeakShape<KIND_F8, true>::MMAS;
    default: return 0.0;
  }
}

int tc_peak_max_clusters(int kind) {
  switch (kind) {
    case 0: return max_clusters_kind<KIND_F16, false>();
    case 1: return max_clusters_kind<KIND_F8, false>();
    case 2: return max_clusters_kind<KIND_F16, true>();
    default: return max_clusters_kind<KIND_F8, true>();
  }
}

cudaError_t launch_tc_peak(int kind, int64_t iters, uint32_t idesc, uint64_t wait_ns, unsigned long long* cycles,
                           int* err, int clusters, cudaStream_t stream) {
  switch (kind) {
    case 0: return launch_peak_kind<KIND_F16, false>(iters, idesc, wait_ns, cycles, err, clusters, stream);
    case 1: return launch_peak_kind<KIND_F8, false>(iters, idesc, wait_ns, cycles, err, clusters, stream);
    case 2: return launch_peak_kind<KIND_F16, true>(iters, idesc, wait_ns, cycles, err, clusters, stream);
    default: return launch_peak_kind<KIND_F8, true>(iters, idesc, wait_ns, cycles, err, clusters, stream);
  }
}

}  // namespace mma42
