// feed_probe.cu -- how fast TMA fills the pipeline ring of a CTA pair, measured
// with nothing consuming the data.
//
// Every SM pair (a cluster of two CTAs) runs the producer loop of the CTA-pair GEMM
// kernels alone: for each stage, lane 0 of warp 0 of both CTAs waits for the
// stage's empty barrier and issues its boxes with the pair form of the tiled TMA
// load (cp.async.bulk.tensor ... cta_group::2), all completing on CTA 0's full
// barrier; one thread of CTA 0 waits for each stage to fill and releases it to
// both producers at once, with no MMA.  So the rate is the ceiling that TMA, L2 and
// the SM's shared-memory fill path give the GEMMs' pipelines for that stage shape,
// and the box shapes (rows x row bytes, boxes per stage) can be varied to see
// whether bytes or box rows set it.
//
// The source is a device buffer the host allocates, read as 2-D byte matrices of
// 16384-byte rows, one quarter per box of the stage.  CTA r of cluster c reads the
// row band starting at (2 c + r) * 128 (wrapped), advancing along the rows' bytes
// stage by stage; a buffer that fits in L2 measures the L2 -> shared memory feed.
// The consumer counts SM cycles (clock64) over all but the first stages, so the
// figure does not depend on the clock the power limit allows.  Every wait is
// bounded; a wait that runs out raises the device error word, and the consumer
// then waits out the limit twice so that every issued load has landed.
#include <cstdint>

#include "gemm_kernel.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace mma42 {

namespace {

constexpr int kFeedThreads = 64;
constexpr int kFeedRowBytes = 16384;   // row pitch of the source matrices
constexpr int kFeedWarmStages = 128;   // stages before the cycle count starts

struct FeedArgs {
  int nbox;
  int rows[4];
  int row_bytes[4];
  int smem_off[4];
  int stages;
  int stage_bytes;
  int iters;          // stages per CTA
  int height;         // rows of each source quarter
  unsigned long long wait_ns;
  int* err;
  unsigned long long* cycles;   // per cluster
};

// Bounded wait on an mbarrier phase (the probe has no abort flag: every role
// gives up on its own after the limit).
__device__ __forceinline__ bool feed_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, 1);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kFeedThreads, 1)
    feed_probe_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                      const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
                      const FeedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + a.stages * a.stage_bytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (a.stages + s); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_id_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_fence_init();
  }
  cluster_sync();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    // (the box loop is unrolled so that each map is named directly: a map picked
    // through a runtime-indexed pointer would be copied to local memory and read
    // from there by every copy, as the GEMM kernels never do)
    int y[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const CUtensorMap* m = b == 0 ? &m0 : b == 1 ? &m1 : b == 2 ? &m2 : &m3;
      if (b < a.nbox) prefetch_tensormap(m);
      y[b] = b < a.nbox ? ((2 * cid + rank) * 128) % (a.height - a.rows[b] + 1) : 0;
    }
    int stage = 0;
    uint32_t phase = 0;
    for (int it = 0; it < a.iters; ++it) {
      if (!feed_wait(empty_bar(stage), phase ^ 1u, a.wait_ns, a.err)) break;
      const uint32_t fb = mapa_shared(full_bar(stage), 0);
      if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2u * static_cast<uint32_t>(a.stage_bytes));
      const uint32_t dst = sbase + stage * a.stage_bytes;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const CUtensorMap* m = b == 0 ? &m0 : b == 1 ? &m1 : b == 2 ? &m2 : &m3;
        if (b < a.nbox) {
          const int x = (it * a.row_bytes[b]) & (kFeedRowBytes - 1);
          tma_load_2d_pair(dst + a.smem_off[b], m, x, y[b], fb);
        }
      }
      if (++stage == a.stages) { stage = 0; phase ^= 1u; }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------------------------------------------------------- consumer
    int stage = 0;
    uint32_t phase = 0;
    long long t0 = 0, t1 = 0;
    bool ok = true;
    for (int it = 0; it < a.iters; ++it) {
      if (!feed_wait(full_bar(stage), phase, a.wait_ns, a.err)) { ok = false; break; }
      if (it == kFeedWarmStages - 1) t0 = clock64();
      t1 = clock64();
      // both CTAs' copies of this stage have landed: hand it back to both producers
      mbar_arrive_cluster(mapa_shared(empty_bar(stage), 0));
      mbar_arrive_cluster(mapa_shared(empty_bar(stage), 1));
      if (++stage == a.stages) { stage = 0; phase ^= 1u; }
    }
    a.cycles[cid] = ok ? static_cast<unsigned long long>(t1 - t0) : 0ull;
    if (!ok) {
      // the producers stop within one limit of their own; their issued loads land
      // microseconds later
      const uint64_t w0 = global_timer_ns();
      while (global_timer_ns() - w0 < 2 * a.wait_ns) {
      }
    }
  }
  __syncwarp();
  __syncthreads();
  cluster_sync();
}

}  // namespace

int feed_probe_max_clusters(int smem_bytes) {
  if (cudaFuncSetAttribute(feed_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(kFeedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(feed_probe_kernel), &cfg) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_feed_probe(const FeedProbe& p, const CUtensorMap* maps, int clusters, uint64_t wait_ns, int* err,
                              unsigned long long* cycles, cudaStream_t stream) {
  FeedArgs a = {};
  a.nbox = p.nbox;
  for (int b = 0; b < 4; ++b) {
    a.rows[b] = p.rows[b];
    a.row_bytes[b] = p.row_bytes[b];
    a.smem_off[b] = p.smem_off[b];
  }
  a.stages = p.stages;
  a.stage_bytes = p.stage_bytes;
  a.iters = p.iters;
  a.height = p.height;
  a.wait_ns = wait_ns;
  a.err = err;
  a.cycles = cycles;
  const int smem = p.stages * p.stage_bytes + 1024 + 256;
  cudaError_t e = cudaFuncSetAttribute(feed_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kFeedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, feed_probe_kernel, maps[0], maps[1], maps[2], maps[3], a);
}

int feed_probe_row_pitch() { return kFeedRowBytes; }
int feed_probe_warm_stages() { return kFeedWarmStages; }

}  // namespace mma42
