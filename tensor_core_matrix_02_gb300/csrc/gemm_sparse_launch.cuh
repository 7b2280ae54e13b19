// gemm_sparse_launch.cuh -- instantiation and cluster launch of the 4:2-sparse GEMM.
#pragma once
#include "gemm_sparse_pair_kernel.cuh"
#include "launch.h"

namespace mma42 {

template <int KIND>
SparseInfo sparse_pair_info_of() {
  using Cfg = SparsePairCfg<KIND>;
  SparseInfo i;
  i.bm = Cfg::BM;
  i.bn = Cfg::BN;
  i.bka = Cfg::BKA;
  i.bkl = Cfg::BKL;
  i.mmas = Cfg::MMAS;
  i.meta_slots = Cfg::META_SLOTS;
  i.b_atom_n = Cfg::B_ATOM_N;
  i.b_chunks = Cfg::B_CHUNKS;
  i.b_rows_per_cta = Cfg::BKL;
  i.epi_cols = Cfg::EPI_COLS;
  i.smem_bytes = Cfg::SMEM_BYTES;
  i.threads = Cfg::THREADS;
  return i;
}

inline cudaLaunchConfig_t cluster_config(int grid, int threads, int smem, int cl, cudaStream_t stream,
                                         cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see griddep_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int KIND, bool INTACC = false>
int sparse_pair_max_clusters() {
  using Cfg = SparsePairCfg<KIND>;
  auto kernel = gemm_sparse_pair_kernel<KIND, INTACC>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return 0;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(2 * 256, Cfg::THREADS, Cfg::SMEM_BYTES, 2, nullptr, attr);
  cfg.numAttrs = 1;   // the cluster shape is what the occupancy depends on
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<void*>(kernel), &cfg) != cudaSuccess) return 0;
  return n;
}

template <int KIND, bool INTACC = false>
cudaError_t sparse_pair_launch(const TensorMaps& m, const GemmArgs& args, int grid, cudaStream_t stream) {
  using Cfg = SparsePairCfg<KIND>;
  auto kernel = gemm_sparse_pair_kernel<KIND, INTACC>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(grid, Cfg::THREADS, Cfg::SMEM_BYTES, 2, stream, attr);
  return cudaLaunchKernelEx(&cfg, kernel, m.a, m.b, m.c, m.d, args);
}

}  // namespace mma42
