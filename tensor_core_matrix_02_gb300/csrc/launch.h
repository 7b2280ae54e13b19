// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Internal to libmma42; not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_args.h"

namespace mma42 {

// Launch with programmatic dependent launch allowed (see griddep_wait in ptx.cuh):
// the kernel may be scheduled while the previous kernel in the stream finishes and
// must call griddep_wait() before its first global memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace mma42

namespace mma42 {

// Kernel variants of the tcgen05 GEMM.
enum Variant : int {
  V_DENSE_F16 = 0,   // kind::f16, f16 or bf16 operands, BN = 256
  V_DENSE_F8 = 1,    // kind::f8f6f4, E4M3/E5M2 operands, BN = 256
  V_DENSE_I8 = 2,    // i8 carried exactly as bf16, kind::f16, i32 epilogue, BN = 128
  V_PAIR_F16 = 3,    // CTA pair (cta_group::2), 256 x 256 blocks, f16 or bf16
  V_PAIR_F8 = 4,     // CTA pair, E4M3/E5M2
  V_PAIR_I8 = 5,     // CTA pair, i8 carried exactly as bf16, i32 chunk sums
  V_PAIR_F16_OUTH = 6,    // CTA pair, f16 operands, f16 C and D
  V_PAIR_BF16_OUTH = 7,   // CTA pair, bf16 operands, bf16 C and D
  V_DENSE_F16_N128 = 8,   // as V_DENSE_F16 with BN = 128, for outputs at most 128 columns wide
  V_DENSE_F8_N128 = 9,    // as V_DENSE_F8 with BN = 128, likewise
  V_COUNT = 10
};

inline bool is_pair(Variant v) { return v >= V_PAIR_F16 && v <= V_PAIR_BF16_OUTH; }

// Tile geometry of a variant (what the host needs to build tensor maps).
struct VariantInfo {
  int bm, bn;           // output tile
  int elem;             // bytes per A/B element
  int bka;              // A elements per stage row
  int bkl;              // K per stage
  int b_atom_n;         // B box width (elements)
  int stages;
  int smem_bytes;
  int threads;
};

// Geometry of the 4:2-sparse CTA-pair kernel for one type kind.
struct SparseInfo {
  int bm, bn;           // rows per CTA (2*bm per instruction), columns per pair
  int bka;              // compressed A elements per stage row (64 bytes)
  int bkl;              // logical K per stage
  int mmas;             // tcgen05.mma.sp per stage
  int meta_slots;       // index slots (64 logical K each) per stage
  int b_atom_n;         // B box width (elements)
  int b_chunks;         // b_atom_n-wide column chunks of B per CTA and stage
  int b_rows_per_cta;   // K rows of each B box
  int epi_cols;         // f32 columns of the epilogue's C and D boxes (32: 128-byte rows, or 16)
  int smem_bytes;
  int threads;
};

struct TensorMaps {
  CUtensorMap a, b, meta, c, d, p;
};

VariantInfo variant_info(Variant v);
VariantInfo pair_variant_info(Variant v);
int pair_variant_max_clusters(Variant v);
cudaError_t pair_variant_launch(Variant v, const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_gemm(Variant v, const TensorMaps& maps, const GemmArgs& args, int grid,
                        cudaStream_t stream);

// CTA-pair (cta_group::2) sparse GEMM: 256 x 256 blocks on clusters of two CTAs.
SparseInfo sparse_pair_f16_info();
SparseInfo sparse_pair_f8_info();
int sparse_pair_f16_max_clusters();
int sparse_pair_f8_max_clusters();
cudaError_t sparse_pair_f16_launch(const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t sparse_pair_f8_launch(const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s);
// the exact i8 variant of the kind::f16 kernel (bf16 operands, i32 chunk sums; C and D i32)
int sparse_pair_i8_max_clusters();
cudaError_t sparse_pair_i8_launch(const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s);
// Device-native index layout for the sparse GEMM: slot z holds the index of logical K
// [64 z, 64 z + 64); for each of `rows` rows (a multiple of 16, at least M), the 8
// bytes TMEM lane r % 128 needs (kind::f16 pairs rows r and r^8, one 32-bit word per
// 32-K MMA; FP8 uses each row's own 8 bytes).  Rows past M and slots from K / 64 up
// to `slots_out` (a last stage that runs past K) hold positions {0, 1} everywhere.
cudaError_t launch_meta_native(const uint8_t* idx, void* native, int64_t M, int64_t K, bool f16, int64_t rows,
                               int64_t slots_out, int num_sms, cudaStream_t stream);

// D = C + sum_s P[s]   (P: ksplit x M x N f32, fixed summation order); out: C and D
// type, 0 f32, 1 f16, 2 bf16 (the f32 sum rounded to nearest even).
cudaError_t launch_splitk_reduce(const float* P, int ksplit, const void* C, void* D, int64_t MN, int out,
                                 int num_sms, cudaStream_t stream);
// D = C + sum_s P[s] for i32 partials (ksplit x M x N), exact in 64 bits; clamp
// saturates to the i32 range, otherwise the sum wraps modulo 2^32.
// rowsum / colsum / alpha / beta / K / N: the corrections of unsigned operands run as
// signed ones (D += beta * rowsum[i] + alpha * colsum[j] + alpha * beta * K).
// Throughput ceiling of the warp-level MMA path (legacy_peak.cu): kind 0 s8, 1 s8
// 4:2-sparse, 2 bf16, 3 E4M3.  The kernel runs legacy_peak_grid(num_sms) blocks and
// writes one word per thread to sink (legacy_peak_sink_words); legacy_peak_ops is the
// work of one launch in ops (2 per multiply-add, logical K for the sparse kind).
double legacy_peak_ops_per_mma(int kind);
int legacy_peak_grid(int num_sms);
size_t legacy_peak_sink_words(int num_sms);
double legacy_peak_ops(int kind, int64_t iters, int num_sms);
cudaError_t launch_legacy_peak(int kind, int64_t iters, uint32_t* sink, int num_sms, cudaStream_t stream);

// Throughput ceiling of tcgen05.mma (tc_peak.cu): kind 0 kind::f16 dense (bf16), 1
// kind::f8f6f4 dense (E4M3), 2 and 3 their 4:2-sparse forms; CTA-pair instructions
// (M = N = 256) on one resident stage per pair.  The kernel runs `clusters` clusters
// of two CTAs (at most tc_peak_max_clusters(kind)) and writes each cluster's SM
// cycles from its first MMA to the completion of its last to cycles[cluster];
// tc_peak_ops_per_cluster_iter is the ops one cluster does per iteration.
double tc_peak_ops_per_cluster_iter(int kind);
int tc_peak_max_clusters(int kind);
cudaError_t launch_tc_peak(int kind, int64_t iters, uint32_t idesc, uint64_t wait_ns, unsigned long long* cycles,
                           int* err, int clusters, cudaStream_t stream);

// Short-K GEMM (gemm_small.cu): one CTA per 128 x 128 block, K at most kb_max * bk,
// f32 C and D; C and D maps of 32 x 32 f32 boxes (128-byte swizzle), A of bk x 128,
// B of b_atom_n x bk boxes.  Launched with programmatic dependent launch.
struct SmallInfo {
  int bm, bn, bk, b_atom_n, kb_max;
};
// `narrow`: 64-column blocks (16-bit operands only; FP8 blocks stay 128 wide).
SmallInfo small_info(bool f8, bool narrow);
// bn: 128, or 64 for 16-bit operands; anything else is cudaErrorInvalidValue.
cudaError_t launch_small(bool f8, int bn, const TensorMaps& m, const GemmArgs& a, cudaStream_t stream);

// TMA feed probe (feed_probe.cu): the producer loop of the CTA-pair kernels alone.
// Up to four boxes per stage (rows x row_bytes each, placed at smem_off within the
// stage), `stages` stages of stage_bytes, iters stages per CTA; the maps are 2-D
// byte matrices of feed_probe_row_pitch()-byte rows and `height` rows, one per box.
// cycles[cluster] receives the SM cycles of the stages after the first
// feed_probe_warm_stages() (0 if a wait ran out).
struct FeedProbe {
  int nbox;
  int rows[4], row_bytes[4], smem_off[4];
  int stages, stage_bytes, iters, height;
};
int feed_probe_max_clusters(int smem_bytes);
int feed_probe_row_pitch();
int feed_probe_warm_stages();
cudaError_t launch_feed_probe(const FeedProbe& p, const CUtensorMap* maps, int clusters, uint64_t wait_ns, int* err,
                              unsigned long long* cycles, cudaStream_t stream);

// Tail split of the CTA-pair kernel: D = C + sum_s P[s] over the tail tiles only.
// P is compact: tail_split x (T * tile_rows) x tile_cols, tile t of the tail being
// raster tile tail_from + t of the GEMM described by g (tiles_m, tiles_n, group_m).
// out: 0 f32, 1 f16, 2 bf16 (f32 partials, summed in slice order, then + C), 3 i32
// (i32 partials, wrapping, plus the corrections of unsigned operands run as signed
// ones when alpha or beta is non-zero).
struct TailReduce {
  const void* P;
  int S, T;                 // K slices, tail tiles
  int tile_rows, tile_cols;
  const void* C;
  void* D;
  int64_t M, N, K;
  int out;
  const int32_t* rowsum;
  const int32_t* colsum;
  int alpha, beta;
};
cudaError_t launch_tail_reduce(const TailReduce& r, const GemmArgs& g, int num_sms, cudaStream_t stream);
cudaError_t launch_splitk_reduce_i32(const int32_t* P, int ksplit, const int32_t* C, int32_t* D, int64_t MN,
                                     bool clamp, const int32_t* rowsum, const int32_t* colsum, int alpha, int beta,
                                     int64_t K, int64_t N, int num_sms, cudaStream_t stream);
// a16[i] = (bf16) (a[i] - a_offset), b16[i] = (bf16) (b[i] - b_offset) for 8-bit
// integers a and b, each read as signed or unsigned, in one launch; exact while the
// shifted values stay within 8 significant bits.  na and nb multiples of 16.
cudaError_t launch_i8_to_bf16(const void* a, bool a_unsigned, int a_offset, uint16_t* a16, int64_t na, const void* b,
                              bool b_unsigned, int b_offset, uint16_t* b16, int64_t nb, int num_sms,
                              cudaStream_t stream);
// r[i] = sum_k (A[i][k] - offset) for an M x K 8-bit A (K % 16 == 0); exact i32.
cudaError_t launch_int8_rowsum(const void* A, bool is_unsigned, int offset, int64_t M, int64_t K, int32_t* r,
                               int num_sms, cudaStream_t stream);
// c[j] = sum_k (B[k][j] - offset) for a K x N 8-bit B (N % 16 == 0); exact i32.
cudaError_t launch_int8_colsum(const void* B, bool is_unsigned, int offset, int64_t K, int64_t N, int32_t* c,
                               int num_sms, cudaStream_t stream);
// f32 -> kind (0 f16, 1 bf16, 2 E4M3, 3 E5M2): saturate, round to nearest even.
// x 16-byte aligned, y 16-byte aligned; any n >= 0.
cudaError_t launch_quantize(const float* x, void* y, int64_t n, int kind, int num_sms, cudaStream_t stream);
// f32 A (M x K, K % 32 == 0) -> quantised to qkind (0 f16, 1 bf16, 2 E4M3, 3 E5M2),
// pruned to 4:2 by the quantised magnitudes and compressed, in one pass.
cudaError_t launch_quantize_prune(const float* A, void* vals, uint8_t* idx, int64_t M, int64_t K, int qkind,
                                  int32_t* d_dropped, int num_sms, cudaStream_t stream);
// 4:2 compression (prune == 0), or pruning by magnitude then compression (see
// mma42.h for both rules; prune 1 floating types, 2 i8, 3 u8); elem is 1 or 2 bytes;
// d_violations counts groups with more than two non-zeros (kept as the two lowest,
// or pruned to the two largest).
cudaError_t launch_compress42(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K,
                              int elem, int zero_mask, int prune, int32_t* d_violations, int num_sms,
                              cudaStream_t stream);

}  // namespace mma42
