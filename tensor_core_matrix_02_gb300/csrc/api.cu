// api.cu -- the C ABI of libmma42 (declared in include/mma42.h): argument
// checks, tensor-map encoding, tile/split planning and kernel dispatch.
//
// Every check that can fail is made on the host before any CUDA call, so a
// rejected call launches nothing and returns its status at once.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/mma42.h"
#include "launch.h"

namespace mma42 {

VariantInfo dense_variant_info(Variant v);
cudaError_t launch_dense(Variant v, const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s);

VariantInfo variant_info(Variant v) { return dense_variant_info(v); }
cudaError_t launch_gemm(Variant v, const TensorMaps& m, const GemmArgs& a, int grid, cudaStream_t s) {
  return launch_dense(v, m, a, grid, s);
}

}  // namespace mma42

using namespace mma42;

// Device error word: raised by a kernel whose bounded pipeline wait ran out.
__device__ int g_mma42_error;

namespace {

constexpr int kMaxDevices = 64;
// K elements per exactly accumulated f32 chunk for 8-bit integer operands: the
// largest power of two (at most 1024, at least one 64-element k-step) whose
// products, of magnitude at most amax * bmax (128 signed, 255 unsigned), sum to
// at most 2^sum_bits.  Every integer of magnitude <= 2^24 is exact in f32, and a
// sum that stays within it loses no bit to alignment in the tensor core's f32
// accumulation (its inputs never exceed 2^24 - 2^14 before the last step), so
// sum_bits is 24: signed x signed 1024, mixed 512, unsigned x unsigned 256.
// MMA42_INT_SUM_BITS (18..24) lowers it for tests and measurements.
int int_sum_bits() {
  int bits = 24;
  if (const char* env = std::getenv("MMA42_INT_SUM_BITS")) {
    const int v = std::atoi(env);
    if (v >= 18 && v <= 24) bits = v;
  }
  return bits;
}

int int_chunk_k(int a, int b) {
  const int64_t amax = (a == MMA_U8) ? 255 : 128, bmax = (b == MMA_U8) ? 255 : 128;
  const int64_t bound = int64_t(1) << int_sum_bits();
  int chunk = 1024;
  while (chunk > 64 && chunk * amax * bmax > bound) chunk /= 2;
  return chunk;
}

bool is_int8(int t) { return t == MMA_I8 || t == MMA_U8; }

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int* err = nullptr;
  cudaMemPool_t pool = nullptr;
  // co-resident clusters of the persistent kernels on this device, plus one (0: not yet
  // queried), per dense pair variant and per sparse kind (f16, FP8, exact i8)
  mutable std::atomic<int> pair_clusters[V_COUNT];
  mutable std::atomic<int> sparse_clusters[3];
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_inject{0};
std::atomic<unsigned long long> g_launches{0};

// The armed test hook if it is `mode` (then disarmed), else 0: mode 1 is taken by
// the next one-SM dense launch, mode 2 by the next CTA-pair launch (dense or sparse).
int take_inject(int mode) {
  int want = mode;
  return g_inject.compare_exchange_strong(want, 0) ? mode : 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int elem_bytes(int t) {
  switch (t) {
    case MMA_F16: case MMA_BF16: return 2;
    case MMA_E4M3: case MMA_E5M2: case MMA_I8: case MMA_U8: return 1;
    case MMA_F32: case MMA_I32: return 4;
    default: return 0;
  }
}
bool is_fp8(int t) { return t == MMA_E4M3 || t == MMA_E5M2; }

// Dense combinations: (F16,F16,F32), (BF16,BF16,F32), (F16,F16,F16), (BF16,BF16,BF16),
// {I8,U8} x {I8,U8} -> I32, FP8 x FP8 -> F32.
bool dense_types_ok(const mma_dtypes_t& t) {
  if (t.a == MMA_F16 && t.b == MMA_F16 && (t.acc == MMA_F32 || t.acc == MMA_F16)) return true;
  if (t.a == MMA_BF16 && t.b == MMA_BF16 && (t.acc == MMA_F32 || t.acc == MMA_BF16)) return true;
  if (is_int8(t.a) && is_int8(t.b) && t.acc == MMA_I32) return true;
  return is_fp8(t.a) && is_fp8(t.b) && t.acc == MMA_F32;
}
bool sparse_types_ok(const mma_dtypes_t& t) {
  if (t.a == MMA_F16 && t.b == MMA_F16 && t.acc == MMA_F32) return true;
  if (t.a == MMA_BF16 && t.b == MMA_BF16 && t.acc == MMA_F32) return true;
  if (is_int8(t.a) && is_int8(t.b) && t.acc == MMA_I32) return true;
  return is_fp8(t.a) && is_fp8(t.b) && t.acc == MMA_F32;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) overlap (empty ranges never do)
bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (na <= 0 || nb <= 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

mma_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MMA_OK : MMA_ERR_CUDA; }

// Per-device set-up, once, with that device current: SM count, the device
// error word's address, the scratch pool and the tensor-map encoder.
// The driver's tensor-map encoder, looked up once (g_mutex held).
bool load_encoder_locked() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return true;
}

mma_status_t device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MMA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    if (!load_encoder_locked()) return MMA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MMA_ERR_CUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_mma42_error) != cudaSuccess) return MMA_ERR_CUDA;
    s.err = static_cast<int*>(addr);
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&s.pool, &props) != cudaSuccess) return MMA_ERR_CUDA;
    uint64_t keep = ~0ull;   // keep freed scratch in the pool for the next call
    if (cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) return MMA_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return MMA_OK;
}

// 2-D (or 3-D) tiled tensor map over a row-major matrix.
bool encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
            const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  CUresult r = g_encode(map, dt, rank, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

CUtensorMapDataType raw_type(int bytes) {
  return bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                    : bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32;
}

// tcgen05 instruction descriptor (kind::f16 / kind::f8f6f4): f32 accumulator,
// A K-major, B MN-major (B is row-major K x N), M = bm, N = bn.
uint32_t make_idesc(int a_fmt, int b_fmt, int bn, bool sparse, int bm = 128) {
  uint32_t d = 0;
  d |= sparse ? (1u << 2) : 0u;               // sparsity flag (selector bits 0-1 stay 0)
  d |= 1u << 4;                                // D format: f32
  d |= static_cast<uint32_t>(a_fmt) << 7;      // A format
  d |= static_cast<uint32_t>(b_fmt) << 10;     // B format
  d |= 0u << 15;                               // A K-major
  d |= 1u << 16;                               // B MN-major
  d |= static_cast<uint32_t>(bn >> 3) << 17;   // N / 8
  d |= static_cast<uint32_t>(bm >> 4) << 24;   // M / 16 (256 for a CTA pair)
  return d;
}
// format codes: kind::f16 -> F16 0, BF16 1; kind::f8f6f4 -> E4M3 0, E5M2 1
int fmt_code(int t) { return (t == MMA_BF16 || t == MMA_E5M2) ? 1 : 0; }

// Choose the number of K splits: enough work units to fill the SMs, without
// paying more partial-sum traffic than the balance gains.
int plan_ksplit(int64_t tiles, int64_t kblocks, int num_sms, int64_t M, int64_t N, int64_t k_per_block) {
  if (tiles >= num_sms || kblocks < 8) return 1;
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= 16 && s <= kblocks / 4; ++s) {
    const int64_t units = tiles * s;
    const int64_t waves = (units + num_sms - 1) / num_sms;
    // main-loop time in k-block steps of one SM, plus partial traffic expressed in
    // the same unit (a 128 x 256 tile step moves ~48 KB; partials cost 8 B per output)
    const double mainloop = static_cast<double>(waves) * (static_cast<double>(kblocks) / s);
    const double traffic = (s > 1) ? (8.0 * s * M * N) / (48.0 * 1024.0 * num_sms) : 0.0;
    const double cost = mainloop + traffic;
    if (cost < best * 0.98) {
      best = cost;
      best_s = s;
    }
  }
  (void)k_per_block;
  return best_s;
}

struct Plan {
  Variant v;
  VariantInfo vi;
  GemmArgs args;
  int grid;
};

// int_chunk: the integer path's exact chunk length in K elements (0 otherwise).
mma_status_t run_gemm(const DeviceState& ds, Variant v, const void* A, int64_t a_cols, int a_bytes,
                      const void* B, int b_bytes, const void* C, void* D, int acc_bytes,
                      int64_t M, int64_t N, int64_t K, uint32_t idesc, int int_chunk, cudaStream_t stream) {
  Plan p;
  p.v = v;
  p.vi = variant_info(v);
  const VariantInfo& vi = p.vi;
  GemmArgs& a = p.args;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + vi.bm - 1) / vi.bm);
  a.tiles_n = static_cast<int>((N + vi.bn - 1) / vi.bn);
  a.kblocks = static_cast<int>((K + vi.bkl - 1) / vi.bkl);
  const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  const bool intacc = (v == V_DENSE_I8);
  a.ksplit = intacc ? 1 : plan_ksplit(tiles, a.kblocks, ds.num_sms, M, N, vi.bkl);
  if (a.ksplit > 1 && M * N * 4 >= (int64_t(1) << 39)) a.ksplit = 1;   // 3-D map stride limit
  a.chunk_kb = intacc ? std::max(1, int_chunk / vi.bkl) : 0;
  a.group_m = 16;
  a.idesc = idesc;
  a.err = ds.err;
  a.wait_ns = g_wait_ns.load();
  a.inject = (v == V_DENSE_F16 || v == V_DENSE_F8 || v == V_DENSE_F16_N128 || v == V_DENSE_F8_N128)
                 ? take_inject(1)
                 : 0;
  const int64_t units = tiles * a.ksplit;
  p.grid = static_cast<int>(std::min<int64_t>(units, ds.num_sms));

  TensorMaps m;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a_cols), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(a_cols) * a_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.bka), static_cast<uint32_t>(vi.bm)};
    if (!encode(&m.a, raw_type(a_bytes), 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * b_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.b_atom_n), static_cast<uint32_t>(vi.bkl)};
    if (!encode(&m.b, raw_type(b_bytes), 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  m.meta = m.a;   // unused by the dense kernel
  const CUtensorMapDataType acc_t = raw_type(acc_bytes);
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * acc_bytes};
    const uint32_t box[2] = {32u, 32u};
    if (!encode(&m.c, acc_t, 2, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
    if (!encode(&m.d, acc_t, 2, D, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  float* partial = nullptr;
  if (a.ksplit > 1) {
    const size_t bytes = static_cast<size_t>(a.ksplit) * M * N * 4;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&partial), bytes, ds.pool, stream) != cudaSuccess)
      return MMA_ERR_CUDA;
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M), static_cast<uint64_t>(a.ksplit)};
    const uint64_t str[2] = {static_cast<uint64_t>(N) * 4, static_cast<uint64_t>(M) * N * 4};
    const uint32_t box[3] = {32u, 32u, 1u};
    if (!encode(&m.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, partial, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
      cudaFreeAsync(partial, stream);
      return MMA_ERR_CUDA;
    }
  } else {
    m.p = m.d;
  }
  cudaError_t e = launch_gemm(v, m, a, p.grid, stream);
  if (e == cudaSuccess) g_launches.fetch_add(1);
  if (e == cudaSuccess && partial) {
    e = launch_splitk_reduce(partial, a.ksplit, C, D, M * N, 0, ds.num_sms, stream);
    if (e == cudaSuccess) g_launches.fetch_add(1);
  }
  if (partial) cudaFreeAsync(partial, stream);
  return from_cuda(e);
}

// `intacc`: the exact 8-bit integer variant; vals and B then hold the bf16-widened
// values, t is (BF16, BF16, I32) and int_chunk the exact chunk in logical K.
mma_status_t run_sparse(const DeviceState& ds, const void* vals, const uint8_t* idx, const void* B, const void* C,
                        void* D, int64_t M, int64_t N, int64_t K, mma_dtypes_t t, bool intacc, int int_chunk,
                        cudaStream_t stream, const int32_t* rowsum = nullptr, int beta = 0) {
  const bool f16 = !is_fp8(t.a);
  std::atomic<int>& cached = ds.sparse_clusters[intacc ? 2 : (f16 ? 0 : 1)];
  int c = cached.load();
  if (!c) {
    c = 1 + (intacc ? sparse_pair_i8_max_clusters()
                    : (f16 ? sparse_pair_f16_max_clusters() : sparse_pair_f8_max_clusters()));
    cached.store(c);
  }
  const int max_clusters = c - 1;
  if (max_clusters <= 0) return MMA_ERR_CUDA;
  const SparseInfo si = f16 ? sparse_pair_f16_info() : sparse_pair_f8_info();
  const int ea = elem_bytes(t.a), eb = elem_bytes(t.b);

  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + 2 * si.bm - 1) / (2 * si.bm));   // 256-row blocks of a CTA pair
  a.tiles_n = static_cast<int>((N + si.bn - 1) / si.bn);
  a.kblocks = static_cast<int>((K + si.bkl - 1) / si.bkl);   // an FP8 K of 128 mod 256 ends on half a stage
  a.ksplit = 1;
  a.chunk_kb = intacc ? std::max(1, int_chunk / si.bkl) : 0;
  a.c = C;
  a.rowsum = rowsum;
  a.beta = beta;
  a.group_m = 8;
  a.idesc = make_idesc(fmt_code(t.a), fmt_code(t.b), si.bn, true, 2 * si.bm);
  a.err = ds.err;
  a.wait_ns = g_wait_ns.load();
  a.inject = take_inject(2);
  const int64_t units = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  const int grid = static_cast<int>(std::min<int64_t>(units, max_clusters)) * 2;

  // the index in the tensor cores' layout (pool scratch, 8 bytes per row per 64
  // logical K, over whole stages and whole 256-row blocks, which the kernel's index
  // writers read without bounds checks)
  const int64_t slots = static_cast<int64_t>(a.kblocks) * si.meta_slots;
  const int64_t rows = static_cast<int64_t>(a.tiles_m) * 2 * si.bm;
  void* native = nullptr;
  if (cudaMallocFromPoolAsync(&native, static_cast<size_t>(slots * rows * 8), ds.pool, stream) != cudaSuccess)
    return MMA_ERR_CUDA;
  cudaError_t e = launch_meta_native(idx, native, M, K, f16, rows, slots, ds.num_sms, stream);
  a.meta = native;
  a.meta_rows = rows;
  if (e == cudaSuccess) g_launches.fetch_add(1);

  TensorMaps m;
  bool ok = e == cudaSuccess;
  if (ok) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(K / 2) * ea};
    const uint32_t box[2] = {static_cast<uint32_t>(si.bka), static_cast<uint32_t>(si.bm)};
    ok = encode(&m.a, raw_type(ea), 2, vals, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (ok) {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * eb};
    const uint32_t box[2] = {static_cast<uint32_t>(si.b_atom_n), static_cast<uint32_t>(si.b_rows_per_cta)};
    if (si.b_chunks == 2 && N % si.b_atom_n == 0) {
      // B as (b_atom_n columns, K rows, N / b_atom_n chunks): the strides need not grow
      // with the dimension, and one box brings both of a stage's 64-column chunks
      const uint64_t d3[3] = {static_cast<uint64_t>(si.b_atom_n), static_cast<uint64_t>(K),
                              static_cast<uint64_t>(N / si.b_atom_n)};
      const uint64_t s3[2] = {static_cast<uint64_t>(N) * eb, static_cast<uint64_t>(si.b_atom_n) * eb};
      const uint32_t b3[3] = {static_cast<uint32_t>(si.b_atom_n), static_cast<uint32_t>(si.b_rows_per_cta), 2u};
      ok = encode(&m.b, raw_type(eb), 3, B, d3, s3, b3, CU_TENSOR_MAP_SWIZZLE_128B);
      a.b_chunks_3d = 1;
    } else {
      ok = encode(&m.b, raw_type(eb), 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
  }
  if (ok) {
    // 32 rows x epi_cols f32 boxes: 128-byte rows 128-byte swizzled, 64-byte rows 64-byte
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(si.epi_cols), 32u};
    const CUtensorMapSwizzle swz = si.epi_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    ok = encode(&m.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, str, box, swz) &&
         encode(&m.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, str, box, swz);
  }
  m.p = m.d;
  if (ok) {
    e = intacc ? sparse_pair_i8_launch(m, a, grid, stream)
               : (f16 ? sparse_pair_f16_launch(m, a, grid, stream) : sparse_pair_f8_launch(m, a, grid, stream));
    if (e == cudaSuccess) g_launches.fetch_add(1);
  }
  cudaFreeAsync(native, stream);
  if (!ok) return MMA_ERR_CUDA;
  return from_cuda(e);
}

// Short K: the one-CTA-per-block kernel with all of a block's operands in flight at
// once (gemm_small.cu), when K fits its shared memory and the blocks fit one wave.
// MMA42_DENSE_KERNEL=small forces it whenever K fits; =single or =pair keep it out.
bool use_small(const DeviceState& ds, int64_t M, int64_t N, int64_t K, bool f8) {
  const SmallInfo si = small_info(f8, false);
  if (K > static_cast<int64_t>(si.kb_max) * si.bk) return false;
  if (const char* env = std::getenv("MMA42_DENSE_KERNEL")) {
    if (std::strcmp(env, "small") == 0) return true;
    if (std::strcmp(env, "single") == 0 || std::strcmp(env, "pair") == 0) return false;
  }
  const int64_t blocks = ((M + si.bm - 1) / si.bm) * ((N + si.bn - 1) / si.bn);
  return blocks <= ds.num_sms;
}

// Block width of the short-K kernel: 16-bit operands take 64-column blocks while
// those still give at most one block per SM (each SM then loads and stores half as
// much), otherwise 128.  MMA42_SMALL_BN=64|128 overrides the choice (tests).
bool small_narrow(const DeviceState& ds, int64_t M, int64_t N, bool f8) {
  if (f8) return false;
  if (const char* env = std::getenv("MMA42_SMALL_BN")) {
    if (std::strcmp(env, "64") == 0) return true;
    if (std::strcmp(env, "128") == 0) return false;
  }
  return ((M + 127) / 128) * ((N + 63) / 64) <= ds.num_sms;
}

mma_status_t run_small(const DeviceState& ds, bool f8, const void* A, int a_bytes, const void* B, int b_bytes,
                       const void* C, void* D, int64_t M, int64_t N, int64_t K, int a_fmt, int b_fmt,
                       cudaStream_t stream) {
  const SmallInfo si = small_info(f8, small_narrow(ds, M, N, f8));
  const uint32_t idesc = make_idesc(a_fmt, b_fmt, si.bn, false, si.bm);
  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + si.bm - 1) / si.bm);
  a.tiles_n = static_cast<int>((N + si.bn - 1) / si.bn);
  a.kblocks = static_cast<int>((K + si.bk - 1) / si.bk);
  a.ksplit = 1;
  a.group_m = 1;
  a.idesc = idesc;
  a.err = ds.err;
  a.wait_ns = g_wait_ns.load();
  a.inject = take_inject(3);
  TensorMaps m;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(K) * a_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(si.bk), static_cast<uint32_t>(si.bm)};
    if (!encode(&m.a, raw_type(a_bytes), 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * b_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(si.b_atom_n), static_cast<uint32_t>(si.bk)};
    if (!encode(&m.b, raw_type(b_bytes), 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * 4};
    const uint32_t box[2] = {32u, 32u};
    if (!encode(&m.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&m.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MMA_ERR_CUDA;
  }
  m.meta = m.a;
  m.p = m.d;
  const cudaError_t e = launch_small(f8, si.bn, m, a, stream);
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

// The CTA-pair kernel (256 x 256 blocks) when there are enough blocks to give
// every SM pair work, or when K is long enough that one wave of K slices (of at
// least kMinSliceSteps k-steps) fills most pairs; otherwise the one-SM kernel.
// `ksteps` is the number of k-steps of K; `split_ok` is false for the integer
// path, which does not split K in the pair kernel.
// MMA42_DENSE_KERNEL=single|pair overrides the choice (benchmarking and tests).
constexpr int kMinSliceSteps = 8;
bool use_pair(const DeviceState& ds, int64_t M, int64_t N, int64_t ksteps, bool split_ok) {
  if (const char* env = std::getenv("MMA42_DENSE_KERNEL")) {
    if (std::strcmp(env, "single") == 0) return false;
    if (std::strcmp(env, "pair") == 0) return true;
  }
  const int64_t blocks = ((M + 255) / 256) * ((N + 255) / 256);
  const int64_t pairs = ds.num_sms / 2;
  if (blocks >= pairs) return true;
  if (!split_ok || blocks == 0) return false;
  // the one wave of (block, slice) units that the pair kernel would run must keep
  // at least three quarters of the SM pairs busy
  const int64_t slices = std::min<int64_t>(pairs / blocks, std::min<int64_t>(64, ksteps / kMinSliceSteps));
  return 4 * blocks * slices >= 3 * pairs;
}

// K slices for the pair kernel: as many as fit in one wave of (block, slice)
// units over the SM pairs, each slice at least kMinSliceSteps k-steps long.  On
// the 1024 x 1024 x 65536 bf16 shape (16 blocks, 76 pairs) one wave of 4 slices
// measured 92.5 us, against 94-134 us for 8 to 38 slices in two to seven waves,
// where per-unit partial stores and pipeline fills outweigh the fuller last wave.
// MMA42_KSPLIT=n overrides (benchmarking and tests).
int plan_ksplit_pair(int64_t blocks, int64_t ksteps, int clusters) {
  if (const char* env = std::getenv("MMA42_KSPLIT")) {
    const int s = std::atoi(env);
    if (s >= 1) return static_cast<int>(std::min<int64_t>(s, std::max<int64_t>(1, ksteps)));
  }
  if (blocks <= 0 || blocks >= clusters) return 1;
  const int64_t s = std::min<int64_t>(clusters / blocks, std::min<int64_t>(64, ksteps / kMinSliceSteps));
  return static_cast<int>(std::max<int64_t>(1, s));
}

// Tail split for the pair kernel when the blocks take more than one round of the
// SM pairs: the T = blocks % pairs blocks of the last round are cut into s K
// slices (s = pairs / T, at most 4, each slice at least kMinSliceSteps k-steps)
// when that round would otherwise leave more than half of the pairs idle.  The
// last round then takes about 1/s of a block's time; the partials of those blocks
// (s x T x 256 KB) and one small reduction are the price.  0: no tail split.
// MMA42_TAIL_SPLIT=0 turns it off; =n (n >= 2) forces n slices, with every block
// a tail block when there are fewer blocks than pairs (tests).
int plan_tail_split(int64_t blocks, int64_t ksteps, int clusters, int64_t* tail) {
  *tail = 0;
  if (blocks <= 0) return 0;
  if (const char* env = std::getenv("MMA42_TAIL_SPLIT")) {
    const int s = std::atoi(env);
    if (s <= 1) return 0;
    const int64_t t = blocks < clusters ? blocks : blocks % clusters;
    if (t == 0) return 0;
    *tail = t;
    return static_cast<int>(std::min<int64_t>(s, std::max<int64_t>(1, ksteps)));
  }
  if (blocks <= clusters) return 0;
  const int64_t t = blocks % clusters;
  if (t == 0 || 2 * t > clusters) return 0;
  const int64_t s = std::min<int64_t>(clusters / t, std::min<int64_t>(4, ksteps / kMinSliceSteps));
  if (s < 2) return 0;
  *tail = t;
  return static_cast<int>(s);
}

// clamp_steps (integer path only): saturate D to the i32 range, with K cut into
// slices of at most clamp_steps k-steps whose product sums fit i32 (0: wrap).
mma_status_t run_pair(const DeviceState& ds, Variant v, const void* A, int a_bytes, const void* B, int b_bytes,
                      const void* C, void* D, int acc_bytes, int64_t M, int64_t N, int64_t K, int a_fmt, int b_fmt,
                      int int_chunk, cudaStream_t stream, int clamp_steps = 0,
                      const int32_t* rowsum = nullptr, const int32_t* colsum = nullptr, int alpha = 0,
                      int beta = 0) {
  int c = ds.pair_clusters[v].load();
  if (!c) {
    c = 1 + pair_variant_max_clusters(v);
    ds.pair_clusters[v].store(c);
  }
  const int max_clusters = c - 1;
  if (max_clusters <= 0) return MMA_ERR_CUDA;
  const VariantInfo vi = pair_variant_info(v);
  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + 2 * vi.bm - 1) / (2 * vi.bm));
  a.tiles_n = static_cast<int>((N + vi.bn - 1) / vi.bn);
  a.kblocks = static_cast<int>((K + vi.bkl - 1) / vi.bkl);
  const int64_t blocks = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  int64_t tail = 0;
  const int tail_split = clamp_steps == 0 ? plan_tail_split(blocks, a.kblocks, max_clusters, &tail) : 0;
  if (v == V_PAIR_I8)
    a.ksplit = clamp_steps > 0 ? (a.kblocks + clamp_steps - 1) / clamp_steps : 1;
  else
    a.ksplit = tail_split > 1 ? 1 : plan_ksplit_pair(blocks, a.kblocks, max_clusters);
  if (a.ksplit > 1 && M * N * 4 >= (int64_t(1) << 39)) {   // 3-D map stride limit
    if (clamp_steps > 0) return MMA_ERR_SHAPE;
    a.ksplit = 1;
  }
  if (tail_split > 1 && a.ksplit == 1) {
    a.tail_split = tail_split;
    a.tail_from = static_cast<int>(blocks - tail);
  }
  a.clamp = clamp_steps > 0 ? 1 : 0;
  a.rowsum = rowsum;
  a.colsum = colsum;
  a.alpha = alpha;
  a.beta = beta;
  a.chunk_kb = (v == V_PAIR_I8) ? std::max(1, int_chunk / vi.bkl) : 0;
  a.c = C;
  a.group_m = 8;
  a.idesc = make_idesc(a_fmt, b_fmt, vi.bn, false, 2 * vi.bm);
  a.err = ds.err;
  a.wait_ns = g_wait_ns.load();
  a.inject = take_inject(2);
  const int64_t units = a.tail_split > 1 ? a.tail_from + tail * a.tail_split : blocks * a.ksplit;
  const int grid = static_cast<int>(std::min<int64_t>(units, max_clusters)) * 2;

  TensorMaps m;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(K) * a_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.bka), static_cast<uint32_t>(vi.bm)};
    if (!encode(&m.a, raw_type(a_bytes), 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * b_bytes};
    const uint32_t box[2] = {static_cast<uint32_t>(vi.b_atom_n), static_cast<uint32_t>(vi.bkl)};
    if (!encode(&m.b, raw_type(b_bytes), 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  {
    const CUtensorMapDataType acc_t = raw_type(acc_bytes);
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t str[1] = {static_cast<uint64_t>(N) * acc_bytes};
    const uint32_t box[2] = {128u / static_cast<uint32_t>(acc_bytes), 32u};   // 128-byte rows: 32 f32, 64 halves
    if (!encode(&m.c, acc_t, 2, C, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
    if (!encode(&m.d, acc_t, 2, D, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MMA_ERR_CUDA;
  }
  m.meta = m.a;
  m.p = m.d;
  float* partial = nullptr;
  const int tile_rows = 2 * vi.bm, tile_cols = vi.bn;
  if (a.tail_split > 1) {   // compact partials of the tail blocks: tail_split x (tail * 256) x 256
    const size_t bytes = static_cast<size_t>(a.tail_split) * tail * tile_rows * tile_cols * 4;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&partial), bytes, ds.pool, stream) != cudaSuccess)
      return MMA_ERR_CUDA;
    const uint64_t dims[3] = {static_cast<uint64_t>(tile_cols), static_cast<uint64_t>(tail * tile_rows),
                              static_cast<uint64_t>(a.tail_split)};
    const uint64_t str[2] = {static_cast<uint64_t>(tile_cols) * 4,
                             static_cast<uint64_t>(tail) * tile_rows * tile_cols * 4};
    const uint32_t box[3] = {32u, 32u, 1u};
    if (!encode(&m.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, partial, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
      cudaFreeAsync(partial, stream);
      return MMA_ERR_CUDA;
    }
  } else if (a.ksplit > 1) {   // ksplit x M x N f32 partials, summed in slice order by the reduction
    const size_t bytes = static_cast<size_t>(a.ksplit) * M * N * 4;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&partial), bytes, ds.pool, stream) != cudaSuccess)
      return MMA_ERR_CUDA;
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M), static_cast<uint64_t>(a.ksplit)};
    const uint64_t str[2] = {static_cast<uint64_t>(N) * 4, static_cast<uint64_t>(M) * N * 4};
    const uint32_t box[3] = {32u, 32u, 1u};
    if (!encode(&m.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, partial, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
      cudaFreeAsync(partial, stream);
      return MMA_ERR_CUDA;
    }
  }
  cudaError_t e = pair_variant_launch(v, m, a, grid, stream);
  if (e == cudaSuccess) g_launches.fetch_add(1);
  if (e == cudaSuccess && partial && a.tail_split > 1) {
    TailReduce r;
    r.P = partial;
    r.S = a.tail_split;
    r.T = static_cast<int>(tail);
    r.tile_rows = tile_rows;
    r.tile_cols = tile_cols;
    r.C = C;
    r.D = D;
    r.M = M;
    r.N = N;
    r.K = K;
    r.out = (v == V_PAIR_I8) ? 3 : (v == V_PAIR_F16_OUTH) ? 1 : (v == V_PAIR_BF16_OUTH) ? 2 : 0;
    r.rowsum = rowsum;
    r.colsum = colsum;
    r.alpha = alpha;
    r.beta = beta;
    e = launch_tail_reduce(r, a, ds.num_sms, stream);
    if (e == cudaSuccess) g_launches.fetch_add(1);
  } else if (e == cudaSuccess && partial) {
    if (v == V_PAIR_I8) {
      e = launch_splitk_reduce_i32(reinterpret_cast<const int32_t*>(partial), a.ksplit, static_cast<const int32_t*>(C),
                                   static_cast<int32_t*>(D), M * N, a.clamp != 0, rowsum, colsum, alpha, beta, K, N,
                                   ds.num_sms, stream);
    } else {
      const int out = (v == V_PAIR_F16_OUTH) ? 1 : (v == V_PAIR_BF16_OUTH) ? 2 : 0;
      e = launch_splitk_reduce(partial, a.ksplit, C, D, M * N, out, ds.num_sms, stream);
    }
    if (e == cudaSuccess) g_launches.fetch_add(1);
  }
  if (partial) cudaFreeAsync(partial, stream);
  return from_cuda(e);
}

// Shared checks of the dense and sparse GEMM entry points.
mma_status_t check_common(const void* A, int64_t a_row_bytes, int64_t a_total, const void* B, const void* C,
                          void* D, int64_t M, int64_t N, int64_t K, int eb, int eacc) {
  if (M < 0 || N < 0 || K < 0) return MMA_ERR_INVALID_ARG;
  const int64_t lim = int64_t(1) << 31;
  if (M >= lim || N >= lim || K >= lim) return MMA_ERR_SHAPE;
  if (M == 0 || N == 0) return MMA_OK;
  if (!C || !D || (K > 0 && (!A || !B))) return MMA_ERR_INVALID_ARG;
  if (!aligned16(C) || !aligned16(D) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return MMA_ERR_ALIGN;
  if ((N * eacc) % 16 != 0) return MMA_ERR_ALIGN;
  if (K > 0 && ((a_row_bytes % 16) != 0 || (N * eb) % 16 != 0)) return MMA_ERR_ALIGN;
  const int64_t cd = M * N * eacc;
  if (C != D && overlaps(C, cd, D, cd)) return MMA_ERR_INVALID_ARG;
  if (K > 0 && (overlaps(D, cd, A, a_total) || overlaps(D, cd, B, K * N * eb))) return MMA_ERR_INVALID_ARG;
  return MMA_OK;
}

}  // namespace

// sparse42_compress and sparse42_prune: the same checks and kernel, two rules.
namespace {

mma_status_t compress_or_prune(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K, mma_dtype_t a,
                               bool prune, int32_t* d_violations, void* stream) {
  const int e = (a == MMA_F16 || a == MMA_BF16) ? 2 : (a == MMA_E4M3 || a == MMA_E5M2 || is_int8(a)) ? 1 : 0;
  if (e == 0) return MMA_ERR_UNSUPPORTED;
  if (M < 0 || K < 0) return MMA_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || K % 32 != 0) return MMA_ERR_SHAPE;
  const int64_t na = M * K * e, nv = M * (K / 2) * e, ni = M * (K / 8);
  if (na > 0 && (!A || !vals || !idx)) return MMA_ERR_INVALID_ARG;
  if (na > 0 && (!aligned16(A) || !aligned16(vals) || !aligned16(idx))) return MMA_ERR_ALIGN;
  if (d_violations && (reinterpret_cast<uintptr_t>(d_violations) & 3u)) return MMA_ERR_ALIGN;
  if (overlaps(vals, nv, A, na) || overlaps(idx, ni, A, na) || overlaps(idx, ni, vals, nv) ||
      (d_violations && (overlaps(d_violations, 4, A, na) || overlaps(d_violations, 4, vals, nv) ||
                        overlaps(d_violations, 4, idx, ni))))
    return MMA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  const int zero_mask = (e == 2) ? 0x7fff : (is_int8(a) ? 0xff : 0x7f);
  const int mode = prune ? (a == MMA_I8 ? 2 : (a == MMA_U8 ? 3 : 1)) : 0;
  const cudaError_t ce = launch_compress42(A, vals, idx, M, K, e, zero_mask, mode, d_violations, ds->num_sms,
                                           static_cast<cudaStream_t>(stream));
  if (ce == cudaSuccess && M * K > 0) g_launches.fetch_add(1);
  return from_cuda(ce);
}

}  // namespace

extern "C" {

int32_t mma_abi_version(void) { return MMA42_ABI_VERSION; }

const char* mma_status_string(mma_status_t s) {
  switch (s) {
    case MMA_OK: return "MMA_OK";
    case MMA_ERR_INVALID_ARG: return "MMA_ERR_INVALID_ARG: null pointer, negative size or overlapping buffers";
    case MMA_ERR_UNSUPPORTED: return "MMA_ERR_UNSUPPORTED: type combination not provided";
    case MMA_ERR_SHAPE: return "MMA_ERR_SHAPE: size outside the supported range";
    case MMA_ERR_ALIGN: return "MMA_ERR_ALIGN: base pointer or row pitch not a multiple of 16 bytes";
    case MMA_ERR_NOT_SPARSE: return "MMA_ERR_NOT_SPARSE: a group of four holds more than two non-zeros";
    case MMA_ERR_TIMEOUT: return "MMA_ERR_TIMEOUT: a device-side pipeline wait ran past its limit";
    case MMA_ERR_CUDA: return "MMA_ERR_CUDA: the CUDA runtime reported an error";
    default: return "unknown mma_status_t";
  }
}

void mma_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : 1); }

void mma_debug_inject(int32_t mode) { g_inject.store(mode); }

uint64_t mma_launch_count(void) { return g_launches.load(); }

mma_status_t mma_legacy_mma_peak(int32_t kind, double* ops_per_s, void* stream) {
  if (kind < 0 || kind > 3 || !ops_per_s) return MMA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* sink = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&sink), legacy_peak_sink_words(ds->num_sms) * 4, ds->pool, s) !=
      cudaSuccess)
    return MMA_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  // a short launch to size the timed one at about 25 ms
  int64_t iters = 256;
  float ms = 0.f;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = launch_legacy_peak(kind, iters, sink, ds->num_sms, s);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && pass == 0)
      iters = std::max<int64_t>(256, std::min<int64_t>(int64_t(1) << 24, static_cast<int64_t>(iters * 25.0 / std::max(ms, 1e-3f))));
  }
  if (e == cudaSuccess) *ops_per_s = legacy_peak_ops(kind, iters, ds->num_sms) / (static_cast<double>(ms) * 1e-3);
  cudaFreeAsync(sink, s);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return from_cuda(e);
}

mma_status_t mma_tcgen05_peak(int32_t kind, double* ops_per_s, double* ops_per_clk_sm, void* stream) {
  if (kind < 0 || kind > 3 || !ops_per_s) return MMA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  const int clusters = tc_peak_max_clusters(kind);
  if (clusters <= 0) return MMA_ERR_CUDA;
  const bool f8 = (kind & 1) != 0, sparse = kind >= 2;
  // bf16 (kind::f16 format 1) or E4M3 (kind::f8f6f4 format 0), M = N = 256 per pair
  const uint32_t idesc = make_idesc(f8 ? 0 : 1, f8 ? 0 : 1, 256, sparse, 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* cycles = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&cycles), static_cast<size_t>(clusters) * 8, ds->pool, s) !=
      cudaSuccess)
    return MMA_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  // a short launch to size the timed one at about 25 ms
  int64_t iters = 64;
  float ms = 0.f;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) e = launch_tc_peak(kind, iters, idesc, g_wait_ns.load(), cycles, ds->err, clusters, s);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && pass == 0)
      iters = std::max<int64_t>(64, std::min<int64_t>(int64_t(1) << 26, static_cast<int64_t>(iters * 25.0 / std::max(ms, 1e-3f))));
  }
  std::vector<unsigned long long> cyc(static_cast<size_t>(clusters), 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(cyc.data(), cycles, cyc.size() * 8, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  const double per_cluster = tc_peak_ops_per_cluster_iter(kind) * static_cast<double>(iters);
  if (e == cudaSuccess) {
    *ops_per_s = per_cluster * clusters / (static_cast<double>(ms) * 1e-3);
    if (ops_per_clk_sm) {
      double mean = 0.0;
      for (unsigned long long c : cyc) mean += static_cast<double>(c);
      mean /= static_cast<double>(cyc.size());
      *ops_per_clk_sm = mean > 0.0 ? per_cluster / 2.0 / mean : 0.0;   // two SMs per cluster
    }
  }
  cudaFreeAsync(cycles, s);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return from_cuda(e);
}

mma_status_t mma_tma_feed_probe(int32_t nbox, const int32_t* box_rows, const int32_t* box_row_bytes, int32_t stages,
                                int32_t clusters, int64_t src_bytes, double* bytes_per_clk_sm, double* rows_per_clk_sm,
                                void* stream) {
  if (nbox < 1 || nbox > 4 || !box_rows || !box_row_bytes || !bytes_per_clk_sm || clusters < 0 || stages < 2)
    return MMA_ERR_INVALID_ARG;
  FeedProbe p = {};
  p.nbox = nbox;
  int off = 0, rows = 0;
  for (int b = 0; b < nbox; ++b) {
    const int r = box_rows[b], rb = box_row_bytes[b];
    if ((rb != 64 && rb != 128 && rb != 256) || r < 8 || r > 256 || r % 8 != 0 || (r * rb) % 1024 != 0)
      return MMA_ERR_INVALID_ARG;
    p.rows[b] = r;
    p.row_bytes[b] = rb;
    p.smem_off[b] = off;   // r * rb is a multiple of 1024: every box keeps the swizzle alignment
    off += r * rb;
    rows += r;
  }
  p.stages = stages;
  p.stage_bytes = off;
  const int pitch = feed_probe_row_pitch();
  const int64_t quarter = src_bytes / 4;
  if (src_bytes < 0 || quarter / pitch < 512 || quarter / pitch > (int64_t(1) << 30)) return MMA_ERR_SHAPE;
  p.height = static_cast<int>(quarter / pitch);
  const int smem = stages * off + 1024 + 256;
  if (smem > 232448) return MMA_ERR_SHAPE;
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  const int fit = feed_probe_max_clusters(smem);
  if (fit <= 0) return MMA_ERR_CUDA;
  const int n = clusters == 0 ? fit : std::min(clusters, fit);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* src = nullptr;
  unsigned long long* cycles = nullptr;
  if (cudaMallocFromPoolAsync(&src, static_cast<size_t>(src_bytes), ds->pool, s) != cudaSuccess) return MMA_ERR_CUDA;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&cycles), static_cast<size_t>(n) * 8, ds->pool, s) !=
      cudaSuccess) {
    cudaFreeAsync(src, s);
    return MMA_ERR_CUDA;
  }
  CUtensorMap maps[4];
  bool ok = true;
  for (int b = 0; b < 4 && ok; ++b) {
    const int bb = b < nbox ? b : 0;
    const uint64_t dims[2] = {static_cast<uint64_t>(pitch), static_cast<uint64_t>(p.height)};
    const uint64_t str[1] = {static_cast<uint64_t>(pitch)};
    const uint32_t box[2] = {static_cast<uint32_t>(p.row_bytes[bb]), static_cast<uint32_t>(p.rows[bb])};
    const CUtensorMapSwizzle swz = p.row_bytes[bb] == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : p.row_bytes[bb] == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                           : CU_TENSOR_MAP_SWIZZLE_NONE;
    ok = encode(&maps[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, static_cast<uint8_t*>(src) + bb * quarter, dims, str, box,
                swz);
  }
  cudaError_t e = ok ? cudaSuccess : cudaErrorInvalidValue;
  // a first launch warms L2 and sizes the timed one at about 10 ms
  p.iters = 1024;
  std::vector<unsigned long long> cyc(static_cast<size_t>(n));
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
    e = launch_feed_probe(p, maps, n, g_wait_ns.load(), ds->err, cycles, s);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (e == cudaSuccess) e = cudaMemcpyAsync(cyc.data(), cycles, cyc.size() * 8, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && pass == 0) {
      double mean = 0.0;
      for (unsigned long long c : cyc) mean += static_cast<double>(c);
      mean /= static_cast<double>(cyc.size());
      const double per_stage = mean / (p.iters - feed_probe_warm_stages());
      // about 2e7 cycles (10 ms at 2 GHz)
      p.iters = static_cast<int>(std::max(1024.0, std::min(1e6, 2e7 / std::max(per_stage, 1.0))));
    }
  }
  if (e == cudaSuccess) {
    double mean = 0.0;
    int counted = 0;
    for (unsigned long long c : cyc)
      if (c) {
        mean += static_cast<double>(c);
        ++counted;
      }
    if (counted == 0) {
      e = cudaErrorUnknown;
    } else {
      mean /= counted;
      const double stages_timed = p.iters - feed_probe_warm_stages();
      *bytes_per_clk_sm = p.stage_bytes * stages_timed / mean;   // each SM fills its own stage_bytes per stage
      if (rows_per_clk_sm) *rows_per_clk_sm = rows * stages_timed / mean;
    }
  }
  cudaFreeAsync(cycles, s);
  cudaFreeAsync(src, s);
  if (!ok) return MMA_ERR_CUDA;
  return from_cuda(e);
}

mma_status_t mma_gemm(const void* A, const void* B, const void* C, void* D, int64_t M, int64_t N, int64_t K,
                      mma_dtypes_t t, void* stream) {
  return mma_gemm_ex(A, B, C, D, M, N, K, t, 0u, stream);
}

mma_status_t mma_gemm_ex(const void* A, const void* B, const void* C, void* D, int64_t M, int64_t N, int64_t K,
                         mma_dtypes_t t, uint32_t flags, void* stream) {
  if (flags & ~static_cast<uint32_t>(MMA_FLAG_CLAMP)) return MMA_ERR_INVALID_ARG;
  const bool clamp = (flags & MMA_FLAG_CLAMP) != 0;
  if (!dense_types_ok(t)) return MMA_ERR_UNSUPPORTED;
  if (clamp && !is_int8(t.a)) return MMA_ERR_UNSUPPORTED;   // saturation is an integer-path option
  const int ea = elem_bytes(t.a), eb = elem_bytes(t.b), eacc = elem_bytes(t.acc);
  mma_status_t st = check_common(A, K * ea, M * K * ea, B, C, D, M, N, K, eb, eacc);
  if (st != MMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {   // D = C
    if (C == D) return MMA_OK;
    return from_cuda(cudaMemcpyAsync(D, C, static_cast<size_t>(M * N * eacc), cudaMemcpyDeviceToDevice, s));
  }
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != MMA_OK) return st;
  if (is_int8(t.a)) {
    // Exact widening to bf16 in pool scratch, then the bf16 path with i32 chunk sums.
    // An unsigned operand is shifted into the signed range (A = A' + alpha, B = B' +
    // beta, alpha / beta = 128 for unsigned operands), so every combination runs with
    // the signed x signed chunk length, and D gets beta * rowsum(A') + alpha *
    // colsum(B') + alpha * beta * K added by the epilogue.
    const int alpha = (t.a == MMA_U8) ? 128 : 0, beta = (t.b == MMA_U8) ? 128 : 0;
    void* scratch = nullptr;
    const size_t na = static_cast<size_t>(M * K), nb = static_cast<size_t>(K * N);
    const size_t abytes = (na * 2 + 255) & ~size_t(255), bbytes = (nb * 2 + 255) & ~size_t(255);
    const size_t rbytes = (static_cast<size_t>(M) * 4 + 255) & ~size_t(255), cbytes = static_cast<size_t>(N) * 4;
    if (cudaMallocFromPoolAsync(&scratch, abytes + bbytes + rbytes + cbytes, ds->pool, s) != cudaSuccess)
      return MMA_ERR_CUDA;
    uint8_t* base = static_cast<uint8_t*>(scratch);
    uint16_t* a16 = reinterpret_cast<uint16_t*>(base);
    uint16_t* b16 = reinterpret_cast<uint16_t*>(base + abytes);
    int32_t* rsum = reinterpret_cast<int32_t*>(base + abytes + bbytes);
    int32_t* csum = reinterpret_cast<int32_t*>(base + abytes + bbytes + rbytes);
    cudaError_t e = launch_i8_to_bf16(A, t.a == MMA_U8, alpha, a16, static_cast<int64_t>(na), B, t.b == MMA_U8, beta,
                                      b16, static_cast<int64_t>(nb), ds->num_sms, s);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (e == cudaSuccess && beta != 0) {
      e = launch_int8_rowsum(A, t.a == MMA_U8, alpha, M, K, rsum, ds->num_sms, s);
      if (e == cudaSuccess) g_launches.fetch_add(1);
    }
    if (e == cudaSuccess && alpha != 0) {
      e = launch_int8_colsum(B, t.b == MMA_U8, beta, K, N, csum, ds->num_sms, s);
      if (e == cudaSuccess) g_launches.fetch_add(1);
    }
    if (e == cudaSuccess) {
      const int chunk = int_chunk_k(MMA_I8, MMA_I8);   // operands are signed after the shift
      // clamp: K slices short enough that each slice's product sum fits i32, C added
      // and saturated in 64 bits (the pair kernel at any shape)
      const int clamp_steps = clamp ? static_cast<int>(std::max<int64_t>(1, (INT32_MAX / (128 * 128)) / 64)) : 0;
      const bool shifted = alpha != 0 || beta != 0;
      st = (clamp || shifted || use_pair(*ds, M, N, (K + 63) / 64, false))
               ? run_pair(*ds, V_PAIR_I8, a16, 2, b16, 2, C, D, 4, M, N, K, 1, 1, chunk, s, clamp_steps,
                          beta != 0 ? rsum : nullptr, alpha != 0 ? csum : nullptr, alpha, beta)
               : run_gemm(*ds, V_DENSE_I8, a16, K, 2, b16, 2, C, D, 4, M, N, K, make_idesc(1, 1, 128, false),
                          chunk, s);
    } else {
      st = MMA_ERR_CUDA;
    }
    cudaFreeAsync(scratch, s);
    return st;
  }
  if (t.acc == MMA_F16 || t.acc == MMA_BF16)   // half-precision C and D: the pair kernel at any shape
    return run_pair(*ds, t.acc == MMA_F16 ? V_PAIR_F16_OUTH : V_PAIR_BF16_OUTH, A, ea, B, eb, C, D, 2, M, N, K,
                    fmt_code(t.a), fmt_code(t.b), 0, s);
  const bool f8 = is_fp8(t.a);
  if (use_small(*ds, M, N, K, f8))
    return run_small(*ds, f8, A, ea, B, eb, C, D, M, N, K, fmt_code(t.a), fmt_code(t.b), s);
  if (use_pair(*ds, M, N, (K + (f8 ? 127 : 63)) / (f8 ? 128 : 64), true))
    return run_pair(*ds, f8 ? V_PAIR_F8 : V_PAIR_F16, A, ea, B, eb, C, D, 4, M, N, K, fmt_code(t.a),
                    fmt_code(t.b), 0, s);
  // outputs at most 128 wide take 128-column blocks: no MMA or B staging on columns past N
  const Variant v = N <= 128 ? (f8 ? V_DENSE_F8_N128 : V_DENSE_F16_N128) : (f8 ? V_DENSE_F8 : V_DENSE_F16);
  return run_gemm(*ds, v, A, K, ea, B, eb, C, D, 4, M, N, K,
                  make_idesc(fmt_code(t.a), fmt_code(t.b), variant_info(v).bn, false), 0, s);
}

mma_status_t sparse42_gemm(const void* vals, const uint8_t* idx, const void* B, const void* C, void* D, int64_t M,
                           int64_t N, int64_t K, mma_dtypes_t t, void* stream) {
  if (!sparse_types_ok(t)) return MMA_ERR_UNSUPPORTED;
  const int ea = elem_bytes(t.a), eb = elem_bytes(t.b), eacc = elem_bytes(t.acc);
  mma_status_t st = check_common(vals, (K / 2) * ea, M * (K / 2) * ea, B, C, D, M, N, K, eb, eacc);
  if (st != MMA_OK || M == 0 || N == 0) return st;
  if (K % 128 != 0) return MMA_ERR_SHAPE;
  if (K > 0) {
    if (!idx) return MMA_ERR_INVALID_ARG;
    if (!aligned16(idx)) return MMA_ERR_ALIGN;
    if (overlaps(D, M * N * eacc, idx, M * (K / 8))) return MMA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    if (C == D) return MMA_OK;
    return from_cuda(cudaMemcpyAsync(D, C, static_cast<size_t>(M * N * eacc), cudaMemcpyDeviceToDevice, s));
  }
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != MMA_OK) return st;
  if (is_int8(t.a)) {
    // Exact widening of the kept values and of B to bf16 in pool scratch, then the
    // sparse bf16 kernel with i32 chunk sums.  An unsigned B is shifted into the
    // signed range (B = B' + beta, beta = 128), which lengthens the exact chunks; D
    // then gets beta * rowsum(A)[i], and the row sums of A are those of its kept
    // values.  A keeps its values: a shift would break the zeros of the 4:2 pattern.
    const int beta = (t.b == MMA_U8) ? 128 : 0;
    void* scratch = nullptr;
    const size_t nv = static_cast<size_t>(M * (K / 2)), nb = static_cast<size_t>(K * N);
    const size_t vbytes = (nv * 2 + 255) & ~size_t(255), bbytes = (nb * 2 + 255) & ~size_t(255);
    const size_t rbytes = static_cast<size_t>(M) * 4;
    if (cudaMallocFromPoolAsync(&scratch, vbytes + bbytes + rbytes, ds->pool, s) != cudaSuccess) return MMA_ERR_CUDA;
    uint16_t* v16 = static_cast<uint16_t*>(scratch);
    uint16_t* b16 = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(scratch) + vbytes);
    int32_t* rsum = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + vbytes + bbytes);
    cudaError_t e = launch_i8_to_bf16(vals, t.a == MMA_U8, 0, v16, static_cast<int64_t>(nv), B, t.b == MMA_U8, beta,
                                      b16, static_cast<int64_t>(nb), ds->num_sms, s);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    if (e == cudaSuccess && beta != 0) {
      e = launch_int8_rowsum(vals, t.a == MMA_U8, 0, M, K / 2, rsum, ds->num_sms, s);
      if (e == cudaSuccess) g_launches.fetch_add(1);
    }
    if (e == cudaSuccess) {
      const mma_dtypes_t t16 = {MMA_BF16, MMA_BF16, MMA_I32};
      // a chunk of L logical K meets L/2 products per output
      const int chunk = 2 * int_chunk_k(t.a, beta != 0 ? MMA_I8 : t.b);
      st = run_sparse(*ds, v16, idx, b16, C, D, M, N, K, t16, true, chunk, s, beta != 0 ? rsum : nullptr, beta);
    } else {
      st = MMA_ERR_CUDA;
    }
    cudaFreeAsync(scratch, s);
    return st;
  }
  return run_sparse(*ds, vals, idx, B, C, D, M, N, K, t, false, 0, s);
}

mma_status_t sparse42_compress(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K, mma_dtype_t a,
                               int32_t* d_violations, void* stream) {
  return compress_or_prune(A, vals, idx, M, K, a, false, d_violations, stream);
}

mma_status_t sparse42_prune(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K, mma_dtype_t a,
                            int32_t* d_dropped, void* stream) {
  return compress_or_prune(A, vals, idx, M, K, a, true, d_dropped, stream);
}

mma_status_t sparse42_quantize_prune(const float* A, void* vals, uint8_t* idx, int64_t M, int64_t K, mma_dtype_t t,
                                     int32_t* d_dropped, void* stream) {
  const int kind = (t == MMA_F16) ? 0 : (t == MMA_BF16) ? 1 : (t == MMA_E4M3) ? 2 : (t == MMA_E5M2) ? 3 : -1;
  if (kind < 0) return MMA_ERR_UNSUPPORTED;
  if (M < 0 || K < 0) return MMA_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || K % 32 != 0) return MMA_ERR_SHAPE;
  const int e = elem_bytes(t);
  const int64_t na = M * K * 4, nv = M * (K / 2) * e, ni = M * (K / 8);
  if (na > 0 && (!A || !vals || !idx)) return MMA_ERR_INVALID_ARG;
  if (na > 0 && (!aligned16(A) || !aligned16(vals) || !aligned16(idx))) return MMA_ERR_ALIGN;
  if (d_dropped && (reinterpret_cast<uintptr_t>(d_dropped) & 3u)) return MMA_ERR_ALIGN;
  if (overlaps(vals, nv, A, na) || overlaps(idx, ni, A, na) || overlaps(idx, ni, vals, nv) ||
      (d_dropped && (overlaps(d_dropped, 4, A, na) || overlaps(d_dropped, 4, vals, nv) ||
                     overlaps(d_dropped, 4, idx, ni))))
    return MMA_ERR_INVALID_ARG;
  if (na == 0 && !d_dropped) return MMA_OK;   // nothing to do and no count to clear
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  const cudaError_t ce = launch_quantize_prune(A, vals, idx, M, K, kind, d_dropped, ds->num_sms,
                                               static_cast<cudaStream_t>(stream));
  if (ce == cudaSuccess && M * K > 0) g_launches.fetch_add(1);
  return from_cuda(ce);
}

mma_status_t mma_quantize(const float* x, void* y, int64_t n, mma_dtype_t t, void* stream) {
  const int kind = (t == MMA_F16) ? 0 : (t == MMA_BF16) ? 1 : (t == MMA_E4M3) ? 2 : (t == MMA_E5M2) ? 3 : -1;
  if (kind < 0) return MMA_ERR_UNSUPPORTED;
  if (n < 0) return MMA_ERR_INVALID_ARG;
  if (n == 0) return MMA_OK;
  if (!x || !y) return MMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return MMA_ERR_ALIGN;
  if (overlaps(x, n * 4, y, n * elem_bytes(t))) return MMA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  mma_status_t st = device_state(&ds);
  if (st != MMA_OK) return st;
  const cudaError_t e = launch_quantize(x, y, n, kind, ds->num_sms, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

mma_status_t mma_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MMA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mma42_error, sizeof(int)) != cudaSuccess) return MMA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_mma42_error, &zero, sizeof(int)) != cudaSuccess) return MMA_ERR_CUDA;
    return MMA_ERR_TIMEOUT;
  }
  return MMA_OK;
}

}  // extern "C"

// Host helpers shared with the allocation-free entry point (noalloc.cu); thin
// wrappers over the functions above, declared in host_util.h.
namespace mma42 {
namespace host {

bool encode_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  return encode(map, dt, rank, base, dims, strides_bytes, box, swz);
}
CUtensorMapDataType map_type(int bytes) { return raw_type(bytes); }
uint32_t instr_desc(int a_fmt, int b_fmt, int bn, bool sparse) { return make_idesc(a_fmt, b_fmt, bn, sparse); }
int format_code(int t) { return fmt_code(t); }
int elem_size(int t) { return elem_bytes(t); }
bool fp8_type(int t) { return is_fp8(t); }
mma_status_t check_gemm_args(const void* A, int64_t a_row_bytes, int64_t a_total, const void* B, const void* C,
                             void* D, int64_t M, int64_t N, int64_t K, int eb, int eacc) {
  return check_common(A, a_row_bytes, a_total, B, C, D, M, N, K, eb, eacc);
}
bool ensure_encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  return load_encoder_locked();
}
int* error_word() {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_mma42_error) != cudaSuccess) return nullptr;
  return static_cast<int*>(addr);
}
unsigned long long wait_limit_ns() { return g_wait_ns.load(); }
void count_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

}  // namespace host
}  // namespace mma42
