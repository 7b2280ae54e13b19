// gemm_small.cu -- D = A*B + C for short K: one CTA per 128 x 128 (or, for 16-bit
// operands and few blocks, 128 x 64) output block, everything in flight at once.
//
// The operation is the matrix multiply-accumulate of "CDNA dense MFMA builtins",
// section "Naming convention", over whole matrices, for K up to 4 k-blocks (256 for
// f16 / bf16, 512 for FP8), where all of a block's A, B and C fit in shared memory.
// Such a problem is latency-bound: the persistent kernels spend its time on their
// scheduler, their ring's handshakes and a C load that waits for the accumulator.
// Here one thread issues every A and B box (one barrier per k-block, so the MMAs of
// a k-block start as it lands), each warp issues the C boxes of its own 32 rows at
// the same time, one thread issues the MMAs (M = 128, N = BN) and commits once,
// and each warp then adds C to its TMEM lanes in the C staging buffer, box by box,
// and stores each 32 x 32 box of D by TMA as soon as it is added.  No ring, no
// persistent loop, BN TMEM columns.
//
// One SM takes in a k-block (A and B boxes) about every 540 SM clocks from L2, and
// the block's loads, MMAs and epilogue run one after the other, so with few blocks
// the 64-column form (16-bit operands) halves each SM's share: A is read by both
// CTAs of a 128-row band, B, C and D are split between them.
//
// Every wait is bounded: a wait that runs out raises the device error word and the
// abort flag; the MMA thread still commits, so TMEM is released only after the
// MMAs it issued have completed, D is not stored, and the loads already issued land
// before the block exits.
#include <cstdint>

#include "gemm_kernel.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace mma42 {

namespace {

template <int KIND, int BN_>
struct SmallCfg {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;                          // 128, or 64 for 16-bit operands
  static constexpr int ELEM = (KIND == KIND_F16) ? 2 : 1;
  static constexpr int BK = 128 / ELEM;                   // K per box: one 128-byte row of A
  static constexpr int KB_MAX = 4;                        // k-blocks held at once
  static constexpr int UMMA_K = (KIND == KIND_F16) ? 16 : 32;
  static constexpr int MMAS = BK / UMMA_K;                // 4
  static constexpr int A_BYTES = BM * 128;                // 16 KB per k-block
  static constexpr int B_ATOM_N = 128 / ELEM;
  static constexpr int B_CHUNKS = BN / B_ATOM_N;          // 2 (16-bit, BN 128), 1 (FP8, or BN 64)
  static constexpr int B_CHUNK_BYTES = BK * 128;
  static constexpr int B_BYTES = B_CHUNKS * B_CHUNK_BYTES;   // 16 KB per k-block (8 KB at BN 64)
  static constexpr int B_KSTEP = UMMA_K * 128;
  static constexpr int KB_BYTES = A_BYTES + B_BYTES;
  static constexpr int C_BOX_BYTES = 32 * 32 * 4;         // 32 rows x 32 f32
  static constexpr int NB = BN / 32;                      // C / D boxes per warp
  static constexpr int C_BYTES = (BM / 32) * NB * C_BOX_BYTES;   // 64 KB (32 KB at BN 64)
  static constexpr int MISC_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + KB_MAX * KB_BYTES + C_BYTES + MISC_BYTES;
  static constexpr int TMEM_COLS = BN;
  static constexpr int THREADS = 128;
  static_assert(KB_BYTES % 1024 == 0, "k-blocks keep 1024-byte alignment");
  static_assert(B_CHUNKS >= 1 && BN % B_ATOM_N == 0, "B tile is whole 128-byte chunks");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Bounded wait without a role loop around it: false once the limit has passed (the
// error word and the abort flag are raised) or another thread has aborted.
__device__ __forceinline__ bool small_wait(uint32_t bar, uint32_t parity, const GemmArgs& a,
                                           volatile int* abort_flag) {
  return wait_phase(bar, parity, a, abort_flag);
}

template <int KIND, int BN>
__global__ void __launch_bounds__(SmallCfg<KIND, BN>::THREADS, 1)
    gemm_small_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                      const GemmArgs args) {
  using Cfg = SmallCfg<KIND, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t cbase = sbase + Cfg::KB_MAX * Cfg::KB_BYTES;
  uint8_t* misc = smem + Cfg::KB_MAX * Cfg::KB_BYTES + Cfg::C_BYTES;
  const uint32_t bar0 = smem_addr(misc);
  // barrier slots: kb[KB_MAX], acc, c[4]
  auto kb_bar = [&](int kb) { return bar0 + 8u * kb; };
  const uint32_t acc_bar = bar0 + 8u * Cfg::KB_MAX;
  auto c_bar = [&](int w) { return bar0 + 8u * (Cfg::KB_MAX + 1 + w); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (Cfg::KB_MAX + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * (Cfg::KB_MAX + 5) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = blockIdx.x % args.tiles_m;
  const int nt = blockIdx.x / args.tiles_m;
  const int m0 = mt * Cfg::BM, n0 = nt * Cfg::BN;
  const int kbs = args.kblocks;   // 1 .. KB_MAX, checked on the host

  if (threadIdx.x == 0) {
    for (int kb = 0; kb < Cfg::KB_MAX; ++kb) mbar_init(kb_bar(kb), 1);
    mbar_init(acc_bar, 1);
    for (int w = 0; w < 4; ++w) mbar_init(c_bar(w), 1);
    *abort_flag = 0;
    mbar_fence_init();
    // launched with programmatic dependent launch: global memory only after the
    // previous kernel in the stream has completed
    griddep_wait();
    for (int kb = 0; kb < kbs; ++kb) {
      const uint32_t sa = sbase + kb * Cfg::KB_BYTES;
      // test hook (mma_debug_inject(3)): block 0 arms its first k-block for 16 bytes
      // more than its loads bring, so that barrier never completes and the MMA
      // thread's bounded wait runs out; every load is still issued and lands
      const uint32_t extra = (args.inject == 3 && blockIdx.x == 0 && kb == 0) ? 16u : 0u;
      mbar_arrive_expect_tx(kb_bar(kb), Cfg::KB_BYTES + extra);
      tma_load_2d(sa, &tmA, kb * Cfg::BK, m0, kb_bar(kb));
#pragma unroll
      for (int c = 0; c < Cfg::B_CHUNKS; ++c)
        tma_load_2d(sa + Cfg::A_BYTES + c * Cfg::B_CHUNK_BYTES, &tmB, n0 + c * Cfg::B_ATOM_N, kb * Cfg::BK,
                    kb_bar(kb));
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t tmem_base = *tmem_slot;
  // C of this warp's 32 rows: NB boxes of 32 x 32, one barrier
  const uint32_t cw = cbase + warp * Cfg::NB * Cfg::C_BOX_BYTES;
  if (lane == 0) {
    mbar_arrive_expect_tx(c_bar(warp), Cfg::NB * Cfg::C_BOX_BYTES);
#pragma unroll
    for (int j = 0; j < Cfg::NB; ++j)
      tma_load_2d(cw + j * Cfg::C_BOX_BYTES, &tmC, n0 + 32 * j, m0 + 32 * warp, c_bar(warp));
  }
  if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------- MMA issuer
    for (int kb = 0; kb < kbs; ++kb) {
      if (!small_wait(kb_bar(kb), 0, args, abort_flag)) break;
      tc_fence_after();
      const uint32_t sa = sbase + kb * Cfg::KB_BYTES;
      const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < Cfg::MMAS; ++kk) {
        const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, LAYOUT_SW128);
        const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
        umma<KIND>(tmem_base, ad, bd, args.idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
    }
    umma_commit(acc_bar);   // also after an abort: arrives once the issued MMAs are done
  }
  // ----------------------------------------------------------- epilogue (all warps)
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  bool ok = warp_wait_phase(acc_bar, 0, args, abort_flag) && !*abort_flag;
  uint32_t R[BN];
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int j = 0; j < Cfg::NB; ++j) tmem_ld_32x32b_x32_to(tmem_base + lane_off + j * 32, R + j * 32);
    tmem_wait_ld();
  }
  tc_fence_before();
  ok = ok && warp_wait_phase(c_bar(warp), 0, args, abort_flag);
  if (ok) {
    uint8_t* rows = smem + (cw - sbase) + lane * 128;
#pragma unroll
    for (int j = 0; j < Cfg::NB; ++j) {
      // a box's eight 16-byte chunks of C are all loaded before any sum is stored
      // back (loads issued after a store to the same buffer would wait for it)
      uint8_t* box = rows + j * Cfg::C_BOX_BYTES;
      uint4 cv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) cv[c] = *reinterpret_cast<const uint4*>(box + ((c ^ (lane & 7)) << 4));
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 v;
        v.x = __float_as_uint(__uint_as_float(cv[c].x) + __uint_as_float(R[j * 32 + 4 * c + 0]));
        v.y = __float_as_uint(__uint_as_float(cv[c].y) + __uint_as_float(R[j * 32 + 4 * c + 1]));
        v.z = __float_as_uint(__uint_as_float(cv[c].z) + __uint_as_float(R[j * 32 + 4 * c + 2]));
        v.w = __float_as_uint(__uint_as_float(cv[c].w) + __uint_as_float(R[j * 32 + 4 * c + 3]));
        *reinterpret_cast<uint4*>(box + ((c ^ (lane & 7)) << 4)) = v;
      }
      // the box of D leaves while the next one is added
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tma_store_2d(&tmD, n0 + 32 * j, m0 + 32 * warp, cw + j * Cfg::C_BOX_BYTES);
    }
    if (lane == 0) {
      bulk_commit();
      bulk_wait_read_all();
    }
  } else if (lane == 0) {
    // the C loads were issued: let them land before the block's memory is released
    drain_wait(c_bar(warp), 0, args.wait_ns);
  }
  // the A and B loads land before the block's shared memory is released: after a
  // normal run every k-block's barrier has completed (the MMA thread waited on each
  // before its commit) and these waits return at once; after an abort they cover
  // the loads still in flight, whichever thread gave up
  if (threadIdx.x == 0) {
    for (int kb = 0; kb < kbs; ++kb) drain_wait(kb_bar(kb), 0, args.wait_ns);
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <int KIND, int BN>
cudaError_t launch_small_kind(const TensorMaps& m, const GemmArgs& a, cudaStream_t stream) {
  using Cfg = SmallCfg<KIND, BN>;
  auto kernel = gemm_small_kernel<KIND, BN>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, a.tiles_m * a.tiles_n, Cfg::THREADS, Cfg::SMEM_BYTES, stream, m.a, m.b, m.c, m.d, a);
}

}  // namespace

SmallInfo small_info(bool f8, bool narrow) {
  SmallInfo i;
  if (f8) {
    i.bk = SmallCfg<KIND_F8, 128>::BK;
    i.b_atom_n = SmallCfg<KIND_F8, 128>::B_ATOM_N;
    i.kb_max = SmallCfg<KIND_F8, 128>::KB_MAX;
    i.bn = 128;
  } else {
    i.bk = SmallCfg<KIND_F16, 128>::BK;
    i.b_atom_n = SmallCfg<KIND_F16, 128>::B_ATOM_N;
    i.kb_max = SmallCfg<KIND_F16, 128>::KB_MAX;
    i.bn = narrow ? 64 : 128;
  }
  i.bm = 128;
  return i;
}

cudaError_t launch_small(bool f8, int bn, const TensorMaps& m, const GemmArgs& a, cudaStream_t stream) {
  if (f8) return bn == 128 ? launch_small_kind<KIND_F8, 128>(m, a, stream) : cudaErrorInvalidValue;
  if (bn == 64) return launch_small_kind<KIND_F16, 64>(m, a, stream);
  return bn == 128 ? launch_small_kind<KIND_F16, 128>(m, a, stream) : cudaErrorInvalidValue;
}

}  // namespace mma42
