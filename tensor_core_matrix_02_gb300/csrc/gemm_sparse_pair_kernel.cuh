// gemm_sparse_pair_kernel.cuh -- persistent 4:2-sparse GEMM on CTA pairs
// (tcgen05 cta_group::2): D = A*B + C with A given compressed as (vals, idx).
//
// The operation is the compressed-A product of "CDNA3 sparse MFMA builtins",
// section "Structured sparsity (4:2 pattern)": the two kept elements of each
// group of four meet the rows of B that the index names.
//
// Each output block is 256 x 256 and belongs to a cluster of two CTAs on two SMs.
// CTA r (r = 0, 1) stages rows [128 r, 128 r + 128) of compressed A and of the
// index, and columns [128 r, 128 r + 128) of B; one thread of CTA 0 issues
// tcgen05.mma.sp.cta_group::2 (M = 256, N = 256, K = 32 logical for f16, 64 for
// FP8), which reads both CTAs' shared memory and accumulates each CTA's 128 rows
// in its own TMEM.  Per SM this moves half the B bytes per flop of a one-SM
// 128 x 256 tile, which is what lets the sparse rate (twice the dense one) be fed.
//
// Barriers: both CTAs' TMA loads complete on CTA 0's full barrier; CTA 0's MMA
// thread commits to the empty and accumulator-full barriers of both CTAs; the
// epilogue warps of both CTAs arrive on CTA 0's accumulator-empty barrier.
// The index reaches TMEM through a device-native layout made by a pre-pass
// (meta_native_kernel): 128 x 16-byte tiles whose row r holds the index word(s) of
// TMEM lane r, copied by tcgen05.cp .128x128b into 16-column-aligned slots (an
// unaligned index address faults).
//
// INTACC (the exact sparse 8-bit integer path, values and B widened to bf16): the
// K loop is cut into chunks (args.chunk_kb stages) whose f32 sums are integers of
// magnitude <= 2^24 (2048 logical K, i.e. 1024 products per output, for signed
// A; 1024 for unsigned A; an unsigned B arrives shifted to signed, its correction
// beta * rowsum(A) added with C).  After each chunk the epilogue converts the accumulator to i32 and adds
// it to running sums in registers (wrapping), and after the last one adds C
// (brought by TMA through the staging buffer, its first slice loaded and the
// rest prefetched into L2 when the block starts) and stores D.  With one accumulator
// the MMAs wait for each chunk's drain.
#pragma once
#include "gemm_args.h"
#include "gemm_kernel.cuh"
#include "ptx.cuh"

namespace mma42 {

template <int KIND>
struct SparsePairCfg {
  static constexpr int BM = 128;                          // rows per CTA (256 per pair)
  static constexpr int BN = 256;                          // columns per pair (128 of B per CTA)
  static constexpr int ELEM = (KIND == KIND_F16) ? 2 : 1;
  static constexpr int A_ROW = 64;                        // bytes of compressed A per row per stage
  static constexpr int BKA = A_ROW / ELEM;
  static constexpr int BKL = 2 * BKA;                     // logical K per stage: 64 (f16), 128 (FP8)
  static constexpr int UMMA_KL = (KIND == KIND_F16) ? 32 : 64;
  static constexpr int MMAS = BKL / UMMA_KL;              // 2
  static constexpr int A_BYTES = BM * A_ROW;              // 8 KB
  static constexpr int B_ATOM_N = 128 / ELEM;
  static constexpr int B_COLS = BN / 2;                   // columns of B staged by one CTA
  static constexpr int B_CHUNKS = B_COLS / B_ATOM_N;      // 2 (f16), 1 (FP8)
  static constexpr int B_CHUNK_BYTES = BKL * 128;
  static constexpr int B_BYTES = B_CHUNKS * B_CHUNK_BYTES;   // 16 KB
  static constexpr int B_KSTEP = UMMA_KL * 128;
  static constexpr int META_SLOT_BYTES = BM * 16;
  // kind::f16: both MMAs' 32-bit index words share one 128-bit TMEM slot and are picked
  // with the sparsity selector (columns 0 and 1).  kind::f8f6f4 raised an illegal
  // instruction with a non-zero selector on sm_103a, so each FP8 MMA has its own slot.
  static constexpr int META_SLOTS = (KIND == KIND_F16) ? 1 : MMAS;   // per stage
  static constexpr int META_BYTES = META_SLOTS * META_SLOT_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + META_BYTES;   // 28 KB per CTA
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_BUF_BYTES = 32 * 32 * 4;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUF_BYTES;
  static constexpr int MISC_BYTES = 512;
  static constexpr int STAGES_FIT = (232448 - 1024 - MISC_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + MISC_BYTES;
  static constexpr int META_SLOT_COLS = 16;
  static constexpr int META_COL0 = BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
  static_assert(STAGES >= 4, "pipeline too shallow");
  static_assert(BN + STAGES * META_SLOTS * META_SLOT_COLS <= TMEM_COLS, "tensor memory overflow");
};

template <int KIND, bool INTACC>
__global__ void __launch_bounds__(SparsePairCfg<KIND>::THREADS, 1)
    gemm_sparse_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmMeta, const __grid_constant__ CUtensorMap tmC,
                            const __grid_constant__ CUtensorMap tmD, const GemmArgs args) {
  using Cfg = SparsePairCfg<KIND>;
  constexpr int S = Cfg::STAGES;
  constexpr uint16_t kPair = 3;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t epi_base = sbase + S * Cfg::STAGE_BYTES;
  uint8_t* misc = smem + S * Cfg::STAGE_BYTES + Cfg::EPI_BYTES;
  const uint32_t bar0 = smem_addr(misc);
  // barrier slots: full[S], empty[S], tfull, tempty, epi[8], drain
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * S);
  const uint32_t tempty_bar = bar0 + 8u * (2 * S + 1);
  auto epi_bar = [&](int w) { return bar0 + 8u * (2 * S + 2 + w); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * S + 11));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * (2 * S + 11) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());   // 0 issues the MMAs
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * Cfg::EPI_WARPS);
    for (int w = 0; w < Cfg::EPI_WARPS; ++w) mbar_init(epi_bar(w), 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), Cfg::TMEM_COLS);   // both CTAs, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // launched with programmatic dependent launch: the set-up above overlapped the end
  // of the previous kernel; global memory is touched only after it has completed
  griddep_launch_dependents();
  griddep_wait();
  const int units = args.tiles_m * args.tiles_n;   // 256 x 256 blocks

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
      prefetch_tensormap(&tmMeta);
      int stage = 0;
      uint32_t phase = 0;
      bool issued[S];
      uint32_t issued_phase[S];
      for (int s = 0; s < S; ++s) issued[s] = false;
      bool ok = true;
      bool first = true;
      for (int u = cid; u < units && ok; u += ncl) {
        int mt, nt;
        tile_coords(u, args, mt, nt);
        const int m0 = mt * 2 * Cfg::BM + rank * Cfg::BM;
        const int nb = nt * Cfg::BN + rank * Cfg::B_COLS;
        for (int kb = 0; kb < args.kblocks; ++kb) {
          if (!wait_phase(empty_bar(stage), phase ^ 1u, args, abort_flag)) { ok = false; break; }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          // test hook (mma_debug_inject(2)): cluster 0 arms its first stage for 16 bytes
          // more than its loads bring, so that stage never completes and the MMA
          // thread's bounded wait runs out; every load is still issued and lands
          const uint32_t extra = (args.inject == 2 && cid == 0 && first) ? 16u : 0u;
          first = false;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2u * Cfg::STAGE_BYTES + extra);
          const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
          const uint32_t sb = sa + Cfg::A_BYTES;
          const uint32_t sm = sb + Cfg::B_BYTES;
          tma_load_2d_pair(sa, &tmA, kb * Cfg::BKA, m0, fb);
          tma_load_3d_pair(sm, &tmMeta, 0, m0 / 16, kb * Cfg::META_SLOTS, fb);
#pragma unroll
          for (int c = 0; c < Cfg::B_CHUNKS; ++c)
            tma_load_2d_pair(sb + c * Cfg::B_CHUNK_BYTES, &tmB, nb + c * Cfg::B_ATOM_N, kb * Cfg::BKL, fb);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      // after an abort, CTA 0's full barriers of the stages it armed complete only
      // once both CTAs' loads for them have landed
      if (*abort_flag && rank == 0) {
        for (int s = 0; s < S; ++s)
          if (issued[s]) drain_wait(full_bar(s), issued_phase[s], args.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (CTA 0)
    if (rank == 0 && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t round = 0;
      bool ok = true;
      const int chunk = INTACC ? max(1, args.chunk_kb) : args.kblocks;
      for (int u = cid; u < units && ok; u += ncl) {
        for (int c0 = 0; c0 < args.kblocks && ok; c0 += chunk, ++round) {
          const int c1 = min(args.kblocks, c0 + chunk);
          if (!wait_phase(tempty_bar, (round & 1u) ^ 1u, args, abort_flag)) { ok = false; break; }
          tc_fence_after();
          for (int kb = c0; kb < c1; ++kb) {
            if (!wait_phase(full_bar(stage), phase, args, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
            const uint32_t sb = sa + Cfg::A_BYTES;
            const uint32_t sm = sb + Cfg::B_BYTES;
            const uint32_t meta = tmem_base + Cfg::META_COL0 + stage * Cfg::META_SLOTS * Cfg::META_SLOT_COLS;
#pragma unroll
            for (int sl = 0; sl < Cfg::META_SLOTS; ++sl)
              tmem_cp_pair_128x128b(meta + sl * Cfg::META_SLOT_COLS,
                                    smem_desc(sm + sl * Cfg::META_SLOT_BYTES, Cfg::META_SLOT_BYTES, 128, LAYOUT_NONE));
#pragma unroll
            for (int kk = 0; kk < Cfg::MMAS; ++kk) {
              const uint64_t ad = smem_desc(sa + kk * 32, 16, 8 * Cfg::A_ROW, LAYOUT_SW64);
              const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
              // f16: same slot, selector kk; FP8: slot kk, selector 0
              const uint32_t mslot = (Cfg::META_SLOTS == 1) ? meta : meta + kk * Cfg::META_SLOT_COLS;
              const uint32_t idesc = (Cfg::META_SLOTS == 1) ? (args.idesc | static_cast<uint32_t>(kk)) : args.idesc;
              umma_sp_pair<KIND>(tmem_base, ad, bd, mslot, idesc, (kb > c0 || kk > 0) ? 1u : 0u);
            }
            umma_commit_pair_mc(empty_bar(stage), kPair);
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          umma_commit_pair_mc(tfull_bar, kPair);
        }
      }
      umma_commit_pair_mc(drain_bar, kPair);
      drain_wait(drain_bar, 0, args.wait_ns);
    }
  } else {
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;                 // 0..7
    const int q = warp & 3;                  // TMEM lane quadrant
    const int half = ew >> 2;                // which 128 of the 256 columns
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t buf = epi_base + ew * Cfg::EPI_BUF_BYTES;
    uint8_t* bufp = smem + (buf - sbase);
    const uint32_t eb = epi_bar(ew);
    const uint32_t tempty_leader = mapa_shared(tempty_bar, 0);
    uint32_t loads = 0;
    bool c_pending = false;
    bool ok = true;
    uint32_t round = 0;
    for (int u = cid; u < units && ok; u += ncl) {
      int mt, nt;
      tile_coords(u, args, mt, nt);
      const int y0 = mt * 2 * Cfg::BM + rank * Cfg::BM + q * 32;
      const int x0 = nt * Cfg::BN + half * 128;
      // 32-column slices of this warp's columns that hold columns of D (the rest of a
      // ragged last block column is neither loaded nor stored)
      const int live = x0 < args.N ? min(4, (args.N - x0 + 31) / 32) : 0;
      uint32_t R[128];
      if constexpr (INTACC) {
        // ------------------------------------------------ exact integer epilogue
        // C comes by TMA, one 32 x 32 slice at a time, through the swizzled staging
        // buffer: the first slice now, once the previous block's D has left the
        // buffer, the others into L2, so that no chunk waits for C.
        if (live > 0) {
          if (lane == 0) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0, y0, eb);
            for (int j = 1; j < live; ++j) tma_prefetch_2d(&tmC, x0 + j * 32, y0);
          }
          c_pending = true;
        }
#pragma unroll
        for (int i = 0; i < 128; ++i) R[i] = 0u;
        const int chunk = max(1, args.chunk_kb);
        for (int c0 = 0; c0 < args.kblocks; c0 += chunk, ++round) {
          if (!warp_wait_phase(tfull_bar, round & 1u, args, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            __syncwarp();
            tmem_ld_32x32b_x32(tmem_base + lane_off + half * 128 + j * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              R[j * 32 + i] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i])));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_leader);
        }
        if (!ok) break;
        uint8_t* rowp = bufp + lane * 128;
        // an unsigned B run as B' = B - beta: D gets beta * rowsum(A) of this row (wrapping)
        const int row = y0 + lane;
        const uint32_t rfix = (args.beta != 0 && row < args.M)
                                  ? static_cast<uint32_t>(args.beta) * static_cast<uint32_t>(args.rowsum[row])
                                  : 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j >= live) break;
          // D = C + the sums (wrapping): C's slice arrived in the buffer, D replaces it
          if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
          ++loads;
          c_pending = false;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4));
            const uint4 cv = *p;
            *p = make_uint4(R[j * 32 + 4 * c + 0] + cv.x + rfix, R[j * 32 + 4 * c + 1] + cv.y + rfix,
                            R[j * 32 + 4 * c + 2] + cv.z + rfix, R[j * 32 + 4 * c + 3] + cv.w + rfix);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, x0 + j * 32, y0, buf);
            bulk_commit();
            if (j + 1 < live) {
              bulk_wait_read_all();
              mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
              tma_load_2d(buf, &tmC, x0 + (j + 1) * 32, y0, eb);
            }
          }
          if (j + 1 < live) c_pending = true;
        }
        continue;
      }
      // ---------------------------------------------------- floating-point epilogue
      const uint32_t rnd = round++;
      if (live > 0) {
        if (lane == 0) {   // C of the first slice while the main loop runs
          bulk_wait_read_all();
          mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
          tma_load_2d(buf, &tmC, x0, y0, eb);
        }
        c_pending = true;
      }
      if (!warp_wait_phase(tfull_bar, rnd & 1u, args, abort_flag)) { ok = false; break; }
      tc_fence_after();
      __syncwarp();
      // all slices' loads in flight together, one wait: the accumulator goes back sooner
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32_to(tmem_base + lane_off + half * 128 + j * 32, R + j * 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);   // this CTA's half of the accumulator is free
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j >= live) break;
        if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
        ++loads;
        c_pending = false;
        uint8_t* rowp = bufp + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4));
          const uint4 cv = *p;
          uint4 v;
          v.x = __float_as_uint(__uint_as_float(cv.x) + __uint_as_float(R[j * 32 + 4 * c + 0]));
          v.y = __float_as_uint(__uint_as_float(cv.y) + __uint_as_float(R[j * 32 + 4 * c + 1]));
          v.z = __float_as_uint(__uint_as_float(cv.z) + __uint_as_float(R[j * 32 + 4 * c + 2]));
          v.w = __float_as_uint(__uint_as_float(cv.w) + __uint_as_float(R[j * 32 + 4 * c + 3]));
          *p = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmD, x0 + j * 32, y0, buf);
          bulk_commit();
          if (j + 1 < live) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0 + (j + 1) * 32, y0, eb);
          }
        }
        if (j + 1 < live) c_pending = true;
      }
    }
    if (lane == 0) {
      if (c_pending) drain_wait(eb, loads & 1u, args.wait_ns);
      bulk_wait_all();
    }
    tc_fence_before();
    __syncwarp();
  }

  __syncthreads();
  // neither CTA leaves while the pair's MMAs, loads or arrivals may still touch it
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace mma42
