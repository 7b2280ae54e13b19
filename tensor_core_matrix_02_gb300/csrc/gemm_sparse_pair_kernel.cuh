// gemm_sparse_pair_kernel.cuh -- persistent 4:2-sparse GEMM on CTA pairs
// (tcgen05 cta_group::2): D = A*B + C with A given compressed as (vals, idx).
//
// The operation is the compressed-A product of "CDNA3 sparse MFMA builtins",
// section "Structured sparsity (4:2 pattern)": the two kept elements of each
// group of four meet the rows of B that the index names.
//
// Each output block is 256 x 256 and belongs to a cluster of two CTAs on two SMs.
// CTA r (r = 0, 1) stages rows [128 r, 128 r + 128) of compressed A and columns
// [128 r, 128 r + 128) of B; one thread of CTA 0 issues
// tcgen05.mma.sp.cta_group::2 (M = 256, N = 256, K = 32 logical for f16, 64 for
// FP8), which reads both CTAs' shared memory and index and accumulates each CTA's
// 128 rows in its own TMEM.  Per SM this moves half the B bytes per flop of a
// one-SM 128 x 256 tile.
//
// Stages are long: one 128-byte row of compressed A per row (128 logical K for
// f16, 256 for FP8: four MMAs) and the matching rows of B.  Each stage costs the
// TMA producer a fixed ~280 SM clocks plus ~80 per box whatever the box's size
// (measured with mma_tma_feed_probe), and the 4:2 MMA consumes a stage in half the
// time of a dense one; with 64-byte rows the sparse GEMMs stayed at ~42% of the
// tensor cores' rate.  The index does not travel through the shared-memory ring: a
// warpgroup of its own (one warp per TMEM lane quadrant) loads each row's index
// words from global memory a ring's depth ahead into registers and writes them
// into the stage's TMEM slots with tcgen05.st, so the ring holds A and B only and
// four stages fit (an index box per stage cost the FP8 kernel its fourth stage and
// a fifth of its rate).
//
// Roles (512 threads, four warpgroups): warp 0 TMA producer, warp 1 TMEM owner
// and, in CTA 0, MMA issuer, warps 2-3 idle; warps 4-7 the index writers; warps
// 8-15 the epilogue, two per lane quadrant, 128 columns each.  Barriers: both
// CTAs' TMA loads complete on CTA 0's full barrier and both CTAs' index writers
// arrive on CTA 0's index barrier of the stage; CTA 0's MMA thread commits to the
// empty and accumulator-full barriers of both CTAs; the epilogue warps of both
// CTAs arrive on CTA 0's accumulator-empty barrier.  With one accumulator the
// epilogue copies it to registers and hands it back before adding C.
//
// The index reaches the writers in a device-native layout made by a pre-pass
// (meta_native_kernel): for each 64 logical K and each row, the 8 bytes that TMEM
// lane (row % 128) needs, in a 16-column-aligned TMEM slot (an unaligned index
// address faults).
//
// INTACC (the exact sparse 8-bit integer path, values and B widened to bf16): the
// K loop is cut into chunks (args.chunk_kb stages) whose f32 sums are integers of
// magnitude <= 2^24 (2048 logical K, i.e. 1024 products per output, for signed
// A; 1024 for unsigned A; an unsigned B arrives shifted to signed, its correction
// beta * rowsum(A) added with C).  After each chunk the epilogue converts the
// accumulator to i32 and adds it to running sums in registers (wrapping), and after
// the last one adds C (brought by TMA through the staging buffer, its first slice
// loaded and the rest prefetched into L2 when the block starts) and stores D.  With
// one accumulator the MMAs wait for each chunk's drain.
#pragma once
#include "gemm_args.h"
#include "gemm_kernel.cuh"
#include "ptx.cuh"

namespace mma42 {

// Register budgets: 512 threads x 128 at launch >= 128 x 40 (producer / MMA
// warpgroup) + 128 x 64 (index writers) + 256 x 200 (epilogue).
constexpr int kSparseLowRegs = 40;
constexpr int kSparseMetaRegs = 64;
constexpr int kSparseHighRegs = 200;
static_assert(128 * kSparseLowRegs + 128 * kSparseMetaRegs + 256 * kSparseHighRegs <= 512 * 128,
              "register split exceeds the launch");

template <int KIND>
struct SparsePairCfg {
  static constexpr int BM = 128;                          // rows per CTA (256 per pair)
  static constexpr int BN = 256;                          // columns per pair (128 of B per CTA)
  static constexpr int ELEM = (KIND == KIND_F16) ? 2 : 1;
  static constexpr int A_ROW = 128;                       // bytes of compressed A per row per stage
  static constexpr int BKA = A_ROW / ELEM;                // compressed elements per row per stage
  static constexpr int BKL = 2 * BKA;                     // logical K per stage: 128 (f16), 256 (FP8)
  static constexpr int UMMA_KL = (KIND == KIND_F16) ? 32 : 64;
  static constexpr int MMAS = BKL / UMMA_KL;              // 4
  static constexpr int A_BYTES = BM * A_ROW;              // 16 KB
  static constexpr int B_ATOM_N = 128 / ELEM;
  static constexpr int B_COLS = BN / 2;                   // columns of B staged by one CTA
  static constexpr int B_CHUNKS = B_COLS / B_ATOM_N;      // 2 (f16), 1 (FP8)
  static constexpr int B_CHUNK_BYTES = BKL * 128;         // 16 KB (f16), 32 KB (FP8)
  static constexpr int B_BYTES = B_CHUNKS * B_CHUNK_BYTES;   // 32 KB
  static constexpr int B_KSTEP = UMMA_KL * 128;
  // The index of 64 logical K sits in one 16-column TMEM slot per lane: kind::f16
  // keeps two MMAs' 32-bit words in its first two columns and picks them with the
  // sparsity selector; kind::f8f6f4 (a non-zero selector raised an illegal
  // instruction on sm_103a) gives each MMA its own slot, 64 bits in two columns.
  static constexpr int MMAS_PER_SLOT = (KIND == KIND_F16) ? 2 : 1;
  static constexpr int META_SLOTS = MMAS / MMAS_PER_SLOT;    // per stage: 2 (f16), 4 (FP8)
  // one stage's index as 128 x 16-byte tiles: the form the tcgen05 peak measurement
  // copies into TMEM with tcgen05.cp (the GEMM's index writers use tcgen05.st)
  static constexpr int META_SLOT_BYTES = BM * 16;
  static constexpr int META_BYTES = META_SLOTS * META_SLOT_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_COLS = 32;                     // staging: 32 rows x 32 f32, 128-byte swizzled
  static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 4;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUF_BYTES;
  static constexpr int MISC_BYTES = 512;
  static constexpr int STAGES_FIT = (232448 - 1024 - MISC_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;   // 4
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + MISC_BYTES;
  static constexpr int META_SLOT_COLS = 16;
  static constexpr int META_COL0 = BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr int META_WARP0 = 4;                    // warpgroup 1
  static constexpr int EPI_WARP0 = 8;                     // warpgroups 2 and 3
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static_assert(THREADS == 512, "the register split assumes four warpgroups");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
  static_assert(STAGES >= 4, "pipeline too shallow");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(BN + STAGES * META_SLOTS * META_SLOT_COLS <= TMEM_COLS, "tensor memory overflow");
  static_assert(MISC_BYTES >= 8 * (3 * STAGES + 11) + 8, "barrier area");
};

// Byte offset of 16-byte chunk c of row `row` in an epilogue staging buffer of
// EPI_COLS f32 columns: the 128-byte swizzle (chunk ^ row % 8) for 128-byte rows,
// the 64-byte swizzle (chunk ^ (row / 2) % 4) for 64-byte rows.
template <int EPI_COLS>
__device__ __forceinline__ uint32_t epi_chunk_off(int row, int c) {
  if constexpr (EPI_COLS == 32) return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
  else return static_cast<uint32_t>(row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
}

template <int KIND, bool INTACC>
__global__ void __launch_bounds__(SparsePairCfg<KIND>::THREADS, 1)
    gemm_sparse_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                            const GemmArgs args) {
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
  // barrier slots: full[S], empty[S], meta[S], tfull, tempty, epi[8], drain
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto meta_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
  const uint32_t tfull_bar = bar0 + 8u * (3 * S);
  const uint32_t tempty_bar = bar0 + 8u * (3 * S + 1);
  auto epi_bar = [&](int w) { return bar0 + 8u * (3 * S + 2 + w); };
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (3 * S + 11));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8 * (3 * S + 11) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());   // 0 issues the MMAs
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(meta_bar(s), 8);   // four index-writer warps in each CTA
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

  if (warp < Cfg::META_WARP0) {
    regs_lower<kSparseLowRegs>();   // warps 2 and 3 only give their registers up
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
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
            tma_load_2d_pair(sa, &tmA, kb * Cfg::BKA, m0, fb);
            if (Cfg::B_CHUNKS == 2 && args.b_chunks_3d) {
              // both 64-column chunks in one box of a 3-D view of B (x: the chunk's
              // columns, y: K, z: chunk): one box fewer per stage
              tma_load_3d_pair(sb, &tmB, 0, kb * Cfg::BKL, nb / Cfg::B_ATOM_N, fb);
            } else {
#pragma unroll
              for (int c = 0; c < Cfg::B_CHUNKS; ++c)
                tma_load_2d_pair(sb + c * Cfg::B_CHUNK_BYTES, &tmB, nb + c * Cfg::B_ATOM_N, kb * Cfg::BKL, fb);
            }
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
      // ---------------------------------------------------- MMA issuer (CTA 0)
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
              if (!wait_phase(meta_bar(stage), phase, args, abort_flag)) { ok = false; break; }
              tc_fence_after();
              const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
              const uint32_t sb = sa + Cfg::A_BYTES;
              const uint32_t meta = tmem_base + Cfg::META_COL0 + stage * Cfg::META_SLOTS * Cfg::META_SLOT_COLS;
#pragma unroll
              for (int kk = 0; kk < Cfg::MMAS; ++kk) {
                // A: 32 bytes of each 128-byte swizzled row per MMA, as the dense kernels
                const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, LAYOUT_SW128);
                const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
                // f16: slot kk / 2, selector kk % 2; FP8: slot kk, selector 0
                const uint32_t mslot = meta + (kk / Cfg::MMAS_PER_SLOT) * Cfg::META_SLOT_COLS;
                const uint32_t idesc = args.idesc | static_cast<uint32_t>(kk % Cfg::MMAS_PER_SLOT);
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
    }
  } else if (warp < Cfg::EPI_WARP0) {
    regs_lower<kSparseMetaRegs>();
    // ---------------------------------------------------- index writers (both CTAs)
    // Warp q of this warpgroup serves TMEM lanes [32 q, 32 q + 32): lane l writes the
    // index of row m0 + 32 q + l.  The words of stage g are loaded PF stages ahead
    // into registers (a load does not wait for any stage); a stage's TMEM slots are
    // written once its previous MMAs have completed (its empty barrier), then CTA 0's
    // index barrier of the stage is told.  The tcgen05 fences order the writes
    // against the MMAs, so the arrive releases at CTA scope only: a cluster-scope
    // release also waited for the loads still in flight for later stages, and the
    // kernel ran at 37% of its speed.
    constexpr int PF = S;
    constexpr int SL = Cfg::META_SLOTS;
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint2* meta_src = static_cast<const uint2*>(args.meta);
    const int64_t mrows = args.meta_rows;
    const uint32_t mbar_leader = mapa_shared(meta_bar(0), 0);
    // the load cursor runs PF stages ahead of the write cursor over the same walk
    int lu = cid, lkb = 0;
    auto load_stage = [&](uint2 (&w)[SL]) {
      if (lu < units) {
        int mt, nt;
        tile_coords(lu, args, mt, nt);
        const int64_t row = static_cast<int64_t>(mt) * 2 * Cfg::BM + rank * Cfg::BM + q * 32 + lane;
#pragma unroll
        for (int sl = 0; sl < SL; ++sl)
          w[sl] = __ldg(meta_src + (static_cast<int64_t>(lkb) * SL + sl) * mrows + row);
        if (++lkb == args.kblocks) { lkb = 0; lu += ncl; }
      }
    };
    uint2 buf[PF][SL];
#pragma unroll
    for (int p = 0; p < PF; ++p) load_stage(buf[p]);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int64_t total = static_cast<int64_t>((units - cid + ncl - 1) / ncl) * args.kblocks;
    for (int64_t g0 = 0; g0 < total && ok; g0 += PF) {
#pragma unroll
      for (int p = 0; p < PF; ++p) {
        if (g0 + p >= total) break;
        if (!warp_wait_phase(empty_bar(stage), phase ^ 1u, args, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t slot0 = tmem_base + lane_off + Cfg::META_COL0 + stage * SL * Cfg::META_SLOT_COLS;
#pragma unroll
        for (int sl = 0; sl < SL; ++sl) tmem_st_32x32b_x2(slot0 + sl * Cfg::META_SLOT_COLS, buf[p][sl].x, buf[p][sl].y);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mbar_leader + 8u * stage);
        load_stage(buf[p]);   // the stage PF ahead
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    regs_raise<kSparseHighRegs>();
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - Cfg::EPI_WARP0;    // 0..7
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
      // EC-column slices of this warp's 128 columns that hold columns of D (the rest of
      // a ragged last block column is neither loaded nor stored)
      constexpr int EC = Cfg::EPI_COLS;
      constexpr int NSL = 128 / EC;
      constexpr int CPR = EC / 4;   // 16-byte chunks per staged row
      const int live = x0 < args.N ? min(NSL, (args.N - x0 + EC - 1) / EC) : 0;
      uint32_t R[128];
      if constexpr (INTACC) {
        // ------------------------------------------------ exact integer epilogue
        // C comes by TMA, one 32-row slice at a time, through the swizzled staging
        // buffer: the first slice now, once the previous block's D has left the
        // buffer, the others into L2, so that no chunk waits for C.
        if (live > 0) {
          if (lane == 0) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0, y0, eb);
            for (int j = 1; j < live; ++j) tma_prefetch_2d(&tmC, x0 + j * EC, y0);
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
        // an unsigned B run as B' = B - beta: D gets beta * rowsum(A) of this row (wrapping)
        const int row = y0 + lane;
        const uint32_t rfix = (args.beta != 0 && row < args.M)
                                  ? static_cast<uint32_t>(args.beta) * static_cast<uint32_t>(args.rowsum[row])
                                  : 0u;
#pragma unroll
        for (int j = 0; j < NSL; ++j) {
          if (j >= live) break;
          // D = C + the sums (wrapping): C's slice arrived in the buffer, D replaces it
          if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
          ++loads;
          c_pending = false;
#pragma unroll
          for (int c = 0; c < CPR; ++c) {
            uint4* p = reinterpret_cast<uint4*>(bufp + epi_chunk_off<EC>(lane, c));
            const uint4 cv = *p;
            *p = make_uint4(R[j * EC + 4 * c + 0] + cv.x + rfix, R[j * EC + 4 * c + 1] + cv.y + rfix,
                            R[j * EC + 4 * c + 2] + cv.z + rfix, R[j * EC + 4 * c + 3] + cv.w + rfix);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, x0 + j * EC, y0, buf);
            bulk_commit();
            if (j + 1 < live) {
              bulk_wait_read_all();
              mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
              tma_load_2d(buf, &tmC, x0 + (j + 1) * EC, y0, eb);
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
      for (int j = 0; j < NSL; ++j) {
        if (j >= live) break;
        if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
        ++loads;
        c_pending = false;
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
          uint4* p = reinterpret_cast<uint4*>(bufp + epi_chunk_off<EC>(lane, c));
          const uint4 cv = *p;
          uint4 v;
          v.x = __float_as_uint(__uint_as_float(cv.x) + __uint_as_float(R[j * EC + 4 * c + 0]));
          v.y = __float_as_uint(__uint_as_float(cv.y) + __uint_as_float(R[j * EC + 4 * c + 1]));
          v.z = __float_as_uint(__uint_as_float(cv.z) + __uint_as_float(R[j * EC + 4 * c + 2]));
          v.w = __float_as_uint(__uint_as_float(cv.w) + __uint_as_float(R[j * EC + 4 * c + 3]));
          *p = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmD, x0 + j * EC, y0, buf);
          bulk_commit();
          if (j + 1 < live) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0 + (j + 1) * EC, y0, eb);
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
