// gemm_pair_kernel.cuh -- persistent dense GEMM on CTA pairs (tcgen05 cta_group::2):
// D = A*B + C, the matrix multiply-accumulate of "CDNA dense MFMA builtins",
// section "Naming convention", over whole matrices.
//
// Each output block is 256 x 256 and belongs to a cluster of two CTAs on two SMs.
// CTA r stages rows [128 r, 128 r + 128) of A and columns [128 r, 128 r + 128) of
// B; one thread of CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16
// for f16/bf16, 32 for FP8) reading both CTAs' shared memory; each CTA accumulates
// its 128 rows in its own TMEM.  Per SM this moves two thirds of the operand bytes
// per flop of a one-SM 128 x 256 tile.
//
// When there are fewer blocks than SM pairs and K is long, K is cut into slices:
// a work unit is then one slice of one block, which stores its f32 accumulator as
// a partial (3-D tensor map over ksplit x M x N), and a separate reduction adds
// the partials in slice order, then C (a result that does not depend on timing).
// When there are more blocks than SM pairs but the last round would leave more
// than half of the pairs idle, only the blocks of that round are cut into K
// slices (a tail split): their partials go to a compact buffer of those blocks,
// and a reduction over just them finishes D.
//
// INTACC (the exact 8-bit integer path, operands widened to bf16): the K loop is
// cut into chunks (args.chunk_kb k-blocks) short enough that a chunk's f32 sum is
// an integer of magnitude <= 2^24, exact in f32: 1024 K of signed x signed
// products (<= 2^14; unsigned operands arrive shifted to signed).  The epilogue converts
// each chunk to i32 and adds it to running sums kept in registers (wrapping, like
// i32 arithmetic), adds C after the last chunk and stores D from the sums.  C
// comes by TMA through the swizzled staging buffer (its first slice loaded, the
// rest prefetched into L2, when the block starts): per-lane row loads of C cost
// 22 us on 4096^3, the coalesced path almost nothing.  (256-K chunks converted by one f32 add
// of 1.5 * 2^23, exact for |s| <= 2^22, measured no faster than longer chunks with
// the conversion instruction.)
//
// Roles (384 threads, three warpgroups): warp 0 TMA producer (both CTAs), warp 1
// TMEM owner and, in CTA 0, MMA issuer, warps 2 and 3 idle; that warpgroup gives
// up registers to warps 4..11, the epilogue, two per TMEM lane quadrant, 128
// columns each, which hold the drained accumulator (and, for INTACC, the running
// sums) in registers.  Two TMEM accumulators let the epilogue of one unit overlap
// the main loop of the next.  Barriers as in the sparse pair kernel: both CTAs'
// loads complete on CTA 0's full barrier, CTA 0 commits to both CTAs' empty and
// accumulator-full barriers, both CTAs' epilogues release CTA 0's
// accumulator-empty barriers.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_args.h"
#include "gemm_kernel.cuh"
#include "ptx.cuh"

namespace mma42 {

// One chunk's f32 sum (an exact integer of magnitude <= 2^24) as an i32 term.
__device__ __forceinline__ uint32_t chunk_bits(uint32_t acc) {
  return static_cast<uint32_t>(__float2int_rn(__uint_as_float(acc)));
}

// Register budgets: 384 threads x 168 at launch = 128 x 40 (warpgroup 0) + 256 x 232.
constexpr int kPairLaunchRegs = 168;
constexpr int kPairLowRegs = 40;
constexpr int kPairHighRegs = 232;
static_assert(128 * kPairLowRegs + 256 * kPairHighRegs <= 384 * kPairLaunchRegs, "register split exceeds the launch");

template <int KIND, bool INTACC>
struct PairCfg {
  static constexpr int BM = 128;                          // rows per CTA (256 per pair)
  static constexpr int BN = 256;                          // columns per pair
  static constexpr int ACCS = 512 / BN;                   // TMEM accumulators
  static constexpr int COLS_PER_WARP = BN / 2;            // epilogue columns per warp
  static constexpr int SLICES = COLS_PER_WARP / 32;       // 32 x 32 store slices per warp
  static constexpr int ELEM = (KIND == KIND_F16) ? 2 : 1;
  static constexpr int BK = 128 / ELEM;                   // K per stage (one 128-byte row of A)
  static constexpr int UMMA_K = (KIND == KIND_F16) ? 16 : 32;
  static constexpr int MMAS = BK / UMMA_K;                // 4
  static constexpr int A_BYTES = BM * 128;                // 16 KB
  static constexpr int B_ATOM_N = 128 / ELEM;
  static constexpr int B_COLS = BN / 2;                   // columns of B staged by one CTA
  static constexpr int B_CHUNKS = B_COLS / B_ATOM_N;      // 2 (16-bit, INTACC too), 1 (FP8)
  static constexpr int B_CHUNK_BYTES = BK * 128;
  static constexpr int B_BYTES = B_CHUNKS * B_CHUNK_BYTES;   // 16 KB
  static constexpr int B_KSTEP = UMMA_K * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB per CTA
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_BUF_BYTES = 32 * 32 * 4;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUF_BYTES;
  static constexpr int MISC_BYTES = 512;
  static constexpr int STAGES_FIT = (232448 - 1024 - MISC_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + MISC_BYTES;
  static constexpr int TMEM_COLS = 512;                   // ACCS accumulators of BN columns
  static constexpr int EPI_WARP0 = 4;                     // epilogue = warpgroups 1 and 2
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static_assert(THREADS == 384, "the register split assumes three warpgroups");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
  static_assert(STAGES >= 4, "pipeline too shallow");
  static_assert(B_CHUNKS >= 1 && SLICES >= 1, "tile shape");
  static_assert(MISC_BYTES >= 8 * (2 * STAGES + 2 * ACCS + EPI_WARPS + 1) + 8, "barrier area");
};

// Half-precision D (OUT 1: f16, 2: bf16; C of the same type): D = round-to-nearest-
// even(f32(C) + the f32 accumulator), the accumulate variants of "RDNA3 dense WMMA
// builtins", section "Naming convention" (out_type f16 / bf16), accumulated in f32
// and rounded once.  8 values of type OUT in a 16-byte chunk -> f32 (half in, sum).
template <int OUT>
__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
  if constexpr (OUT == 1) return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  else return __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(h)));
}
template <int OUT>
__device__ __forceinline__ uint32_t float_to_half_bits(float f) {
  if constexpr (OUT == 1) return __half_as_ushort(__float2half_rn(f));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int KIND, bool INTACC, int OUT = 0>
__global__ void __launch_bounds__(PairCfg<KIND, INTACC>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmP, const GemmArgs args) {
  using Cfg = PairCfg<KIND, INTACC>;
  constexpr int S = Cfg::STAGES;
  constexpr uint16_t kPair = 3;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t epi_base = sbase + S * Cfg::STAGE_BYTES;
  uint8_t* misc = smem + S * Cfg::STAGE_BYTES + Cfg::EPI_BYTES;
  const uint32_t bar0 = smem_addr(misc);
  // barrier slots: full[S], empty[S], tfull[ACCS], tempty[ACCS], epi[8], drain
  constexpr int NA = Cfg::ACCS;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + NA + b); };
  auto epi_bar = [&](int w) { return bar0 + 8u * (2 * S + 2 * NA + w); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 2 * NA + Cfg::EPI_WARPS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 8 * (2 * S + 2 * NA + Cfg::EPI_WARPS + 1));
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(misc + 8 * (2 * S + 2 * NA + Cfg::EPI_WARPS + 1) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NA; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * Cfg::EPI_WARPS);
    }
    for (int w = 0; w < Cfg::EPI_WARPS; ++w) mbar_init(epi_bar(w), 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), Cfg::TMEM_COLS);
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
  // work units: (K slice, 256 x BN block); a slice of a split K writes an f32 partial
  const int tiles = args.tiles_m * args.tiles_n;
  const int units = unit_count(tiles, args);

  if (warp < Cfg::EPI_WARP0) {
    regs_lower<kPairLowRegs>();   // warps 2 and 3 only give their registers up
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
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
          const WorkUnit wu = unit_of(u, tiles, args);
          int mt, nt;
          tile_coords(wu.tile, args, mt, nt);
          const int kb0 = wu.kb0, kb1 = wu.kb1;
          const int m0 = mt * 2 * Cfg::BM + rank * Cfg::BM;
          const int nb = nt * Cfg::BN + rank * Cfg::B_COLS;
          for (int kb = kb0; kb < kb1; ++kb) {
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
            tma_load_2d_pair(sa, &tmA, kb * Cfg::BK, m0, fb);
#pragma unroll
            for (int c = 0; c < Cfg::B_CHUNKS; ++c)
              tma_load_2d_pair(sb + c * Cfg::B_CHUNK_BYTES, &tmB, nb + c * Cfg::B_ATOM_N, kb * Cfg::BK, fb);
            issued[stage] = true;
            issued_phase[stage] = phase;
            if (++stage == S) { stage = 0; phase ^= 1u; }
          }
        }
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
        for (int u = cid; u < units && ok; u += ncl) {
          const WorkUnit wu = unit_of(u, tiles, args);
          const int kb0 = wu.kb0, kb1 = wu.kb1;
          const int chunk = INTACC ? max(1, args.chunk_kb) : kb1 - kb0;
          for (int c0 = kb0; c0 < kb1 && ok; c0 += chunk, ++round) {
            const int c1 = min(kb1, c0 + chunk);
            const int acc = static_cast<int>(round % NA);
            if (!wait_phase(tempty_bar(acc), ((round / NA) & 1u) ^ 1u, args, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * Cfg::BN;
            for (int kb = c0; kb < c1; ++kb) {
              if (!wait_phase(full_bar(stage), phase, args, abort_flag)) { ok = false; break; }
              tc_fence_after();
              const uint32_t sa = sbase + stage * Cfg::STAGE_BYTES;
              const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
              for (int kk = 0; kk < Cfg::MMAS; ++kk) {
                const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, LAYOUT_SW128);
                const uint64_t bd = smem_desc(sb + kk * Cfg::B_KSTEP, Cfg::B_CHUNK_BYTES, 1024, LAYOUT_SW128);
                umma_pair<KIND>(d_tmem, ad, bd, args.idesc, (kb > c0 || kk > 0) ? 1u : 0u);
              }
              umma_commit_pair_mc(empty_bar(stage), kPair);
              if (++stage == S) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            umma_commit_pair_mc(tfull_bar(acc), kPair);
          }
        }
        umma_commit_pair_mc(drain_bar, kPair);
        drain_wait(drain_bar, 0, args.wait_ns);
      }
    }
  } else {
    regs_raise<kPairHighRegs>();
    // ------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - Cfg::EPI_WARP0;    // 0..7
    const int q = warp & 3;                  // TMEM lane quadrant
    const int half = ew >> 2;                // which half of the BN columns
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t buf = epi_base + ew * Cfg::EPI_BUF_BYTES;
    uint8_t* bufp = smem + (buf - sbase);
    const uint32_t eb = epi_bar(ew);
    uint32_t loads = 0;
    bool c_pending = false;
    bool ok = true;
    uint32_t round = 0;
    const int chunk = max(1, args.chunk_kb);   // INTACC only
    for (int u = cid; u < units && ok; u += ncl) {
      const WorkUnit wu = unit_of(u, tiles, args);
      int mt, nt;
      tile_coords(wu.tile, args, mt, nt);
      const int kb0 = wu.kb0, kb1 = wu.kb1, split = wu.split;
      const bool partial = wu.partial;   // INTACC: i32 partials
      const int y0 = mt * 2 * Cfg::BM + rank * Cfg::BM + q * 32;
      const int x0 = nt * Cfg::BN + half * Cfg::COLS_PER_WARP;
      // where a partial goes: (x0, y0) of the flat ksplit x M x N layout of a plain
      // split, or the tile-relative column and row ptile * 256 + tile row of the
      // compact tail_split x (T * 256) x 256 layout of a tail split
      const bool tail = args.tail_split > 1;
      const int px0 = tail ? x0 - nt * Cfg::BN : x0;
      const int py0 = tail ? wu.ptile * 2 * Cfg::BM + (y0 - mt * 2 * Cfg::BM) : y0;
      // 32-column slices of this warp's columns that hold columns of D (the rest of a
      // ragged last block column is neither loaded nor stored)
      const int live32 = x0 < args.N ? min(Cfg::SLICES, (args.N - x0 + 31) / 32) : 0;
      constexpr int CW = Cfg::COLS_PER_WARP;
      uint32_t R[CW];
      if constexpr (INTACC) {
        // ------------------------------------------------ exact integer epilogue
        // C comes by TMA, one 32 x 32 slice at a time, through the swizzled staging
        // buffer (rows past M and columns past N read as 0): the first slice now, once
        // the previous block's D has left the buffer, the others into L2, so that no
        // chunk waits for C and the final pass reads it coalesced.
        const int row = y0 + lane;
        const bool row_ok = row < args.M;
        if (!partial && live32 > 0) {
          if (lane == 0) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0, y0, eb);
            for (int j = 1; j < live32; ++j) tma_prefetch_2d(&tmC, x0 + j * 32, y0);
          }
          c_pending = true;
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) R[i] = 0u;
        for (int c0 = kb0; c0 < kb1; c0 += chunk, ++round) {
          const int acc = static_cast<int>(round % NA);
          if (!warp_wait_phase(tfull_bar(acc), (round / NA) & 1u, args, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < Cfg::SLICES; ++j) {
            uint32_t r[32];
            __syncwarp();
            tmem_ld_32x32b_x32(tmem_base + lane_off + acc * Cfg::BN + half * CW + j * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) R[j * 32 + i] += chunk_bits(r[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
        }
        if (!ok) break;
        uint8_t* rowp = bufp + lane * 128;
        if (partial) {
          // a K slice's i32 partial sums, 32 x 32 slices through the staging buffer
#pragma unroll
          for (int j = 0; j < Cfg::SLICES; ++j) {
            if (j >= live32) break;
            if (lane == 0) bulk_wait_read_all();   // the previous slice has left the buffer
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4)) = make_uint4(
                  R[j * 32 + 4 * c + 0], R[j * 32 + 4 * c + 1], R[j * 32 + 4 * c + 2], R[j * 32 + 4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmP, px0 + j * 32, py0, split, buf);
              bulk_commit();
            }
          }
          continue;
        }
        const bool fix = args.alpha != 0 || args.beta != 0;
        // corrections of unsigned operands run as signed ones: beta * rowsum + alpha *
        // beta * K per row, alpha * colsum per column
        const int64_t row_fix =
            static_cast<int64_t>(args.alpha) * args.beta * args.K +
            ((row_ok && args.beta != 0) ? static_cast<int64_t>(args.beta) * args.rowsum[row] : 0);
#pragma unroll
        for (int j = 0; j < Cfg::SLICES; ++j) {
          if (j >= live32) break;
          // D = C + the sums: C's slice arrived in the buffer, D replaces it
          if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
          ++loads;
          c_pending = false;
          if (!fix && !args.clamp) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4));
              const uint4 cv = *p;
              *p = make_uint4(R[j * 32 + 4 * c + 0] + cv.x, R[j * 32 + 4 * c + 1] + cv.y,
                              R[j * 32 + 4 * c + 2] + cv.z, R[j * 32 + 4 * c + 3] + cv.w);
            }
          } else {
            // wrapping, or (clamp) summed exactly in 64 bits and saturated to the i32
            // range; the product sum fits i32 here when clamping (the host splits K
            // otherwise)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4));
              const uint4 cv = *p;
              const uint32_t c4[4] = {cv.x, cv.y, cv.z, cv.w};
              const int col = x0 + j * 32 + 4 * c;
              int4 cs = make_int4(0, 0, 0, 0);
              if (args.alpha != 0 && col < args.N) cs = *reinterpret_cast<const int4*>(args.colsum + col);
              const int cf[4] = {cs.x, cs.y, cs.z, cs.w};
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int64_t extra =
                    static_cast<int32_t>(c4[e]) + row_fix + static_cast<int64_t>(args.alpha) * cf[e];
                const uint32_t s = R[j * 32 + 4 * c + e];
                if (args.clamp) {
                  const int64_t sum = static_cast<int64_t>(static_cast<int32_t>(s)) + extra;
                  o[e] = static_cast<uint32_t>(
                      static_cast<int32_t>(sum > INT32_MAX ? INT32_MAX : (sum < INT32_MIN ? INT32_MIN : sum)));
                } else {
                  o[e] = s + static_cast<uint32_t>(static_cast<uint64_t>(extra));
                }
              }
              *p = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, x0 + j * 32, y0, buf);
            bulk_commit();
            if (j + 1 < live32) {
              bulk_wait_read_all();
              mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
              tma_load_2d(buf, &tmC, x0 + (j + 1) * 32, y0, eb);
            }
          }
          if (j + 1 < live32) c_pending = true;
        }
        continue;
      }
      // ---------------------------------------------------- floating-point epilogue
      // D slices: 32 columns of f32 (128-byte rows), or 64 of f16 / bf16; a K slice's
      // f32 partial always goes out in 32-column slices.
      constexpr int OCOLS = (OUT == 0) ? 32 : 64;
      constexpr int OSL = CW / OCOLS;
      const int live_o = x0 < args.N ? min(OSL, (args.N - x0 + OCOLS - 1) / OCOLS) : 0;
      if (!partial && live_o > 0) {
        // C of the first slice while the main loop runs.  (Prefetching the other
        // slices into L2 here too measured 1% slower on the suite: under the long main
        // loops of large GEMMs the early C lines compete with the operand panels.)
        if (lane == 0) {
          bulk_wait_read_all();
          mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
          tma_load_2d(buf, &tmC, x0, y0, eb);
        }
        c_pending = true;
      }
      if (!warp_wait_phase(tfull_bar(round % NA), (round / NA) & 1u, args, abort_flag)) { ok = false; break; }
      {
        const int acc = static_cast<int>(round % NA);
        tc_fence_after();
        __syncwarp();
        // all slices' loads in flight together, one wait: the accumulator goes back sooner
#pragma unroll
        for (int j = 0; j < Cfg::SLICES; ++j)
          tmem_ld_32x32b_x32_to(tmem_base + lane_off + acc * Cfg::BN + half * CW + j * 32, R + j * 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
        ++round;
      }
      uint8_t* rowp = bufp + lane * 128;
      if (partial) {
        // a K slice's partial: the accumulator itself, f32
#pragma unroll
        for (int j = 0; j < Cfg::SLICES; ++j) {
          if (j >= live32) break;
          if (lane == 0) bulk_wait_read_all();   // the previous slice has left the buffer
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4)) =
                make_uint4(R[j * 32 + 4 * c + 0], R[j * 32 + 4 * c + 1], R[j * 32 + 4 * c + 2], R[j * 32 + 4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmP, px0 + j * 32, py0, split, buf);
            bulk_commit();
          }
        }
        continue;
      }
#pragma unroll
      for (int j = 0; j < OSL; ++j) {
        if (j >= live_o) break;
        // D = C + accumulator: C's slice arrived in the buffer, the sum replaces it
        if (!warp_wait_phase(eb, loads & 1u, args, abort_flag)) { ok = false; break; }
        ++loads;
        c_pending = false;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* p = reinterpret_cast<uint4*>(rowp + ((c ^ (lane & 7)) << 4));
          const uint4 cv = *p;
          uint4 v;
          if constexpr (OUT == 0) {
            v.x = __float_as_uint(__uint_as_float(cv.x) + __uint_as_float(R[j * 32 + 4 * c + 0]));
            v.y = __float_as_uint(__uint_as_float(cv.y) + __uint_as_float(R[j * 32 + 4 * c + 1]));
            v.z = __float_as_uint(__uint_as_float(cv.z) + __uint_as_float(R[j * 32 + 4 * c + 2]));
            v.w = __float_as_uint(__uint_as_float(cv.w) + __uint_as_float(R[j * 32 + 4 * c + 3]));
          } else {
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = half_bits_to_float<OUT>(cw[e] & 0xffffu) + __uint_as_float(R[j * 64 + 8 * c + 2 * e]);
              const float hi = half_bits_to_float<OUT>(cw[e] >> 16) + __uint_as_float(R[j * 64 + 8 * c + 2 * e + 1]);
              o[e] = float_to_half_bits<OUT>(lo) | (float_to_half_bits<OUT>(hi) << 16);
            }
            v = make_uint4(o[0], o[1], o[2], o[3]);
          }
          *p = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmD, x0 + j * OCOLS, y0, buf);
          bulk_commit();
          if (j + 1 < live_o) {
            bulk_wait_read_all();
            mbar_arrive_expect_tx(eb, Cfg::EPI_BUF_BYTES);
            tma_load_2d(buf, &tmC, x0 + (j + 1) * OCOLS, y0, eb);
          }
        }
        if (j + 1 < live_o) c_pending = true;
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
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace mma42
