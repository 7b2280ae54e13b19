// gemm_args.h -- launch arguments shared by the host dispatcher and the GEMM kernel.
#pragma once
#include <cstdint>

namespace mma42 {


struct GemmArgs {
  int M, N, K;             // K is the logical (uncompressed) length
  int tiles_m, tiles_n;    // output tiles
  int ksplit;              // K splits per tile (>1 writes f32 partials)
  int kblocks;             // ceil(K / logical K per stage)
  int chunk_kb;            // integer path: k-blocks per exactly accumulated chunk, chosen on the
                           // host so that a chunk's f32 sum is an integer of magnitude <= 2^24
  int group_m;             // tile raster: tiles of group_m m-rows are walked together
  uint32_t idesc;          // tcgen05 instruction descriptor
  int* err;                // device error word
  unsigned long long wait_ns;
  int inject;              // test hook (see mma_debug_inject)
  const void* c = nullptr; // C itself (the integer path reads it with plain loads)
  int clamp = 0;           // integer path: saturate D to the i32 range instead of wrapping
  // integer path with unsigned operands run as signed ones (A = A' + alpha, B = B' +
  // beta): D gets beta * rowsum[i] + alpha * colsum[j] + alpha * beta * K added
  const int32_t* rowsum = nullptr;
  const int32_t* colsum = nullptr;
  int alpha = 0, beta = 0;
  // tail split (CTA-pair kernel, ksplit == 1): units below tail_from are whole
  // tiles; the tiles from tail_from on (the raster's last, which a grid that does
  // not divide the tiles evenly runs in a short last round) are cut into
  // tail_split K slices that write partials.  0: none.
  int tail_from = 0;
  int tail_split = 0;
  // 4:2-sparse kernel: the index in its device-native layout, 8 bytes per row per 64
  // logical K ([slot][row], meta_rows rows per slot)
  const void* meta = nullptr;
  int64_t meta_rows = 0;
  // 4:2-sparse kernel, 16-bit B: the B map is the 3-D view (64 columns, K, N / 64
  // chunks) and a stage's two column chunks come in one box
  int b_chunks_3d = 0;
};

}  // namespace mma42
