/*
 * mma42.h -- C ABI of libmma42: matrix multiply-accumulate D = A*B + C on the
 * tensor cores of one GB300 (sm_103a) GPU, dense and 4:2 structured-sparse.
 *
 * The operation.  "CDNA dense MFMA builtins", section "Naming convention":
 * a matrix multiply-accumulate takes an M x K panel of A and a K x N panel of
 * B, accumulates their product into an M x N tile of C, and the caller loops
 * over K.  Over whole matrices this is
 *     D[i][j] = C[i][j] + sum_{k<K} A[i][k] * B[k][j].
 * Input types (same page and "CDNA3 sparse MFMA builtins", section "Naming
 * convention"): f16 and bf16 into f32, i8 into i32, and the FP8 formats E4M3
 * and E5M2 in all four A x B combinations into f32.  FP8 is the OCP encoding
 * (the sparse page's note on FP8 encodings: later architectures use OCP E4M3
 * rather than FNUZ).  i8 is signed x signed; the i32 result wraps modulo 2^32.
 *
 * 4:2 sparsity.  "CDNA3 sparse MFMA builtins", section "Structured sparsity
 * (4:2 pattern)": in every contiguous group of four A elements along K at most
 * two are non-zero; compressed A keeps the two (K/2 values per row) and an
 * index records their positions.  Index layout (a reading consistent with the
 * page's keep-{0,2} constants 0x88 and 0x8888): per group one nibble
 * p0 | p1 << 2 with p0 < p1; groups run along K from the low nibble of byte 0,
 * two per byte, so idx is M x K/8 bytes, row-major.  Values within a group are
 * stored in ascending position order.
 *
 * Memory.  Every pointer argument is a DEVICE pointer on the current CUDA
 * device, owned by the caller; the library keeps no reference after the call.
 * All matrices are dense row-major with no padding: A M x K, B K x N, C and D
 * M x N, vals M x K/2, idx M x K/8 bytes.  Base pointers must be 16-byte
 * aligned and every row pitch a multiple of 16 bytes.  D may be the same
 * buffer as C (in place); any other overlap between an output and an input is
 * rejected.
 *
 * Streams and errors.  Calls are asynchronous on `stream` (a cudaStream_t; 0
 * is the legacy default stream).  Argument errors are detected on the host
 * before anything is launched and returned at once.  Errors that arise on the
 * device (a pipeline wait that ran past its time limit) are recorded in a
 * per-process device error word that mma_sync_status() reads.
 *
 * Scratch memory.  The 8-bit integer paths (widened operands, row and column
 * sums of unsigned operands), the K-split paths (partial sums of a few blocks:
 * the long-K split of few output blocks, or the split of a short last round of
 * blocks, at most a few tens of MB) and sparse42_gemm's index layout take
 * stream-ordered scratch from a memory pool the library owns (grown on demand,
 * kept until the process exits).  Nothing else is allocated per call.
 *
 * ABI versions: 1 the calls of the first release; 2 adds MMA_U8, the half-
 * precision outputs, mma_gemm_ex, sparse42_prune, sparse42_quantize_prune and
 * mma_quantize; 3 adds the measurement helper mma_legacy_mma_peak; 4 adds the
 * measurement helper mma_tcgen05_peak (no layout or signature of an earlier
 * version changed).
 */
#ifndef MMA42_H
#define MMA42_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MMA42_ABI_VERSION 5

/* Element types. */
typedef enum {
  MMA_F16 = 1,  /* IEEE binary16 */
  MMA_BF16 = 2, /* bfloat16 */
  MMA_E4M3 = 3, /* OCP FP8 E4M3 (bias 7, no infinities, max 448) */
  MMA_E5M2 = 4, /* OCP FP8 E5M2 (bias 15, IEEE-style inf/NaN) */
  MMA_I8 = 5,   /* signed 8-bit integer */
  MMA_F32 = 6,  /* IEEE binary32 (C and D of float inputs) */
  MMA_I32 = 7,  /* signed 32-bit integer (C and D of 8-bit integer inputs) */
  MMA_U8 = 8    /* unsigned 8-bit integer ("RDNA3 dense WMMA builtins", section
                   "Common parameters": a_neg / b_neg false reads an integer
                   operand as unsigned; each operand chooses on its own) */
} mma_dtype_t;

/* Types of one call: A, B, and the accumulator (the type of both C and D).
 * Accepted: (F16,F16,F32), (BF16,BF16,F32), {I8,U8} x {I8,U8} -> I32 (each
 * integer operand signed or unsigned on its own; exact, wrapping modulo 2^32 like
 * i32 arithmetic), and {E4M3,E5M2} x {E4M3,E5M2} -> F32.  mma_gemm also takes the
 * half-precision accumulate forms (F16,F16,F16) and (BF16,BF16,BF16) ("RDNA3 dense
 * WMMA builtins", section "Naming convention", out_type f16 / bf16): C and D are
 * then f16 / bf16 and D = round-to-nearest-even(C + A*B) with the product
 * accumulated in f32 (the pages do not fix the accumulation precision). */
typedef struct {
  int32_t a;
  int32_t b;
  int32_t acc;
} mma_dtypes_t;

typedef enum {
  MMA_OK = 0,
  MMA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad overlap */
  MMA_ERR_UNSUPPORTED = 2, /* type combination not provided */
  MMA_ERR_SHAPE = 3,       /* a size outside the supported range */
  MMA_ERR_ALIGN = 4,       /* base pointer or row pitch not 16-byte aligned */
  MMA_ERR_NOT_SPARSE = 5,  /* reserved for callers: A broke the 4:2 contract */
  MMA_ERR_TIMEOUT = 6,     /* a device-side pipeline wait ran past its limit */
  MMA_ERR_CUDA = 7         /* the CUDA runtime reported an error */
} mma_status_t;

/* D = A*B + C, dense.
 *   A  M x K elements of t.a        B  K x N elements of t.b
 *   C  M x N elements of t.acc      D  M x N elements of t.acc (may equal C)
 * Sizes: 0 <= M, N, K < 2^31.  M == 0 or N == 0 does nothing; K == 0 copies
 * C into D.  Row pitches must be multiples of 16 bytes: K * sizeof(a),
 * N * sizeof(b) and N * sizeof(acc).
 * Returns MMA_OK once the work is enqueued on `stream`. */
mma_status_t mma_gemm(const void* A, const void* B, const void* C, void* D, int64_t M, int64_t N,
                      int64_t K, mma_dtypes_t t, void* stream);

/* Options of mma_gemm_ex. */
enum { MMA_FLAG_CLAMP = 1 };

/* mma_gemm with options.  flags = 0 is mma_gemm.  MMA_FLAG_CLAMP (8-bit integer
 * types only, else MMA_ERR_UNSUPPORTED): D = the exact C + A*B saturated to the i32
 * range instead of wrapped ("RDNA3 dense WMMA builtins", section "Common
 * parameters", parameter clamp; the page's "range of the input type" is read as the
 * range of the i32 accumulator).  With clamp, K is cut into slices short enough
 * that each slice's product sum fits i32, and their sum with C is formed exactly
 * in 64 bits; this draws ksplit * M * N * 4 bytes of scratch when K needs more
 * than one slice (at least 131071 for signed x signed inputs, 65793 mixed, 33025
 * unsigned x unsigned).  Unknown flags: MMA_ERR_INVALID_ARG. */
mma_status_t mma_gemm_ex(const void* A, const void* B, const void* C, void* D, int64_t M, int64_t N,
                         int64_t K, mma_dtypes_t t, uint32_t flags, void* stream);

/* 4:2 compression of a row-major M x K matrix A of type `a` ("CDNA3 sparse
 * MFMA builtins", section "Structured sparsity (4:2 pattern)": walk K in
 * groups of four and pack the two non-zeros consecutively).
 *   vals  M x K/2 elements of `a`      idx  M x K/8 bytes
 * +0 and -0 count as zero, NaN and infinity as non-zero.  A group with fewer
 * than two non-zeros is padded with its lowest unused positions, whose values
 * are +0.  A group with more than two non-zeros keeps its two lowest; such
 * groups are counted into *d_violations (a device int32 that the call first
 * sets to zero; may be NULL).  Types: F16, BF16, E4M3, E5M2, I8, U8.  0 <= M, K <
 * 2^31 and K must be a multiple of 32. */
mma_status_t sparse42_compress(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K,
                               mma_dtype_t a, int32_t* d_violations, void* stream);

/* Pruning to 4:2, then compression: the step before the path when A is dense
 * (the pages assume A arrives already 4:2, "CDNA3 sparse MFMA builtins",
 * section "Structured sparsity (4:2 pattern)", so the rule is this library's
 * reading).  In every group of four along K the two elements of largest
 * magnitude are kept, the lower position on equal magnitude; floating types
 * rank by the bit pattern with the sign cleared (|x| for finite values,
 * infinity above them, NaN above infinity), I8 by |v| (-128 ranks 128), U8 by v.  Kept
 * elements of zero magnitude are stored as +0, so on a matrix that already
 * obeys 4:2 the output equals sparse42_compress's.  vals, idx, types, shapes
 * and alignment as sparse42_compress; *d_dropped (a device int32 that the call
 * first sets to zero; may be NULL) receives the number of groups that lost a
 * non-zero element.  No counterpart for the pruning rule exists on the pages. */
mma_status_t sparse42_prune(const void* A, void* vals, uint8_t* idx, int64_t M, int64_t K,
                            mma_dtype_t a, int32_t* d_dropped, void* stream);

/* Quantisation of f32 inputs to a floating storage type, the step before the
 * path that the workloads' input recipes describe ("saturated and rounded to
 * their fp8 format"; the pages give no rounding rule, so this is the library's
 * reading): y[i] = round-to-nearest-even(clamp(x[i], -max, +max)) where max is
 * the largest finite value of `t`; NaN stays NaN (bit pattern unspecified); a
 * value that rounds to zero keeps its sign.  Types: F16, BF16, E4M3, E5M2.
 *   x  n f32 values          y  n elements of `t`
 * Both 16-byte aligned and not overlapping; any n >= 0.  No counterpart for the
 * rounding rule exists on the pages. */
mma_status_t mma_quantize(const float* x, void* y, int64_t n, mma_dtype_t t, void* stream);

/* mma_quantize fused ahead of sparse42_prune: a row-major M x K f32 A is
 * quantised to `t` (F16, BF16, E4M3, E5M2; the rule of mma_quantize), pruned to
 * 4:2 by the magnitude of the quantised values (the rule of sparse42_prune) and
 * compressed, in one pass over A.  The result equals sparse42_prune applied to
 * mma_quantize(A).  vals (M x K/2 of `t`), idx, d_dropped, K % 32 == 0 and the
 * alignment rules as sparse42_prune; A is 16-byte aligned.  No counterpart on the
 * pages (the step before the path). */
mma_status_t sparse42_quantize_prune(const float* A, void* vals, uint8_t* idx, int64_t M, int64_t K,
                                     mma_dtype_t t, int32_t* d_dropped, void* stream);

/* D = A*B + C with A given compressed as (vals, idx) from sparse42_compress;
 * K is the uncompressed length and must be a multiple of 128 (the idx row
 * pitch K/8 must be a multiple of 16 bytes).  Types: (F16,F16,F32),
 * (BF16,BF16,F32), {I8,U8} x {I8,U8} -> I32 (exact, wrapping like mma_gemm)
 * and {E4M3,E5M2} x {E4M3,E5M2} -> F32 (the sparse variants of "CDNA3 sparse
 * MFMA builtins", section "Naming convention").  The integer forms draw scratch
 * of M*K + 2*K*N + 4*M bytes from the library's pool (an unsigned B runs as
 * B - 128 with 128 times the row sums of A added).  Other rules as mma_gemm. */
mma_status_t sparse42_gemm(const void* vals, const uint8_t* idx, const void* B, const void* C,
                           void* D, int64_t M, int64_t N, int64_t K, mma_dtypes_t t,
                           void* stream);

/* D = A*B + C for floating-point types (as mma_gemm), computed in `ksplit`
 * K slices whose f32 partial sums are kept in a fixed 32 MiB device array
 * inside the library instead of allocated memory; the slices are then summed
 * in a fixed order and C is added.  The pages have no counterpart to this
 * call: it exists for callers that may not allocate device memory where they
 * call it -- a process whose memory is owned by another framework's caching
 * allocator, a latency-critical loop where cudaMalloc/cudaFree could wait on
 * device-wide synchronisation, a runtime that forbids allocation after
 * start-up.  It calls no allocator.
 *   Types: (F16,F16,F32), (BF16,BF16,F32), FP8 x FP8 -> F32 (i8 is rejected
 *   with MMA_ERR_UNSUPPORTED).  Layout, alignment and aliasing rules as mma_gemm.
 *   A, B, C, D and `stream` must belong to the current device (the array used
 *   is the current device's); a D that is not device memory of the current
 *   device returns MMA_ERR_INVALID_ARG.
 *   Limits: 2 <= ksplit <= 16, ksplit <= the number of K blocks (64 elements
 *   for 16-bit inputs, 128 for FP8), and ksplit * M * N * 4 <= 32 MiB; a call
 *   beyond them returns MMA_ERR_SHAPE and launches nothing.  Unlike mma_gemm,
 *   K == 0 is therefore rejected (MMA_ERR_SHAPE); M == 0 or N == 0 is MMA_OK.
 *   The array is shared by every call on a device and keeps the last call's
 *   contents (no part of it needs clearing: each call writes every partial it
 *   reads).  Calls whose work overlaps on the GPU race on it.
 *   The first call on each device performs a one-time set-up (it looks up the
 *   array's device address); make that first call before any stream capture. */
mma_status_t mma_gemm_splitk_noalloc(const void* A, const void* B, const void* C, void* D, int64_t M,
                                     int64_t N, int64_t K, mma_dtypes_t t, int32_t ksplit, void* stream);

/* Synchronises `stream`, then returns and clears the device error word
 * (MMA_ERR_TIMEOUT if any kernel gave up on a pipeline wait since the last
 * call), or MMA_ERR_CUDA if the runtime reports an error. */
mma_status_t mma_sync_status(void* stream);

/* A static, human-readable name for a status code. */
const char* mma_status_string(mma_status_t s);

/* MMA42_ABI_VERSION of the built library. */
int32_t mma_abi_version(void);

/* Upper bound, in nanoseconds, on every wait inside the pipelined kernels
 * (default 2e9).  A kernel whose wait runs past it stops, records
 * MMA_ERR_TIMEOUT and exits cleanly.  Applies to later launches. */
void mma_set_wait_limit_ns(uint64_t ns);

/* Number of CUDA kernels this library has launched in this process (all
 * devices), for accounting by benchmarks and tests. */
uint64_t mma_launch_count(void);

/* Measurement helper, not part of the GEMM path: the throughput ceiling, in ops/s
 * (2 per multiply-add, logical K for the sparse kind), of the warp-level
 * tensor-core instructions that sm_103a keeps beside tcgen05, measured now on
 * every SM with operands in registers and no memory traffic.  `kind`: 0
 * mma.sync m16n8k32 s8 x s8 -> s32 (the only tensor instruction with an 8-bit
 * integer multiply on this architecture; tcgen05.mma has no integer kind here),
 * 1 mma.sp m16n8k64 s8 4:2-sparse, 2 mma.sync m16n8k16 bf16, 3 mma.sync
 * m16n8k32 E4M3.  Runs for about 25 ms on `stream` and waits for it.  Returns
 * MMA_ERR_INVALID_ARG for another kind or a null `ops_per_s`. */
mma_status_t mma_legacy_mma_peak(int32_t kind, double* ops_per_s, void* stream);

/* Measurement helper, not part of the GEMM path: the throughput ceiling of
 * tcgen05.mma, measured now.  Every SM pair issues one pipeline stage's MMAs of the
 * CTA-pair GEMM kernels (same tile layouts and instruction shapes, M = N = 256)
 * over and over on operands resident in shared memory: no TMA traffic, no
 * epilogue.  `kind`: 0 kind::f16 dense (bf16), 1 kind::f8f6f4 dense (E4M3), 2
 * kind::f16 4:2-sparse, 3 kind::f8f6f4 4:2-sparse (the index names positions
 * {0, 1} of every group).  *ops_per_s receives ops per second (2 per
 * multiply-add, logical K for the sparse kinds) over the whole launch;
 * *ops_per_clk_sm (nullable) the ops per SM clock cycle per SM, counted on the SMs
 * from the first MMA to the completion of the last, which does not depend on the
 * clock the power limit allows.  Runs for about 25 ms on `stream` and waits for
 * it.  Returns MMA_ERR_INVALID_ARG for another kind or a null `ops_per_s`; a wait
 * that runs out is reported by mma_sync_status like the GEMMs' (ABI 4). */
mma_status_t mma_tcgen05_peak(int32_t kind, double* ops_per_s, double* ops_per_clk_sm, void* stream);

/* Measurement helper, not part of the GEMM path: how fast TMA fills the CTA-pair
 * kernels' pipeline ring, measured now with nothing consuming the data.  Every SM
 * pair (at most `clusters`, 0: as many as fit) runs the pair kernels' producer
 * loop alone: per stage, both CTAs load `nbox` boxes (box b: box_rows[b] rows of
 * box_row_bytes[b] bytes; 64-byte rows 64-byte swizzled, 128-byte rows 128-byte
 * swizzled, 256-byte rows unswizzled) with the pair form of the tiled TMA load,
 * completing on the first CTA's barrier, and one thread of that CTA hands each
 * filled stage straight back; `stages` stages form the ring.  The source is a
 * `src_bytes` device buffer drawn from the library's pool (one quarter per box;
 * a buffer that fits in L2 measures the L2 -> shared memory feed).
 * *bytes_per_clk_sm receives the bytes one SM receives per SM clock cycle, and
 * *rows_per_clk_sm (nullable) the box rows, both counted on the SMs (clock64) over
 * about 10 ms after a warm-up launch.  Limits: 1 <= nbox <= 4, rows a multiple of
 * 8 in [8, 256], row bytes 64, 128 or 256, every box a multiple of 1024 bytes,
 * stages >= 2 and the ring within 227
 * KB of shared memory, src_bytes / 4 at least 512 rows of 16384 bytes; otherwise
 * MMA_ERR_INVALID_ARG or MMA_ERR_SHAPE.  Waits for the stream (ABI 5). */
mma_status_t mma_tma_feed_probe(int32_t nbox, const int32_t* box_rows, const int32_t* box_row_bytes, int32_t stages,
                                int32_t clusters, int64_t src_bytes, double* bytes_per_clk_sm,
                                double* rows_per_clk_sm, void* stream);

/* Test hook.  `mode` 1: the next launch of the one-SM dense kernel arms its first
 * pipeline stage but never issues that stage's loads.  `mode` 2: the next launch
 * of a CTA-pair kernel (dense mma_gemm on the pair kernel, or sparse42_gemm) has
 * its first cluster arm its first stage for 16 bytes more than that stage's loads
 * bring (every load is issued and lands).  `mode` 3: the next launch of the short-K
 * kernel (mma_gemm with K of at most four k-blocks) has its first block arm its
 * first k-block for 16 bytes more than its loads bring.  Either way that stage never completes,
 * the MMA thread's bounded wait runs out and the timeout path is exercised
 * (MMA_ERR_TIMEOUT from mma_sync_status).  The hook disarms itself when a launch
 * of its kind takes it; 0 disarms it. */
void mma_debug_inject(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* MMA42_H */
