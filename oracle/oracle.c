/*
 * oracle.c -- the plain, slow CPU oracle for D = A*B + C, dense and 4:2-sparse.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; its element-type codes are its own.
 *
 * What it computes, and where the pages say so:
 *
 *  - Dense MMA semantics.  "CDNA dense MFMA builtins", section "Naming
 *    convention": an instruction multiplies an M x K panel of A by a K x N panel
 *    of B and accumulates into an M x N tile of C; the caller loops over K.
 *    Written out for whole matrices this is the plain definition
 *        D[i][j] = C[i][j] + sum_{k<K} A[i][k] * B[k][j],
 *    which the oracle evaluates with a for-i / for-k / for-j loop, in double
 *    precision for floating inputs and in 64-bit integers for i8 inputs, after
 *    decoding the exact input bit patterns the GPU receives.
 *
 *  - 4:2 structured sparsity.  "CDNA3 sparse MFMA builtins", section
 *    "Structured sparsity (4:2 pattern)": every contiguous group of four A
 *    elements along K holds exactly two non-zeros; the compressed A keeps only
 *    those (K/2 long) and an index records which two of the four positions
 *    they came from; host-side compression walks K in groups of four and packs
 *    the two non-zeros consecutively.  The same page, section "Using sparse
 *    MFMA builtins as a compute policy", gives the index of the keep-{0,2}
 *    pattern as 0x88 for the FP16 variant and 0x8888 for the FP8 variant.
 *
 *    Reading taken for the index (consistent with both constants): each kept
 *    element's position 0..3 takes two bits; a group's nibble is p0 | p1 << 2
 *    with p0 < p1 (keep {0,2} -> 0x8); groups run along K from the least
 *    significant nibble of byte 0, two groups per byte, so a row of K logical
 *    elements has K/8 index bytes.  Values of a group are stored in ascending
 *    position order.
 *
 *    Readings for cases the pages leave open: +0 and -0 are "zero", NaN and
 *    infinity are non-zero.  A group with fewer than two non-zeros is padded
 *    with the lowest unused positions and the padded slots hold +0.  A group
 *    with more than two non-zeros violates the contract: the two lowest
 *    positions are kept and the violation is counted.
 *
 *  - Pruning to 4:2 (the step before the path for a dense A; the same page
 *    assumes A arrives already 4:2, so the rule is this oracle's reading): in
 *    every group keep the two elements of largest magnitude, the lower
 *    position on equal magnitude; infinity ranks above finite values and NaN
 *    above infinity; kept zeros are stored as +0.
 *
 *  - The sparse product is computed directly from (vals, idx), without
 *    decompressing: D[i][j] = C[i][j] + sum_g sum_t vals[i][2g+t] *
 *    B[4g + p_t(i,g)][j]; this is the realignment of compressed A against the
 *    rows of B that the "Structured sparsity (4:2 pattern)" section describes.
 *
 *  - Quantisation of f32 inputs (the step before the path that the workloads'
 *    input recipes describe): saturate to the largest finite magnitude, round to
 *    nearest, ties to the even code; NaN stays NaN.
 *
 *  - Element formats (written from the format definitions, not from any
 *    library): IEEE binary16; bfloat16 (the upper half of binary32); OCP FP8
 *    E4M3 (bias 7, no infinities, S.1111.111 is NaN, max 448) and OCP FP8 E5M2
 *    (bias 15, IEEE-style infinities and NaNs).  The sparse page's note on FP8
 *    encodings says later architectures use the OCP format rather than FNUZ;
 *    the OCP reading is taken.
 *
 * Loops are deliberately unblocked.  OpenMP parallelises over output rows
 * only, which does not change any result (each row is computed by one thread
 * in the same order).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element-type codes of the oracle (its own numbering). */
enum {
  ORC_F16 = 1,
  ORC_BF16 = 2,
  ORC_E4M3 = 3,
  ORC_E5M2 = 4,
  ORC_I8 = 5,
  ORC_F32 = 6,
  ORC_I32 = 7,
  ORC_U8 = 8
};

enum { ORC_OK = 0, ORC_BAD_TYPE = -1, ORC_BAD_SHAPE = -2, ORC_NO_MEM = -3 };

/* ------------------------------------------------------------------ decoders */

static double decode_binary16(uint32_t h) {
  uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
  double sign = s ? -1.0 : 1.0;
  if (e == 0) return sign * ldexp((double)m, -24);          /* subnormal: m/2^10 * 2^-14 */
  if (e == 31) return m == 0 ? sign * INFINITY : NAN;
  return sign * ldexp((double)(1024u + m), (int)e - 25);    /* (1 + m/2^10) * 2^(e-15) */
}

static double decode_bfloat16(uint32_t h) {
  uint32_t s = (h >> 15) & 1u, e = (h >> 7) & 0xffu, m = h & 0x7fu;
  double sign = s ? -1.0 : 1.0;
  if (e == 0) return sign * ldexp((double)m, -133);         /* m/2^7 * 2^-126 */
  if (e == 255) return m == 0 ? sign * INFINITY : NAN;
  return sign * ldexp((double)(128u + m), (int)e - 134);    /* (1 + m/2^7) * 2^(e-127) */
}

static double decode_e4m3(uint32_t b) {
  uint32_t s = (b >> 7) & 1u, e = (b >> 3) & 0xfu, m = b & 0x7u;
  double sign = s ? -1.0 : 1.0;
  if (e == 15 && m == 7) return NAN;                        /* only NaN; no infinities */
  if (e == 0) return sign * ldexp((double)m, -9);           /* m/8 * 2^(1-7) */
  return sign * ldexp((double)(8u + m), (int)e - 10);       /* (1 + m/8) * 2^(e-7) */
}

static double decode_e5m2(uint32_t b) {
  uint32_t s = (b >> 7) & 1u, e = (b >> 2) & 0x1fu, m = b & 0x3u;
  double sign = s ? -1.0 : 1.0;
  if (e == 31) return m == 0 ? sign * INFINITY : NAN;
  if (e == 0) return sign * ldexp((double)m, -16);          /* m/4 * 2^(1-15) */
  return sign * ldexp((double)(4u + m), (int)e - 17);       /* (1 + m/4) * 2^(e-15) */
}

static int elem_bytes(int t) {
  switch (t) {
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_E4M3: case ORC_E5M2: case ORC_I8: case ORC_U8: return 1;
    case ORC_F32: case ORC_I32: return 4;
    default: return 0;
  }
}

/* Raw bit pattern of element n of an array of type t. */
static uint32_t load_bits(const void* p, int t, int64_t n) {
  switch (elem_bytes(t)) {
    case 1: return ((const uint8_t*)p)[n];
    case 2: return ((const uint16_t*)p)[n];
    default: return ((const uint32_t*)p)[n];
  }
}

double oracle_decode(int t, uint32_t bits) {
  switch (t) {
    case ORC_F16: return decode_binary16(bits);
    case ORC_BF16: return decode_bfloat16(bits);
    case ORC_E4M3: return decode_e4m3(bits);
    case ORC_E5M2: return decode_e5m2(bits);
    case ORC_I8: return (double)(int8_t)(uint8_t)bits;
    case ORC_U8: return (double)(uint8_t)bits;
    case ORC_F32: { float f; uint32_t u = bits; memcpy(&f, &u, 4); return (double)f; }
    case ORC_I32: return (double)(int32_t)bits;
    default: return NAN;
  }
}

int oracle_decode_array(int t, const void* src, double* dst, int64_t n) {
  if (elem_bytes(t) == 0) return ORC_BAD_TYPE;
  for (int64_t i = 0; i < n; ++i) dst[i] = oracle_decode(t, load_bits(src, t, i));
  return ORC_OK;
}

/* A decode table over every bit pattern of an 8- or 16-bit type. */
static double* make_table(int t) {
  int nb = elem_bytes(t);
  if (nb != 1 && nb != 2) return NULL;
  size_t n = (size_t)1 << (8 * nb);
  double* tab = (double*)malloc(n * sizeof(double));
  if (!tab) return NULL;
  for (size_t v = 0; v < n; ++v) tab[v] = oracle_decode(t, (uint32_t)v);
  return tab;
}

static int is_float_input(int t) {
  return t == ORC_F16 || t == ORC_BF16 || t == ORC_E4M3 || t == ORC_E5M2;
}

/* ---------------------------------------------------------------- dense GEMM */

/*
 * D = A*B + C in double.  A: M x K row-major, B: K x N row-major, C: M x N f32
 * row-major.  rows == NULL computes every row into D (M x N); otherwise the
 * nrows listed rows, into D (nrows x N).
 */
int oracle_gemm_f64(const void* A, int ta, const void* B, int tb, const float* C,
                    double* D, int64_t M, int64_t N, int64_t K,
                    const int64_t* rows, int64_t nrows) {
  if (!is_float_input(ta) || !is_float_input(tb)) return ORC_BAD_TYPE;
  if (M < 0 || N < 0 || K < 0) return ORC_BAD_SHAPE;
  if (!rows) nrows = M;
  double* ta_tab = make_table(ta);
  double* tb_tab = make_table(tb);
  if (!ta_tab || !tb_tab) { free(ta_tab); free(tb_tab); return ORC_NO_MEM; }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc) { bad = 1; continue; }
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double a = ta_tab[load_bits(A, ta, i * K + k)];
      for (int64_t j = 0; j < N; ++j) acc[j] += a * tb_tab[load_bits(B, tb, k * N + j)];
    }
    for (int64_t j = 0; j < N; ++j) D[r * N + j] = (double)C[i * N + j] + acc[j];
    free(acc);
  }
  free(ta_tab);
  free(tb_tab);
  return bad ? ORC_NO_MEM : ORC_OK;
}

/*
 * Value of an 8-bit integer element.  "RDNA3 dense WMMA builtins", section
 * "Common parameters" (parameters a_neg / b_neg): integer operands are read as
 * signed or unsigned per operand; ORC_I8 is the signed reading, ORC_U8 the
 * unsigned one.
 */
static int64_t int_value(int t, uint32_t bits) {
  if (t == ORC_U8) return (int64_t)(uint8_t)bits;
  return (int64_t)(int8_t)(uint8_t)bits;
}

static int is_int8_type(int t) { return t == ORC_I8 || t == ORC_U8; }

/* D = A*B + C exactly, in 64-bit integers (8-bit A and B, each signed or
 * unsigned; i32 C). */
int oracle_gemm_i64(const void* A, int ta, const void* B, int tb, const int32_t* C, int64_t* D,
                    int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows) {
  if (!is_int8_type(ta) || !is_int8_type(tb)) return ORC_BAD_TYPE;
  if (M < 0 || N < 0 || K < 0) return ORC_BAD_SHAPE;
  if (!rows) nrows = M;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    int64_t* acc = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!acc) { bad = 1; continue; }
    for (int64_t j = 0; j < N; ++j) acc[j] = 0;
    for (int64_t k = 0; k < K; ++k) {
      int64_t a = int_value(ta, load_bits(A, ta, i * K + k));
      for (int64_t j = 0; j < N; ++j) acc[j] += a * int_value(tb, load_bits(B, tb, k * N + j));
    }
    for (int64_t j = 0; j < N; ++j) D[r * N + j] = (int64_t)C[i * N + j] + acc[j];
    free(acc);
  }
  return bad ? ORC_NO_MEM : ORC_OK;
}

/* ------------------------------------------------------- 4:2 compress/expand */

static int is_zero(int t, uint32_t bits) {
  switch (t) {
    case ORC_F16: case ORC_BF16: return (bits & 0x7fffu) == 0;   /* +0 or -0 */
    case ORC_E4M3: case ORC_E5M2: return (bits & 0x7fu) == 0;
    case ORC_I8: case ORC_U8: return (bits & 0xffu) == 0;
    default: return 0;
  }
}

static void store_bits(void* p, int t, int64_t n, uint32_t v) {
  if (elem_bytes(t) == 1) ((uint8_t*)p)[n] = (uint8_t)v;
  else ((uint16_t*)p)[n] = (uint16_t)v;
}

/* Write group g's nibble of row i: two groups per byte, the even group low. */
static void put_nibble(uint8_t* idx, int64_t K, int64_t i, int64_t g, uint32_t nib) {
  uint8_t* byte = &idx[i * (K / 8) + g / 2];
  if (g % 2 == 0) *byte = (uint8_t)((*byte & 0xf0u) | nib);
  else *byte = (uint8_t)((*byte & 0x0fu) | (nib << 4));
}

/*
 * Compress an M x K row-major A obeying 4:2 sparsity into vals (M x K/2, same
 * type) and idx (M x K/8 bytes).  K must be a multiple of 8.  *violations
 * receives the number of groups that held more than two non-zeros.
 */
int oracle_compress(const void* A, int ta, int64_t M, int64_t K, void* vals,
                    uint8_t* idx, int64_t* violations) {
  int nb = elem_bytes(ta);
  if (nb != 1 && nb != 2) return ORC_BAD_TYPE;
  if (M < 0 || K < 0 || K % 8 != 0) return ORC_BAD_SHAPE;
  int64_t viol = 0;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t g = 0; g < K / 4; ++g) {
      int pos[4], n = 0;
      for (int p = 0; p < 4; ++p)
        if (!is_zero(ta, load_bits(A, ta, i * K + 4 * g + p))) pos[n++] = p;
      if (n > 2) { viol++; n = 2; }              /* keep the two lowest positions */
      int keep[2];
      uint32_t v[2];
      if (n == 2) {
        keep[0] = pos[0]; keep[1] = pos[1];
        v[0] = load_bits(A, ta, i * K + 4 * g + keep[0]);
        v[1] = load_bits(A, ta, i * K + 4 * g + keep[1]);
      } else {
        /* pad with the lowest unused positions; padded slots hold +0 */
        int used[4] = {0, 0, 0, 0}, m = 0;
        int chosen[2];
        uint32_t cv[2];
        for (int q = 0; q < n; ++q) used[pos[q]] = 1;
        for (int q = 0; q < n; ++q) { chosen[m] = pos[q]; cv[m] = load_bits(A, ta, i * K + 4 * g + pos[q]); m++; }
        for (int p = 0; p < 4 && m < 2; ++p)
          if (!used[p]) { chosen[m] = p; cv[m] = 0u; m++; }
        if (chosen[0] < chosen[1]) { keep[0] = chosen[0]; keep[1] = chosen[1]; v[0] = cv[0]; v[1] = cv[1]; }
        else { keep[0] = chosen[1]; keep[1] = chosen[0]; v[0] = cv[1]; v[1] = cv[0]; }
      }
      store_bits(vals, ta, i * (K / 2) + 2 * g, v[0]);
      store_bits(vals, ta, i * (K / 2) + 2 * g + 1, v[1]);
      put_nibble(idx, K, i, g, (uint32_t)keep[0] | ((uint32_t)keep[1] << 2));
    }
  }
  if (violations) *violations = viol;
  return ORC_OK;
}

/*
 * Magnitude rank of one element for pruning (larger is kept first).  Floating
 * types: the bit pattern with the sign cleared, which orders |x| for finite
 * values and puts infinity above every finite value and NaN above infinity.
 * i8: |v|, so -128 ranks 128; u8: v.
 */
static uint32_t prune_rank(int t, uint32_t bits) {
  switch (t) {
    case ORC_F16: case ORC_BF16: return bits & 0x7fffu;
    case ORC_E4M3: case ORC_E5M2: return bits & 0x7fu;
    case ORC_I8: {
      int v = (int)(int8_t)(uint8_t)bits;
      return (uint32_t)(v < 0 ? -v : v);
    }
    case ORC_U8: return bits & 0xffu;
    default: return 0u;
  }
}

/*
 * Prune a dense M x K row-major A to 4:2 and compress it: in every group of four
 * along K keep the two elements of largest magnitude (prune_rank; on equal
 * rank the lower position), in the index and value layout of oracle_compress.
 * A kept element of zero magnitude is stored as +0, as compression pads, so on
 * input that already obeys 4:2 the result equals oracle_compress's.  *dropped
 * receives the number of groups that lost a non-zero element.
 */
int oracle_prune(const void* A, int ta, int64_t M, int64_t K, void* vals, uint8_t* idx,
                 int64_t* dropped) {
  int nb = elem_bytes(ta);
  if (nb != 1 && nb != 2) return ORC_BAD_TYPE;
  if (M < 0 || K < 0 || K % 8 != 0) return ORC_BAD_SHAPE;
  int64_t lost = 0;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t g = 0; g < K / 4; ++g) {
      uint32_t bits[4], rank[4];
      int nonzero = 0;
      for (int p = 0; p < 4; ++p) {
        bits[p] = load_bits(A, ta, i * K + 4 * g + p);
        rank[p] = prune_rank(ta, bits[p]);
        if (!is_zero(ta, bits[p])) nonzero++;
      }
      /* first pick: the largest rank, the lowest position among equals */
      int first = 0;
      for (int p = 1; p < 4; ++p)
        if (rank[p] > rank[first]) first = p;
      /* second pick: the same over the other three positions */
      int second = -1;
      for (int p = 0; p < 4; ++p) {
        if (p == first) continue;
        if (second < 0 || rank[p] > rank[second]) second = p;
      }
      int keep0 = first < second ? first : second, keep1 = first < second ? second : first;
      uint32_t v0 = is_zero(ta, bits[keep0]) ? 0u : bits[keep0];
      uint32_t v1 = is_zero(ta, bits[keep1]) ? 0u : bits[keep1];
      if (nonzero > 2) lost++;
      store_bits(vals, ta, i * (K / 2) + 2 * g, v0);
      store_bits(vals, ta, i * (K / 2) + 2 * g + 1, v1);
      put_nibble(idx, K, i, g, (uint32_t)keep0 | ((uint32_t)keep1 << 2));
    }
  }
  if (dropped) *dropped = lost;
  return ORC_OK;
}

/* Position t (0 or 1) of group g in row i, read from the index. */
static int idx_pos(const uint8_t* idx, int64_t K, int64_t i, int64_t g, int t) {
  uint32_t byte = idx[i * (K / 8) + g / 2];
  uint32_t nib = (g % 2 == 0) ? (byte & 0xfu) : (byte >> 4);
  return (int)((nib >> (2 * t)) & 3u);
}

/* Expand (vals, idx) back to the M x K dense A; unlisted positions get +0. */
int oracle_decompress(const void* vals, const uint8_t* idx, int ta, int64_t M, int64_t K,
                      void* A) {
  int nb = elem_bytes(ta);
  if (nb != 1 && nb != 2) return ORC_BAD_TYPE;
  if (M < 0 || K < 0 || K % 8 != 0) return ORC_BAD_SHAPE;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t k = 0; k < K; ++k) store_bits(A, ta, i * K + k, 0u);
  for (int64_t i = 0; i < M; ++i)
    for (int64_t g = 0; g < K / 4; ++g)
      for (int t = 0; t < 2; ++t) {
        int p = idx_pos(idx, K, i, g, t);
        store_bits(A, ta, i * K + 4 * g + p, load_bits(vals, ta, i * (K / 2) + 2 * g + t));
      }
  return ORC_OK;
}

/* --------------------------------------------------------------- sparse GEMM */

/*
 * D = A*B + C with A given compressed as (vals, idx); K is the uncompressed
 * length.  Each compressed element multiplies the row of B its index names.
 */
int oracle_sparse_gemm_f64(const void* vals, const uint8_t* idx, int ta, const void* B,
                           int tb, const float* C, double* D, int64_t M, int64_t N,
                           int64_t K, const int64_t* rows, int64_t nrows) {
  if (!is_float_input(ta) || !is_float_input(tb)) return ORC_BAD_TYPE;
  if (M < 0 || N < 0 || K < 0 || K % 8 != 0) return ORC_BAD_SHAPE;
  if (!rows) nrows = M;
  double* ta_tab = make_table(ta);
  double* tb_tab = make_table(tb);
  if (!ta_tab || !tb_tab) { free(ta_tab); free(tb_tab); return ORC_NO_MEM; }
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc) { bad = 1; continue; }
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    for (int64_t g = 0; g < K / 4; ++g)
      for (int t = 0; t < 2; ++t) {
        double a = ta_tab[load_bits(vals, ta, i * (K / 2) + 2 * g + t)];
        int64_t k = 4 * g + idx_pos(idx, K, i, g, t);
        for (int64_t j = 0; j < N; ++j) acc[j] += a * tb_tab[load_bits(B, tb, k * N + j)];
      }
    for (int64_t j = 0; j < N; ++j) D[r * N + j] = (double)C[i * N + j] + acc[j];
    free(acc);
  }
  free(ta_tab);
  free(tb_tab);
  return bad ? ORC_NO_MEM : ORC_OK;
}

int oracle_sparse_gemm_i64(const void* vals, int ta, const uint8_t* idx, const void* B, int tb,
                           const int32_t* C, int64_t* D, int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, int64_t nrows) {
  if (!is_int8_type(ta) || !is_int8_type(tb)) return ORC_BAD_TYPE;
  if (M < 0 || N < 0 || K < 0 || K % 8 != 0) return ORC_BAD_SHAPE;
  if (!rows) nrows = M;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    int64_t* acc = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!acc) { bad = 1; continue; }
    for (int64_t j = 0; j < N; ++j) acc[j] = 0;
    for (int64_t g = 0; g < K / 4; ++g)
      for (int t = 0; t < 2; ++t) {
        int64_t a = int_value(ta, load_bits(vals, ta, i * (K / 2) + 2 * g + t));
        int64_t k = 4 * g + idx_pos(idx, K, i, g, t);
        for (int64_t j = 0; j < N; ++j) acc[j] += a * int_value(tb, load_bits(B, tb, k * N + j));
      }
    for (int64_t j = 0; j < N; ++j) D[r * N + j] = (int64_t)C[i * N + j] + acc[j];
    free(acc);
  }
  return bad ? ORC_NO_MEM : ORC_OK;
}

/* ------------------------------------------------------------- quantisation */

/*
 * Quantise f32 values to a floating storage type, the step before the path that
 * the workloads' input recipes describe ("saturated and rounded to their fp8
 * format"): clamp to the largest finite magnitude of the type, then round to the
 * nearest representable value, ties to the even code.  Written as a search over
 * the type's codes (decoded with this file's own decoders), not from any
 * conversion routine.  NaN maps to a NaN of the type (its bits are not part of
 * the reading); a zero or a value that rounds to zero keeps its sign.
 */
static int quant_bits(int t) { return elem_bytes(t) * 8; }

/* Largest finite value of type t: the largest positive code that decodes finite. */
static double max_finite(int t) {
  uint32_t top = (1u << (quant_bits(t) - 1)) - 1u;   /* sign clear, all other bits set */
  for (uint32_t c = top;; --c) {
    double v = oracle_decode(t, c);
    if (isfinite(v)) return v;
    if (c == 0) return 0.0;
  }
}

/* tab: the decoded value of every code of t (make_table) */
static uint32_t quantize_one(int t, const double* tab, double mx, double x) {
  const uint32_t sign_bit = 1u << (quant_bits(t) - 1);
  if (isnan(x)) {
    for (uint32_t c = sign_bit - 1u;; --c)   /* the first NaN code from the top */
      if (isnan(tab[c])) return c;
  }
  const uint32_t sign = signbit(x) ? sign_bit : 0u;
  double a = fabs(x);
  if (a > mx) a = mx;
  /* nearest non-negative finite code; codes of one sign increase with the value */
  uint32_t best = 0u;
  double best_d = INFINITY;
  for (uint32_t c = 0; c < sign_bit; ++c) {
    double v = tab[c];
    if (!isfinite(v)) break;
    double d = fabs(v - a);
    if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
      best = c;
      best_d = d;
    }
  }
  return sign | best;
}

int oracle_quantize(const float* x, int t, int64_t n, void* y) {
  if (!is_float_input(t)) return ORC_BAD_TYPE;
  if (n < 0) return ORC_BAD_SHAPE;
  double* tab = make_table(t);
  if (!tab) return ORC_NO_MEM;
  const double mx = max_finite(t);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) store_bits(y, t, i, quantize_one(t, tab, mx, (double)x[i]));
  free(tab);
  return ORC_OK;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
