/*
 * W12 oracle: a plain, slow, obviously correct CPU implementation of the W12
 * lossless 12-bit weight format and of the GEMM that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is used by the test suite, by the
 * smoke check and by the CPU-baseline leg of the benchmark.  It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Source: "SpecPilot: Autonomous Algorithm Discovery and Systems Optimization
 * for Speculative Decoding" (arXiv 2611.02501), section 4.1 (W12):
 *   - each BF16 weight is stored as a sign bit, a 4-bit exponent offset inside
 *     a window of 16 binades chosen per output channel, and the 7 BF16
 *     mantissa bits;
 *   - weights outside the window, zeros and denormals go to an exact escape
 *     list;
 *   - decode restores every tensor bit for bit (checked at load time);
 *   - the GEMM multiplies BF16 activations by the decoded weights with FP32
 *     accumulation (here: the exact FP64 sum, rounded once to BF16).
 * The news-article page of the same paper, part "(1) W12", adds that the
 * window works because BF16 exponents of one output channel are concentrated
 * and that out-of-range weights come back exactly from a sparse list; its part
 * "(3) two-level verification" names the 8-bit view nested in W12, which is
 * why the top 8 bits of every record form a plane of their own.
 *
 * Readings where the pages are silent (each one is stated again where used):
 *   R1 record bit order s|off|m, hi byte = s|off|m[6:4], lo nibble = m[3:0];
 *   R2 window = the 16 binades holding the most normal finite weights of the
 *      row, ties to the largest base;
 *   R3 base in [1,239] so that base+off <= 254 is always a finite normal;
 *   R4 Inf/NaN (exponent 255) are escaped too;
 *   R5 escaped and padding slots hold record 0;
 *   R6 escape list = 32-bit entries key<<16 | raw BF16 bits, ordered
 *      by row stripe (16 rows), then 256-column group, then tile, row and
 *      column; esc_ptr[t*G+g] is the index of the first entry of stripe t,
 *      group g (G = groups per stripe), esc_ptr[T*G] = the entry count.  The
 *      key of weight (n,k) inside its group is (k%256/64)<<10 | (n%16)<<6 | k%64;
 *   R7 an output channel is a row of W[N,K] (Y = A * W^T);
 *   R8 planes are padded to Np = N rounded up to 16 and Kp = K rounded up to
 *      256 (whole escape groups of 4 tiles) and stored tile by tile (16 rows x
 *      64 columns); the in-tile order is fixed by w12ref_hi_offset /
 *      w12ref_lo_position below;
 *   R24 the fused gate/up epilogue silu(g) * u (not on the pages): gate row
 *      16t+i and up row 16t+8+i of stripe t give hidden unit 8t+i.
 *
 * All functions return 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_ERR_INVALID (-1)
#define REF_ERR_CAPACITY (-3)
#define REF_ERR_MISMATCH (-5)
#define REF_ERR_CORRUPT (-7)

/* ---- BF16 fields (IEEE layout: 1 sign, 8 exponent, 7 mantissa bits) ---- */
static int bf_sign(uint16_t b) { return (b >> 15) & 1; }
static int bf_exp(uint16_t b) { return (b >> 7) & 0xFF; }
static int bf_man(uint16_t b) { return b & 0x7F; }

/* Value of a BF16 bit pattern as a double (exact). */
double w12ref_bf16_to_double(uint16_t b)
{
    int s = bf_sign(b), e = bf_exp(b), m = bf_man(b);
    double v;
    if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -133); /* denormal: m * 2^-126 * 2^-7 */
    } else {
        v = ldexp(1.0 + (double)m / 128.0, e - 127);
    }
    return s ? -v : v;
}

/* Round a double to the nearest BF16, ties to even, with gradual underflow
 * and overflow to infinity.  NaN becomes the quiet NaN 0x7FC0 with the sign
 * of the input.  The value is rounded once, straight from the double. */
uint16_t w12ref_bf16_from_double(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return sign | 0x7FC0;
    if (isinf(x)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);     /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;          /* floor(log2(a)) */
    if (E < -126) E = -126;  /* below the normal range the quantum stays 2^-133 */
    double q = ldexp(1.0, E - 7);
    double t = a / q;        /* exact: division by a power of two */
    double r = nearbyint(t); /* default rounding mode: nearest, ties to even */
    double v = r * q;
    if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
    /* v has at most 8 significant bits and lies in the BF16 range, so it is
     * exactly a float whose low 16 bits are zero. */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ---- shape helpers (reading R8) ---- */
int64_t w12ref_rows_padded(int64_t N) { return (N + 15) / 16 * 16; }
int64_t w12ref_cols_padded(int64_t K) { return (K + 255) / 256 * 256; }
int64_t w12ref_hi_bytes(int64_t N, int64_t K) { return w12ref_rows_padded(N) * w12ref_cols_padded(K); }
int64_t w12ref_lo_bytes(int64_t N, int64_t K) { return w12ref_rows_padded(N) * w12ref_cols_padded(K) / 2; }

/* Byte of the hi plane holding the top 8 record bits of weight (n,k).
 * Tiles of 16 rows x 64 columns, stripe-major (tile (t,c) is the c-th tile of
 * row stripe t).  Inside a tile, row i and column j go to "slot"
 * L = 4*(i mod 8) + j/16; rows 0..7 fill the first 512 bytes and rows 8..15
 * the next 512; each slot holds 16 consecutive columns. */
int64_t w12ref_hi_offset(int64_t n, int64_t k, int64_t Kp)
{
    int64_t t = n / 16, c = k / 64, i = n % 16, j = k % 64;
    int64_t tile = (t * (Kp / 64) + c) * 1024;
    return tile + (i / 8) * 512 + ((i % 8) * 4 + j / 16) * 16 + (j % 16);
}

/* Byte and bit shift of the lo-plane nibble of weight (n,k).
 * Tile (t,c) is 512 bytes; slot L (as above) owns 16 bytes: 8 for row i<8
 * and 8 for row i+8.  The 16 nibbles of a slot row (columns j16 = 0..15) sit
 * in two 32-bit little-endian words (j16/8); inside a word, column u (0..7)
 * is the high nibble of byte u when u < 4 and the low nibble of byte u-4
 * otherwise. */
void w12ref_lo_position(int64_t n, int64_t k, int64_t Kp, int64_t *byte, int *shift)
{
    int64_t t = n / 16, c = k / 64, i = n % 16, j = k % 64;
    int64_t tile = (t * (Kp / 64) + c) * 512;
    int64_t L = (i % 8) * 4 + j / 16;
    int64_t j16 = j % 16, word = j16 / 8, u = j16 % 8;
    *byte = tile + L * 16 + (i / 8) * 8 + word * 4 + (u < 4 ? u : u - 4);
    *shift = (u < 4) ? 4 : 0;
}

/* ---- step a1: the per-channel window (reading R2, R3) ----
 * h[e] counts the row's normal finite weights (1 <= e <= 254); the window
 * starting at b holds cnt[b] = h[b] + ... + h[b+15]; base = the largest b in
 * [1,239] with the largest cnt. */
int w12ref_window_base(const uint16_t *row, int64_t K)
{
    int64_t h[256];
    memset(h, 0, sizeof h);
    for (int64_t k = 0; k < K; ++k) {
        int e = bf_exp(row[k]);
        if (e >= 1 && e <= 254) h[e]++;
    }
    int best_b = 1;
    int64_t best = -1;
    for (int b = 1; b <= 239; ++b) {
        int64_t cnt = 0;
        for (int e = b; e <= b + 15; ++e) cnt += h[e];
        if (cnt >= best) { /* ">=" keeps the largest b among ties */
            best = cnt;
            best_b = b;
        }
    }
    return best_b;
}

/* ---- step a2: the escape predicate (section 4.1: out-of-window weights,
 * zeros and denormals; reading R4 adds Inf/NaN) ---- */
int w12ref_is_escape(uint16_t w, int base)
{
    int e = bf_exp(w);
    return e == 0 || e == 255 || e < base || e > base + 15;
}

/* ---- step a3: the 12-bit record of an in-window weight (reading R1) ---- */
int w12ref_record(uint16_t w, int base)
{
    return (bf_sign(w) << 11) | ((bf_exp(w) - base) << 7) | bf_man(w);
}

/* Escape-list geometry (reading R6). */
int64_t w12ref_groups(int64_t K) { return w12ref_cols_padded(K) / 256; }
int64_t w12ref_ptr_len(int64_t N, int64_t K) { return w12ref_rows_padded(N) / 16 * w12ref_groups(K) + 1; }

int w12ref_key(int64_t n, int64_t k) { return (int)(((k % 256) / 64) << 10 | (n % 16) << 6 | (k % 64)); }

/* Row and column of the entry `key` of stripe t, group g. */
static void key_position(int64_t t, int64_t g, int key, int64_t *n, int64_t *k)
{
    *n = 16 * t + ((key >> 6) & 15);
    *k = 256 * g + 64 * (key >> 10) + (key & 63);
}

/* ---- step a3: encode ----
 * W is [N,K] BF16 bits with row stride ldw.  Outputs: hi [Np*Kp], lo
 * [Np*Kp/2], base [N], esc_ptr [w12ref_ptr_len(N,K)], esc [esc_cap].  When the tensor needs more than esc_cap escapes, the planes,
 * base and esc_ptr are still complete, only the first esc_cap escapes are
 * written, and the function returns REF_ERR_CAPACITY with *n_esc = the
 * number needed. */
int w12ref_encode(const uint16_t *W, int64_t N, int64_t K, int64_t ldw,
                  uint8_t *hi, uint8_t *lo, uint8_t *base, int32_t *esc_ptr,
                  uint32_t *esc, int64_t esc_cap, int64_t *n_esc)
{
    if (N < 0 || K < 0 || ldw < K || !n_esc) return REF_ERR_INVALID;
    int64_t Kp = w12ref_cols_padded(K), T = w12ref_rows_padded(N) / 16, G = w12ref_groups(K);
    memset(hi, 0, (size_t)w12ref_hi_bytes(N, K)); /* reading R5: padding = record 0 */
    memset(lo, 0, (size_t)w12ref_lo_bytes(N, K));

    /* a1: the window of every row */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t n = 0; n < N; ++n) base[n] = (uint8_t)w12ref_window_base(W + n * ldw, K);

    /* a2: escapes per (stripe, group), then their offsets */
    int64_t E = 0;
    esc_ptr[0] = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            for (int64_t n = 16 * t; n < 16 * t + 16 && n < N; ++n)
                for (int64_t k = 256 * g; k < 256 * g + 256 && k < K; ++k)
                    E += w12ref_is_escape(W[n * ldw + k], base[n]);
            esc_ptr[t * G + g + 1] = (int32_t)E;
        }
    }
    *n_esc = E;

    /* a3: records into the planes, escapes in (stripe, group, tile, row,
     * column) order */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            int64_t idx = esc_ptr[t * G + g];
            for (int64_t c4 = 0; c4 < 4; ++c4) {
                for (int64_t i = 0; i < 16; ++i) {
                    int64_t n = 16 * t + i;
                    if (n >= N) continue;
                    for (int64_t j = 0; j < 64; ++j) {
                        int64_t k = 256 * g + 64 * c4 + j;
                        if (k >= K) break;
                        uint16_t w = W[n * ldw + k];
                        int b = base[n];
                        int r;
                        if (w12ref_is_escape(w, b)) {
                            if (idx < esc_cap) esc[idx] = ((uint32_t)w12ref_key(n, k) << 16) | w;
                            idx++;
                            r = 0;
                        } else {
                            r = w12ref_record(w, b);
                        }
                        hi[w12ref_hi_offset(n, k, Kp)] = (uint8_t)(r >> 4);
                        int64_t lb;
                        int sh;
                        w12ref_lo_position(n, k, Kp, &lb, &sh);
                        lo[lb] = (uint8_t)(lo[lb] | ((r & 0xF) << sh));
                    }
                }
            }
        }
    }
    return E <= esc_cap ? REF_OK : REF_ERR_CAPACITY;
}

/* The record of weight (n,k) read back from the two planes. */
static int record_at(const uint8_t *hi, const uint8_t *lo, int64_t n, int64_t k, int64_t Kp)
{
    int64_t lb;
    int sh;
    w12ref_lo_position(n, k, Kp, &lb, &sh);
    return (hi[w12ref_hi_offset(n, k, Kp)] << 4) | ((lo[lb] >> sh) & 0xF);
}

/* BF16 bits from a record and its row base.  For a well-formed tensor
 * (base in [1,239]) this is exactly s<<15 | (off+base)<<7 | m; the exponent is
 * taken modulo 256 so that a corrupted base still gives a defined value. */
uint16_t w12ref_decode_record(int r, int base)
{
    int s = (r >> 11) & 1, off = (r >> 7) & 0xF, m = r & 0x7F;
    return (uint16_t)((s << 15) | (((off + base) & 0xFF) << 7) | m);
}

/* Escape-list well-formedness (reading R6): esc_ptr[0] = 0, non-decreasing,
 * esc_ptr[T*G] = n_esc <= esc_cap; inside each group the keys strictly
 * ascend, are below 4096 and name a weight inside the tensor.  Returns the
 * number of violations. */
int64_t w12ref_check_structure(int64_t N, int64_t K, const int32_t *esc_ptr,
                               const uint32_t *esc, int64_t n_esc, int64_t esc_cap)
{
    int64_t T = w12ref_rows_padded(N) / 16, G = w12ref_groups(K), P = T * G;
    int64_t bad = 0;
    if (n_esc < 0 || n_esc > esc_cap) bad++;
    if (esc_ptr[0] != 0) bad++;
    if ((int64_t)esc_ptr[P] != n_esc) bad++;
    for (int64_t i = 0; i < P; ++i)
        if (esc_ptr[i + 1] < esc_ptr[i]) bad++;
    if (bad) return bad; /* the groups cannot be walked safely */
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            for (int64_t e = esc_ptr[t * G + g]; e < esc_ptr[t * G + g + 1]; ++e) {
                int64_t n, k;
                int key = (int)(esc[e] >> 16);
                key_position(t, g, key, &n, &k);
                if (key >= 4096 || n >= N || k >= K) bad++;
                if (e + 1 < esc_ptr[t * G + g + 1] && (esc[e + 1] >> 16) <= (esc[e] >> 16)) bad++;
            }
        }
    }
    return bad;
}

/* Applies the escapes of stripe t that fall in row n to row[] (columns
 * 0..K-1). */
static void patch_row(int64_t n, int64_t K, const int32_t *esc_ptr, const uint32_t *esc,
                      uint16_t *row)
{
    int64_t t = n / 16, G = w12ref_groups(K);
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t e = esc_ptr[t * G + g]; e < esc_ptr[t * G + g + 1]; ++e) {
            int64_t rn, rk;
            key_position(t, g, (int)(esc[e] >> 16), &rn, &rk);
            if (rn == n) row[rk] = (uint16_t)(esc[e] & 0xFFFF);
        }
    }
}

/* One decoded row (no structure check; the caller has done it). */
static void decode_row(int64_t n, int64_t K, int64_t Kp, const uint8_t *hi, const uint8_t *lo,
                       const uint8_t *base, const int32_t *esc_ptr, const uint32_t *esc,
                       uint16_t *row)
{
    for (int64_t k = 0; k < K; ++k) row[k] = w12ref_decode_record(record_at(hi, lo, n, k, Kp), base[n]);
    patch_row(n, K, esc_ptr, esc, row);
}

/* ---- step a4: decode ----  out is [N,K] with row stride ldo.  Every weight
 * comes from its record, then each escape overwrites its position with the
 * stored BF16 bits. */
int w12ref_decode(int64_t N, int64_t K, const uint8_t *hi, const uint8_t *lo,
                  const uint8_t *base, const int32_t *esc_ptr, const uint32_t *esc,
                  int64_t n_esc, uint16_t *out, int64_t ldo)
{
    if (N < 0 || K < 0 || ldo < K) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, n_esc) != 0) return REF_ERR_CORRUPT;
    int64_t Kp = w12ref_cols_padded(K);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t n = 0; n < N; ++n) decode_row(n, K, Kp, hi, lo, base, esc_ptr, esc, out + n * ldo);
    return REF_OK;
}

/* ---- step a5: load-time check ----  *n_mismatch = number of (n,k) whose
 * decoded bits differ from W.  A malformed escape list gives REF_ERR_CORRUPT
 * and *n_mismatch = -1; any mismatch gives REF_ERR_MISMATCH. */
int w12ref_verify(const uint16_t *W, int64_t ldw, int64_t N, int64_t K, const uint8_t *hi,
                  const uint8_t *lo, const uint8_t *base, const int32_t *esc_ptr,
                  const uint32_t *esc, int64_t n_esc, int64_t esc_cap, int64_t *n_mismatch)
{
    if (N < 0 || K < 0 || ldw < K || !n_mismatch) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, esc_cap) != 0) {
        *n_mismatch = -1;
        return REF_ERR_CORRUPT;
    }
    uint16_t *dec = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(N * K > 0 ? N * K : 1));
    if (!dec) return REF_ERR_INVALID;
    w12ref_decode(N, K, hi, lo, base, esc_ptr, esc, n_esc, dec, K);
    int64_t bad = 0;
#pragma omp parallel for reduction(+ : bad)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) bad += dec[n * K + k] != W[n * ldw + k];
    free(dec);
    *n_mismatch = bad;
    return bad ? REF_ERR_MISMATCH : REF_OK;
}

/* ---- steps a6-a9: the GEMM ----
 * Y[m,n] = BF16_RNE( sum_k A[m,k] * W[n,k] ) with W the decoded tensor.
 * Every product of two BF16 values is exact in FP64; the products are added
 * in ascending k in FP64 and the sum is rounded once to BF16.  Optional
 * outputs: Y64 (the FP64 sum) and absdot (sum_k |A[m,k]|*|W[n,k]|), both
 * [M,N] row-major, used by the tolerance rule. */
int w12ref_gemm(const uint16_t *A, int64_t M, int64_t lda, int64_t N, int64_t K,
                const uint8_t *hi, const uint8_t *lo, const uint8_t *base,
                const int32_t *esc_ptr, const uint32_t *esc, int64_t n_esc, uint16_t *Y, int64_t ldy, double *Y64, double *absdot)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldy < N) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, n_esc) != 0) return REF_ERR_CORRUPT;
    int64_t Kp = w12ref_cols_padded(K);
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!a) return REF_ERR_INVALID;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) a[m * K + k] = w12ref_bf16_to_double(A[m * lda + k]);
#pragma omp parallel
    {
        uint16_t *row = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K > 0 ? K : 1));
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t n = 0; n < N; ++n) {
            decode_row(n, K, Kp, hi, lo, base, esc_ptr, esc, row);
            for (int64_t k = 0; k < K; ++k) w[k] = w12ref_bf16_to_double(row[k]);
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, mag = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    acc += a[m * K + k] * w[k];
                    mag += fabs(a[m * K + k]) * fabs(w[k]);
                }
                Y[m * ldy + n] = w12ref_bf16_from_double(acc);
                if (Y64) Y64[m * N + n] = acc;
                if (absdot) absdot[m * N + n] = mag;
            }
        }
        free(row);
        free(w);
    }
    free(a);
    return REF_OK;
}

/* The same GEMM evaluated only at the listed output positions (m_i, n_i):
 * used to check full-size outputs one element at a time.  y, y64 and absdot
 * have `count` entries. */
int w12ref_gemm_sample(const uint16_t *A, int64_t M, int64_t lda, int64_t N, int64_t K,
                       const uint8_t *hi, const uint8_t *lo, const uint8_t *base,
                       const int32_t *esc_ptr, const uint32_t *esc, int64_t n_esc, const int64_t *ms, const int64_t *ns, int64_t count,
                       uint16_t *y, double *y64, double *absdot)
{
    if (M < 0 || N < 0 || K < 0 || lda < K) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, n_esc) != 0) return REF_ERR_CORRUPT;
    int64_t Kp = w12ref_cols_padded(K);
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return REF_ERR_INVALID;
#pragma omp parallel
    {
        uint16_t *row = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < count; ++i) {
            decode_row(ns[i], K, Kp, hi, lo, base, esc_ptr, esc, row);
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double av = w12ref_bf16_to_double(A[ms[i] * lda + k]);
                double wv = w12ref_bf16_to_double(row[k]);
                acc += av * wv;
                mag += fabs(av) * fabs(wv);
            }
            y[i] = w12ref_bf16_from_double(acc);
            y64[i] = acc;
            absdot[i] = mag;
        }
        free(row);
    }
    return REF_OK;
}

/* ---- the nested 8-bit view ----  SpecPilot, section 4.1 and the news
 * article's "two-level verification": a low-precision pass reads the 8-bit
 * weight view nested in W12.  The hi byte of a record holds the sign, the
 * 4-bit exponent offset and the top 3 mantissa bits, so the view of an
 * in-window weight is (-1)^s * 2^(base+off-127) * (1 + m_hi/8): the BF16
 * bits s<<15 | (base+off)<<7 | m_hi<<4.  The pages do not say what the view
 * holds at an escaped position; the reading taken here is the escape's own
 * BF16 bits with the 4 low mantissa bits cleared (truncation toward zero,
 * which keeps outliers, zeros, Inf and NaN in their class).  Padding columns
 * are never read. */
static uint16_t nested8_value(int hi_byte, int base)
{
    int s = (hi_byte >> 7) & 1, off = (hi_byte >> 3) & 15, mh = hi_byte & 7;
    return (uint16_t)((s << 15) | (((base + off) & 0xFF) << 7) | (mh << 4));
}

static void decode_row_nested8(int64_t n, int64_t K, int64_t Kp, const uint8_t *hi, const uint8_t *base,
                               const int32_t *esc_ptr, const uint32_t *esc, uint16_t *row)
{
    for (int64_t k = 0; k < K; ++k) row[k] = nested8_value(hi[w12ref_hi_offset(n, k, Kp)], base[n]);
    int64_t t = n / 16, G = w12ref_groups(K);
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t e = esc_ptr[t * G + g]; e < esc_ptr[t * G + g + 1]; ++e) {
            int64_t rn, rk;
            key_position(t, g, (int)(esc[e] >> 16), &rn, &rk);
            if (rn == n) row[rk] = (uint16_t)(esc[e] & 0xFFF0);
        }
    }
}

/* The nested 8-bit view of the whole tensor, [N,K] with row stride ldo. */
int w12ref_decode_nested8(int64_t N, int64_t K, const uint8_t *hi, const uint8_t *base,
                          const int32_t *esc_ptr, const uint32_t *esc, int64_t n_esc, uint16_t *out, int64_t ldo)
{
    if (N < 0 || K < 0 || ldo < K) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, n_esc) != 0) return REF_ERR_CORRUPT;
    int64_t Kp = w12ref_cols_padded(K);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t n = 0; n < N; ++n) decode_row_nested8(n, K, Kp, hi, base, esc_ptr, esc, out + n * ldo);
    return REF_OK;
}

/* Y = A * V^T with V the nested 8-bit view: the same exact FP64 sum in
 * ascending k, rounded once to BF16, as the GEMM above. */
int w12ref_gemm_nested8(const uint16_t *A, int64_t M, int64_t lda, int64_t N, int64_t K, const uint8_t *hi,
                        const uint8_t *base, const int32_t *esc_ptr, const uint32_t *esc, int64_t n_esc,
                        uint16_t *Y, int64_t ldy, double *Y64, double *absdot)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldy < N) return REF_ERR_INVALID;
    if (w12ref_check_structure(N, K, esc_ptr, esc, n_esc, n_esc) != 0) return REF_ERR_CORRUPT;
    int64_t Kp = w12ref_cols_padded(K);
    double *a = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!a) return REF_ERR_INVALID;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) a[m * K + k] = w12ref_bf16_to_double(A[m * lda + k]);
#pragma omp parallel
    {
        uint16_t *row = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K > 0 ? K : 1));
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t n = 0; n < N; ++n) {
            decode_row_nested8(n, K, Kp, hi, base, esc_ptr, esc, row);
            for (int64_t k = 0; k < K; ++k) w[k] = w12ref_bf16_to_double(row[k]);
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0, mag = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    acc += a[m * K + k] * w[k];
                    mag += fabs(a[m * K + k]) * fabs(w[k]);
                }
                Y[m * ldy + n] = w12ref_bf16_from_double(acc);
                if (Y64) Y64[m * N + n] = acc;
                if (absdot) absdot[m * N + n] = mag;
            }
        }
        free(row);
        free(w);
    }
    free(a);
    return REF_OK;
}

/* ---- fused gate/up epilogue (reading R24) ----
 * The pages do not write the layer an exact pass streams through; a gated
 * MLP's gate/up GEMM is followed by silu(g) * u before the down GEMM, with
 * silu(x) = x / (1 + exp(-x)).  Row layout (R24): in row stripe t of W
 * (rows 16t .. 16t+15), row 16t+i is the gate row and row 16t+8+i the up
 * row of hidden unit 8t+i, i = 0..7, so N is a multiple of 16 and the output
 * has N/2 columns.  g and u are the exact FP64 sums of w12ref_gemm; silu(g)*u
 * is evaluated in FP64 by the formula above and rounded once to BF16.
 * Optional outputs, [M, N/2] row-major: G64, U64 (the two sums), magG, magU
 * (their sum_k |A||W|), used by the tolerance rule. */
int w12ref_gemm_silu_mul(const uint16_t *A, int64_t M, int64_t lda, int64_t N, int64_t K,
                         const uint8_t *hi, const uint8_t *lo, const uint8_t *base,
                         const int32_t *esc_ptr, const uint32_t *esc, int64_t n_esc, uint16_t *Y, int64_t ldy,
                         double *G64, double *U64, double *magG, double *magU)
{
    if (M < 0 || N < 0 || N % 16 != 0 || ldy < N / 2) return REF_ERR_INVALID;
    size_t cells = (size_t)(M * N > 0 ? M * N : 1);
    uint16_t *full = (uint16_t *)malloc(sizeof(uint16_t) * cells);
    double *sum = (double *)malloc(sizeof(double) * cells);
    double *mag = (double *)malloc(sizeof(double) * cells);
    int st = REF_ERR_INVALID;
    if (full && sum && mag) st = w12ref_gemm(A, M, lda, N, K, hi, lo, base, esc_ptr, esc, n_esc, full, N, sum, mag);
    if (st == REF_OK) {
        int64_t H = N / 2;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t j = 0; j < H; ++j) {
                int64_t gate = (j / 8) * 16 + j % 8, up = gate + 8;
                double g = sum[m * N + gate], u = sum[m * N + up];
                double y = g / (1.0 + exp(-g)) * u;
                Y[m * ldy + j] = w12ref_bf16_from_double(y);
                if (G64) G64[m * H + j] = g;
                if (U64) U64[m * H + j] = u;
                if (magG) magG[m * H + j] = mag[m * N + gate];
                if (magU) magU[m * H + j] = mag[m * N + up];
            }
    }
    free(full);
    free(sum);
    free(mag);
    return st;
}

/* Round doubles to BF16 bits, one by one (w12ref_bf16_from_double). */
void w12ref_round_bf16(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = w12ref_bf16_from_double(x[i]);
}

/* Storage cost in bits per weight, counting everything the tensor stores:
 * both planes (with padding), the bases, the group offsets and the escapes
 * (one 32-bit entry each). */
double w12ref_bits_per_weight(int64_t N, int64_t K, int64_t n_esc)
{
    double bytes = (double)w12ref_hi_bytes(N, K) + (double)w12ref_lo_bytes(N, K) + (double)N +
                   4.0 * (double)w12ref_ptr_len(N, K) + 4.0 * (double)n_esc;
    return 8.0 * bytes / ((double)N * (double)K);
}

int w12ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
