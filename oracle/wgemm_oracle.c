/*
 * CPU oracle for the dense GEMM C = A·Bᵀ with fp16 A (M×K), fp16 B (N×K) and
 * fp32 accumulation/output, as "SASS-Level Kernel Generation for Blackwell"
 * (section "The numbers", Setup paragraph) defines the problem:
 *
 *     C[i][j] = Σ_{k<K} A[i][k] · B[j][k]        (row-major, C = A·Bᵀ)
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load this library. The GEMM library never
 * links, loads or calls it, and it shares no code with the GEMM library.
 *
 * It is the plain definition written out: a triple loop accumulating in fp64,
 * one row of C per work item, rows split over host threads. Each fp16 value is
 * decoded from its bit fields (sign, 5-bit exponent, 10-bit fraction), so no
 * half-precision library routine is involved. Products of two fp16 values are
 * exact in fp64 (11 × 11 significand bits), so the only rounding is the fp64
 * summation, far below the fp32 tolerance the GPU result is held to.
 *
 * Besides C it can produce |A|·|B|ᵀ, the magnitude term of the elementwise
 * tolerance |C − C_ref| ≤ 2e-3·(|A|·|B|ᵀ)_ij + 1e-6.
 *
 * The same definition with bf16 operands (decoded from their own bit fields:
 * sign, 8-bit exponent, 7-bit fraction; products of two bf16 values are exact
 * in fp64 too), and the rounding of an fp64 value to fp16 or bf16 (nearest,
 * ties to even, from the formats' definitions) that a 16-bit C is compared
 * against. These follow no passage of the pages, which measure fp16 → fp32
 * only: they are the plain definitions of the adjacent types.
 *
 * Pins (tests marked "not gpu"): the decoder against numpy's float16 for all
 * 65,536 bit patterns; brute force against an independent fp64 matmul and
 * against exact integer arithmetic on shapes 1–64 per dimension; identity and
 * permutation matrices; closed forms (all ones, patterns whose sums are known);
 * NaN-poisoned padding beyond K; sampled evaluation against full evaluation.
 * The bf16 decoder against a reinterpretation of the pattern as the upper
 * half of an fp32 (numpy) for all 65,536 patterns; the fp16 encoder against
 * numpy's float64 → float16 conversion; both encoders on every representable
 * value, every midpoint between neighbours (ties to even) and its two
 * neighbouring doubles, the overflow threshold, and the bf16 encoder against
 * torch's float32 → bfloat16 conversion on float32 inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* fp16 (IEEE 754 binary16) bit pattern → double, from the bit fields. */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int exponent = (h >> 10) & 0x1F;
    const int fraction = h & 0x3FF;
    double v;
    if (exponent == 0)
        v = ldexp((double)fraction, -24); /* zero or subnormal: 0.f × 2^-14 */
    else if (exponent == 31)
        v = fraction ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fraction), exponent - 25); /* 1.f × 2^(e-15) */
    return sign ? -v : v;
}

/* bf16 bit pattern → double, from the bit fields. */
double oracle_bf16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int exponent = (h >> 7) & 0xFF;
    const int fraction = h & 0x7F;
    double v;
    if (exponent == 0)
        v = ldexp((double)fraction, -133); /* zero or subnormal: 0.f × 2^-126 */
    else if (exponent == 255)
        v = fraction ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + fraction), exponent - 134); /* 1.f × 2^(e-127) */
    return sign ? -v : v;
}

/* Operand types of the typed entry points. */
enum { ORACLE_F16 = 1, ORACLE_BF16 = 2 };
typedef double (*decode_fn)(uint16_t);

/* One problem, shared read-only by the worker threads. */
typedef struct {
    decode_fn decode;           /* the operands' bit pattern → double */
    const uint16_t *A, *B;
    const int64_t *rows, *cols; /* NULL = all rows / all columns */
    int64_t n_rows, n_cols, K, lda, ldb;
    double *C, *Cabs;           /* n_rows × ldc, row r of the output is rows[r] */
    int64_t ldc;
    const double *Bd;           /* the selected B rows decoded: n_cols × K */
    int64_t next_row;           /* work counter */
    pthread_mutex_t lock;
} job_t;

static int64_t take_row(job_t *j)
{
    pthread_mutex_lock(&j->lock);
    int64_t r = j->next_row++;
    pthread_mutex_unlock(&j->lock);
    return r;
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    double *a = (double *)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    if (!a)
        return (void *)1;
    for (int64_t r = take_row(j); r < j->n_rows; r = take_row(j)) {
        const int64_t i = j->rows ? j->rows[r] : r;
        for (int64_t k = 0; k < j->K; ++k)
            a[k] = j->decode(j->A[i * j->lda + k]);
        for (int64_t c = 0; c < j->n_cols; ++c) {
            const double *b = j->Bd + c * j->K;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < j->K; ++k)
                s += a[k] * b[k];
            j->C[r * j->ldc + c] = s;
            if (j->Cabs) {
                for (int64_t k = 0; k < j->K; ++k)
                    sa += fabs(a[k]) * fabs(b[k]);
                j->Cabs[r * j->ldc + c] = sa;
            }
        }
    }
    free(a);
    return NULL;
}

static int hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Evaluate C at rows[0..n_rows) × cols[0..n_cols) (NULL selects all M rows /
 * all N columns) for operands of type ab_type (ORACLE_F16 or ORACLE_BF16,
 * both A and B). Output element (r, c) goes to C[r·ldc + c], and to Cabs if
 * it is not NULL. Returns the number of threads used, or a negative value on
 * a bad argument or an allocation failure.
 */
int oracle_gemm_f64_select_t(const uint16_t *A, const uint16_t *B,
                             const int64_t *rows, int64_t n_rows,
                             const int64_t *cols, int64_t n_cols,
                             int64_t K, int64_t lda, int64_t ldb,
                             double *C, double *Cabs, int64_t ldc, int nthreads, int ab_type)
{
    if (n_rows < 0 || n_cols < 0 || K < 0 || ldc < n_cols || lda < K || ldb < K ||
        (ab_type != ORACLE_F16 && ab_type != ORACLE_BF16))
        return -1;
    const decode_fn decode = ab_type == ORACLE_BF16 ? oracle_bf16_to_f64 : oracle_f16_to_f64;
    if (n_rows == 0 || n_cols == 0)
        return 0;
    job_t j;
    memset(&j, 0, sizeof j);
    j.decode = decode;
    j.A = A; j.B = B; j.rows = rows; j.cols = cols;
    j.n_rows = n_rows; j.n_cols = n_cols; j.K = K; j.lda = lda; j.ldb = ldb;
    j.C = C; j.Cabs = Cabs; j.ldc = ldc;
    double *Bd = (double *)malloc(sizeof(double) * (size_t)n_cols * (size_t)(K > 0 ? K : 1));
    if (!Bd)
        return -2;
    for (int64_t c = 0; c < n_cols; ++c) {
        const int64_t jrow = cols ? cols[c] : c;
        for (int64_t k = 0; k < K; ++k)
            Bd[c * K + k] = decode(B[jrow * ldb + k]);
    }
    j.Bd = Bd;
    pthread_mutex_init(&j.lock, NULL);
    int nt = nthreads > 0 ? nthreads : hardware_threads();
    if (nt > n_rows)
        nt = (int)n_rows;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int started = 0, failed = 0;
    for (int t = 0; t < nt && tid; ++t) {
        if (pthread_create(&tid[t], NULL, worker, &j) != 0)
            break;
        ++started;
    }
    if (started == 0) { /* no threads available: do the work here */
        failed = worker(&j) != NULL;
        started = 1;
    } else {
        for (int t = 0; t < started; ++t) {
            void *ret = NULL;
            pthread_join(tid[t], &ret);
            failed |= ret != NULL;
        }
    }
    free(tid);
    pthread_mutex_destroy(&j.lock);
    free(Bd);
    return failed ? -2 : started;
}

/* fp16 operands. */
int oracle_gemm_f64_select(const uint16_t *A, const uint16_t *B,
                           const int64_t *rows, int64_t n_rows,
                           const int64_t *cols, int64_t n_cols,
                           int64_t K, int64_t lda, int64_t ldb,
                           double *C, double *Cabs, int64_t ldc, int nthreads)
{
    return oracle_gemm_f64_select_t(A, B, rows, n_rows, cols, n_cols, K, lda, ldb, C, Cabs, ldc,
                                    nthreads, ORACLE_F16);
}

/* The full problem: C (M×ldc) = A·Bᵀ, and |A|·|B|ᵀ into Cabs when not NULL. */
int oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *C, double *Cabs,
                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                    int64_t ldc, int nthreads)
{
    return oracle_gemm_f64_select(A, B, NULL, M, NULL, N, K, lda, ldb, C, Cabs, ldc, nthreads);
}

/* The same with the operand type given (ORACLE_F16 or ORACLE_BF16). */
int oracle_gemm_f64_t(const uint16_t *A, const uint16_t *B, double *C, double *Cabs,
                      int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                      int64_t ldc, int nthreads, int ab_type)
{
    return oracle_gemm_f64_select_t(A, B, NULL, M, NULL, N, K, lda, ldb, C, Cabs, ldc, nthreads,
                                    ab_type);
}

/*
 * x rounded to the nearest value of a binary format with p significand bits
 * (the leading one included) and an exponent field of ebits bits (bias
 * 2^(ebits-1) - 1, subnormals below the least normal exponent), ties to the
 * value whose last significand bit is 0; returned as the format's 16-bit
 * pattern. Values at or beyond the largest finite value plus half its unit in
 * the last place become infinity; NaN becomes a quiet NaN.
 */
static uint16_t round_to_format(double x, int p, int ebits)
{
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias, emax = bias;
    const uint16_t sign = signbit(x) ? (uint16_t)0x8000 : 0;
    const uint16_t inf = (uint16_t)(((1u << ebits) - 1u) << (p - 1));
    if (isnan(x))
        return (uint16_t)(inf | (1u << (p - 2)));
    const double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | inf);
    int e2;
    frexp(a, &e2);       /* a = m · 2^e2, m in [0.5, 1) */
    int E = e2 - 1;      /* a in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin;        /* subnormal: the quantum stays that of the least binade */
    const double n = ldexp(a, -(E - (p - 1)));  /* a in units of the quantum (exact) */
    const double fl = floor(n), rest = n - fl;
    double r = fl;
    if (rest > 0.5 || (rest == 0.5 && fmod(fl, 2.0) == 1.0))
        r = fl + 1.0;
    if (r == ldexp(1.0, p)) { /* carried into the next binade */
        r = ldexp(1.0, p - 1);
        E += 1;
    }
    if (E > emax)
        return (uint16_t)(sign | inf);
    const uint32_t ri = (uint32_t)r;
    if (ri < (1u << (p - 1)))    /* subnormal: exponent field 0 */
        return (uint16_t)(sign | ri);
    return (uint16_t)(sign | ((uint32_t)(E + bias) << (p - 1)) | (ri - (1u << (p - 1))));
}

uint16_t oracle_f64_to_f16(double x) { return round_to_format(x, 11, 5); }
uint16_t oracle_f64_to_bf16(double x) { return round_to_format(x, 8, 8); }

/* out[i] = bits[i] decoded as ORACLE_F16 or ORACLE_BF16. */
int oracle_decode_array(const uint16_t *bits, double *out, int64_t n, int type)
{
    if (n < 0 || (type != ORACLE_F16 && type != ORACLE_BF16))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = type == ORACLE_BF16 ? oracle_bf16_to_f64(bits[i]) : oracle_f16_to_f64(bits[i]);
    return 0;
}

/* out[i] = x[i] rounded to ORACLE_F16 or ORACLE_BF16 (bit patterns). */
int oracle_round_f64(const double *x, uint16_t *out, int64_t n, int type)
{
    if (n < 0 || (type != ORACLE_F16 && type != ORACLE_BF16))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = type == ORACLE_BF16 ? oracle_f64_to_bf16(x[i]) : oracle_f64_to_f16(x[i]);
    return 0;
}

int oracle_hardware_threads(void) { return hardware_threads(); }
