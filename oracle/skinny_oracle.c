/*
 * CPU oracle for the BF16 skinny GEMM   y[M,N] = x[M,K] . W[N,K]^T
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the package's smoke check and the
 * benchmark's CPU-baseline leg are the only users of this file.  The GPU
 * library never links, calls or includes it, and it includes nothing of the
 * GPU library.
 *
 * What it computes is the plain definition of the operation, written out:
 *
 *     y_ref[m,n] = RNE_bf16( SUM_k  x[m,k] * W[n,k] )        (sum taken EXACTLY)
 *
 *  - The F.linear layout (y = x W^T, W stored [N,K] row-major) is the layout of
 *    the projections in vLLM PR #62949 ("SM121 skinny-GEMM plans for the
 *    GLM-5.3-Flash BF16 decode projections", Validation: results compared with
 *    F.linear).
 *  - The reference is a high-precision one: vLLM PR #65306 ("Add SM90 skinny
 *    GEMM plans for the BF16 decode projections", Validation) compares every
 *    output element with a float64 reference.  Here the sum is not merely
 *    float64 but exact, so the oracle has no rounding-order freedom at all:
 *    the only rounding is the final one to BF16.
 *  - Rounding to BF16 is round-to-nearest, ties-to-even (the pages give BF16
 *    outputs without a rounding mode; RNE is the IEEE default and the
 *    CUDA/PyTorch convention).
 *  - The FP32-output form (oracle_bf16_skinny_gemm_f32) rounds the same exact
 *    sum once to FP32, round-to-nearest, ties-to-even: the outputs of the MoE
 *    router gate (288, 4096), which vLLM PR #62949 (Validation, the nsys
 *    census) names as the one projection kept in FP32.
 *
 * Exactness.  A finite BF16 value is s * 2^e with an integer significand
 * 0 <= s <= 255 and -133 <= e <= 120.  A product of two of them is
 * (s1*s2) * 2^(e1+e2) with s1*s2 < 2^16 and -266 <= e1+e2 <= 240, so every
 * product is an integer multiple of 2^-266 below 2^256.  The accumulator below
 * is a plain fixed-point integer in units of 2^-266 ("long accumulator"), held
 * as 18 signed 64-bit digits of 32 bits each (576 bits, carries deferred).
 * Each digit receives at most K < 2^30 terms below 2^32 each, so no digit
 * overflows, and |sum| < 2^30 * 2^256 = 2^286, i.e. below 2^552 units of
 * 2^-266, well inside 576 bits: the sum is exact.
 *
 * Non-finite inputs follow IEEE semantics: NaN in, or inf*0, or +inf and -inf
 * in one sum give NaN; otherwise any infinite product gives that infinity.
 * An exact zero sum gives +0.
 */
#define _GNU_SOURCE
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ACC_DIGITS 18   /* 18 x 32 = 576 bits */
#define ACC_BIAS 266    /* bit 0 of the accumulator weighs 2^-266 */
#define ACC_MAX_K (1 << 30)

enum { CLS_FINITE = 0, CLS_INF = 1, CLS_NAN = 2 };

/* ---- BF16 decoding -------------------------------------------------------
 * bits: sign(1) | biased exponent(8) | fraction(7)
 *   exponent 0      : subnormal, value = fraction * 2^-133
 *   exponent 1..254 : normal,    value = (128 + fraction) * 2^(exponent-134)
 *   exponent 255    : inf (fraction 0) or NaN
 */
typedef struct {
    uint32_t sig;  /* integer significand, 0..255 */
    int32_t pos;   /* e + 133, so that pos_x + pos_w is the bit index of the product */
    int32_t neg;   /* sign bit */
    int32_t cls;   /* CLS_* */
} bf16_parts;

static bf16_parts decode_bf16(uint16_t b) {
    bf16_parts p;
    uint32_t ex = (b >> 7) & 0xffu, fr = b & 0x7fu;
    p.neg = (b >> 15) & 1;
    if (ex == 0xffu) {
        p.sig = 0;
        p.pos = 0;
        p.cls = fr ? CLS_NAN : CLS_INF;
    } else if (ex == 0) {
        p.sig = fr;
        p.pos = 0;          /* e = -133 */
        p.cls = CLS_FINITE;
    } else {
        p.sig = 128u + fr;
        p.pos = (int32_t)ex - 1;  /* e = ex - 134, pos = e + 133 */
        p.cls = CLS_FINITE;
    }
    return p;
}

/* ---- the exact accumulator ------------------------------------------------ */
typedef struct {
    int64_t d[ACC_DIGITS];
    int nan, pinf, ninf;
} exact_acc;

static void acc_clear(exact_acc *a) { memset(a, 0, sizeof(*a)); }

/* add (or subtract) prod * 2^(bit - ACC_BIAS), 0 <= prod < 2^16, 0 <= bit <= 506 */
static void acc_add(exact_acc *a, uint32_t prod, int bit, int neg) {
    uint64_t v = (uint64_t)prod << (bit & 31); /* < 2^47 */
    int64_t lo = (int64_t)(v & 0xffffffffu);
    int64_t hi = (int64_t)(v >> 32);
    int i = bit >> 5;
    if (neg) {
        a->d[i] -= lo;
        a->d[i + 1] -= hi;
    } else {
        a->d[i] += lo;
        a->d[i + 1] += hi;
    }
}

/* accumulate the product of two decoded BF16 values */
static void acc_mac(exact_acc *a, const bf16_parts *x, const bf16_parts *w) {
    int neg = x->neg ^ w->neg;
    if (x->cls == CLS_NAN || w->cls == CLS_NAN) {
        a->nan = 1;
        return;
    }
    if (x->cls == CLS_INF || w->cls == CLS_INF) {
        /* inf * 0 is NaN; inf * finite-nonzero or inf * inf is a signed inf */
        uint32_t other = (x->cls == CLS_INF) ? (w->cls == CLS_INF ? 1u : w->sig)
                                             : x->sig;
        if (other == 0)
            a->nan = 1;
        else if (neg)
            a->ninf = 1;
        else
            a->pinf = 1;
        return;
    }
    uint32_t prod = x->sig * w->sig;
    if (prod) acc_add(a, prod, x->pos + w->pos, neg);
}

/* floor(v / 2^32) and v mod 2^32 without relying on signed right shifts */
static int64_t floor_div_2p32(int64_t v) {
    int64_t low = (int64_t)((uint64_t)v & 0xffffffffu);
    return (v - low) / 4294967296LL;
}

/* Propagate carries so that digits 0..ACC_DIGITS-2 lie in [0, 2^32).
 * Returns the sign of the value (-1, 0, +1) and leaves |value| in a->d. */
static int acc_normalize(exact_acc *a) {
    int i;
    for (i = 0; i < ACC_DIGITS - 1; ++i) {
        int64_t c = floor_div_2p32(a->d[i]);
        a->d[i] -= c * 4294967296LL;
        a->d[i + 1] += c;
    }
    int sign = 0;
    if (a->d[ACC_DIGITS - 1] < 0) {
        sign = -1;
        for (i = 0; i < ACC_DIGITS; ++i) a->d[i] = -a->d[i];
        for (i = 0; i < ACC_DIGITS - 1; ++i) {
            int64_t c = floor_div_2p32(a->d[i]);
            a->d[i] -= c * 4294967296LL;
            a->d[i + 1] += c;
        }
    } else {
        for (i = 0; i < ACC_DIGITS; ++i)
            if (a->d[i]) {
                sign = 1;
                break;
            }
    }
    return sign;
}

static int acc_bit(const exact_acc *a, int i) {
    return (int)((a->d[i >> 5] >> (i & 31)) & 1);
}

static int acc_msb(const exact_acc *a) {
    int i, b;
    for (i = ACC_DIGITS - 1; i >= 0; --i) {
        if (a->d[i]) {
            for (b = 63; b >= 0; --b)
                if ((a->d[i] >> b) & 1) return i * 32 + b;
        }
    }
    return -1;
}

/* Round the (normalized, non-zero) magnitude to a binary format with p
 * significand bits and smallest ulp 2^umin, round-to-nearest-even.
 * Result: magnitude = q * 2^u with q < 2^p (q >= 2^(p-1) unless u == umin). */
static void acc_round(const exact_acc *a, int p, int umin, uint64_t *q_out, int *u_out) {
    int P = acc_msb(a);
    int E = P - ACC_BIAS;          /* 2^E <= |value| < 2^(E+1) */
    int u = E - (p - 1);
    if (u < umin) u = umin;
    int ql = u + ACC_BIAS;         /* accumulator bit holding the ulp */
    uint64_t q = 0;
    int i;
    if (ql <= 0) {                 /* every bit fits: exact */
        for (i = P; i >= 0; --i) q = (q << 1) | (uint64_t)acc_bit(a, i);
        q <<= -ql;
        *q_out = q;
        *u_out = u;
        return;
    }
    for (i = P; i >= ql; --i) q = (q << 1) | (uint64_t)acc_bit(a, i);
    int round = acc_bit(a, ql - 1);
    int sticky = 0;
    for (i = ql - 2; i >= 0 && !sticky; --i) sticky = acc_bit(a, i);
    if (round && (sticky || (q & 1u))) q += 1;
    if (q == ((uint64_t)1 << p)) { /* carried into a new binade */
        q >>= 1;
        u += 1;
    }
    *q_out = q;
    *u_out = u;
}

/* final BF16 bits of the accumulated sum */
static uint16_t acc_to_bf16(exact_acc *a) {
    if (a->nan || (a->pinf && a->ninf)) return 0x7fc0;
    if (a->pinf) return 0x7f80;
    if (a->ninf) return 0xff80;
    int sign = acc_normalize(a);
    if (sign == 0) return 0x0000;
    uint64_t q;
    int u;
    acc_round(a, 8, -133, &q, &u);
    uint16_t s = sign < 0 ? 0x8000 : 0x0000;
    if (q < 128) return (uint16_t)(s | q);               /* subnormal (u == -133) */
    if (u > 120) return (uint16_t)(s | 0x7f80);          /* q*2^u >= 2^128: overflow */
    return (uint16_t)(s | ((uint32_t)(u + 134) << 7) | (uint32_t)(q - 128));
}

/* final FP32 bits of the accumulated sum: 24 significand bits, smallest ulp
 * 2^-149, largest finite value (2^24 - 1) * 2^104 */
static uint32_t acc_to_f32(exact_acc *a) {
    if (a->nan || (a->pinf && a->ninf)) return 0x7fc00000u;
    if (a->pinf) return 0x7f800000u;
    if (a->ninf) return 0xff800000u;
    int sign = acc_normalize(a);
    if (sign == 0) return 0x00000000u;
    uint64_t q;
    int u;
    acc_round(a, 24, -149, &q, &u);
    uint32_t s = sign < 0 ? 0x80000000u : 0u;
    if (q < ((uint64_t)1 << 23)) return s | (uint32_t)q;          /* subnormal (u == -149) */
    if (u > 104) return s | 0x7f800000u;                           /* q*2^u >= 2^128: overflow */
    return s | ((uint32_t)(u + 150) << 23) | (uint32_t)(q - ((uint64_t)1 << 23));
}

/* ---- exported entry points -------------------------------------------------- */

/* Number of CPUs this process may run on. */
int oracle_cores(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

typedef struct {
    const uint16_t *x, *W;
    uint16_t *y;       /* BF16 outputs, or */
    uint32_t *y32;     /* FP32 outputs (bit patterns) when non-null */
    long long ldx, ldw, ldy;
    int M, K, n0, n1;
    const bf16_parts *xp; /* decoded x, M*K */
} job_t;

static void *run_rows(void *arg) {
    const job_t *j = (const job_t *)arg;
    exact_acc acc;
    int n, m, k;
    for (n = j->n0; n < j->n1; ++n) {
        const uint16_t *wrow = j->W + (long long)n * j->ldw;
        for (m = 0; m < j->M; ++m) {
            const bf16_parts *xr = j->xp + (long long)m * j->K;
            acc_clear(&acc);
            for (k = 0; k < j->K; ++k) {
                bf16_parts wp = decode_bf16(wrow[k]);
                acc_mac(&acc, &xr[k], &wp);
            }
            if (j->y32)
                j->y32[(long long)m * j->ldy + n] = acc_to_f32(&acc);
            else
                j->y[(long long)m * j->ldy + n] = acc_to_bf16(&acc);
        }
    }
    return NULL;
}

static int gemm(const uint16_t *x, long long ldx, const uint16_t *W, long long ldw, uint16_t *y,
                uint32_t *y32, long long ldy, int M, int N, int K, int threads) {
    if (M < 0 || N < 0 || K < 0 || K >= ACC_MAX_K) return -1;
    if (M == 0 || N == 0) return 0;
    if (!x || !W || (!y && !y32) || ldx < K || ldw < K || ldy < N) return -1;
    if (threads <= 0) threads = oracle_cores();
    if (threads > N) threads = N;
    bf16_parts *xp = (bf16_parts *)malloc(sizeof(bf16_parts) * (size_t)M * (size_t)(K ? K : 1));
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)threads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    if (!xp || !jobs || !tids) {
        free(xp);
        free(jobs);
        free(tids);
        return -1;
    }
    int m, k, t;
    for (m = 0; m < M; ++m)
        for (k = 0; k < K; ++k) xp[(long long)m * K + k] = decode_bf16(x[(long long)m * ldx + k]);
    for (t = 0; t < threads; ++t) {
        jobs[t].x = x;
        jobs[t].W = W;
        jobs[t].y = y;
        jobs[t].y32 = y32;
        jobs[t].ldx = ldx;
        jobs[t].ldw = ldw;
        jobs[t].ldy = ldy;
        jobs[t].M = M;
        jobs[t].K = K;
        jobs[t].n0 = (int)((long long)N * t / threads);
        jobs[t].n1 = (int)((long long)N * (t + 1) / threads);
        jobs[t].xp = xp;
    }
    char *live = (char *)calloc((size_t)threads, 1);
    for (t = 1; t < threads; ++t) {
        if (live && pthread_create(&tids[t], NULL, run_rows, &jobs[t]) == 0)
            live[t] = 1;
        else
            run_rows(&jobs[t]); /* could not start a thread: do its rows here */
    }
    run_rows(&jobs[0]);
    for (t = 1; t < threads; ++t)
        if (live && live[t]) pthread_join(tids[t], NULL);
    free(live);
    free(xp);
    free(jobs);
    free(tids);
    return threads;
}

/* y[m*ldy + n] = RNE_bf16(exact sum_k x[m*ldx + k] * W[n*ldw + k])
 * for 0 <= m < M, 0 <= n < N.  All arrays hold raw BF16 bits in host memory.
 * threads <= 0 uses every CPU in the affinity mask.  Rows n are split into
 * contiguous ranges, one per thread; the result does not depend on the
 * thread count.  Returns the number of threads used, or -1 on bad arguments. */
int oracle_bf16_skinny_gemm(const uint16_t *x, long long ldx, const uint16_t *W, long long ldw,
                            uint16_t *y, long long ldy, int M, int N, int K, int threads) {
    if (!y) return -1;
    return gemm(x, ldx, W, ldw, y, NULL, ldy, M, N, K, threads);
}

/* The same sums rounded once to FP32 (RNE): y holds FP32 bit patterns. */
int oracle_bf16_skinny_gemm_f32(const uint16_t *x, long long ldx, const uint16_t *W,
                                long long ldw, uint32_t *y, long long ldy, int M, int N, int K,
                                int threads) {
    if (!y) return -1;
    return gemm(x, ldx, W, ldw, NULL, y, ldy, M, N, K, threads);
}

/* The exact dot product of one x row and one W row, for tests that need the
 * unrounded sum.  On return digits[0..17] hold |sum| in units of 2^-266
 * (digit i weighs 2^(32 i)), *sign is -1/0/+1, and *special is 0 for a finite
 * sum, 1 for +inf, 2 for -inf, 3 for NaN.  The BF16 rounding of the sum is
 * returned. */
uint16_t oracle_exact_dot(const uint16_t *x, const uint16_t *w, int K, int64_t *digits,
                          int *sign, int *special) {
    exact_acc acc;
    int k;
    acc_clear(&acc);
    for (k = 0; k < K; ++k) {
        bf16_parts xp = decode_bf16(x[k]), wp = decode_bf16(w[k]);
        acc_mac(&acc, &xp, &wp);
    }
    exact_acc copy = acc;
    uint16_t r = acc_to_bf16(&copy);
    *special = (acc.nan || (acc.pinf && acc.ninf)) ? 3 : acc.pinf ? 1 : acc.ninf ? 2 : 0;
    *sign = 0;
    memset(digits, 0, sizeof(int64_t) * ACC_DIGITS);
    if (*special == 0) {
        *sign = acc_normalize(&acc);
        memcpy(digits, acc.d, sizeof(int64_t) * ACC_DIGITS);
    }
    return r;
}

/* Constants the Python side needs to rebuild exact values from digits. */
int oracle_acc_digits(void) { return ACC_DIGITS; }
int oracle_acc_bias(void) { return ACC_BIAS; }
