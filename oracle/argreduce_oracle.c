/*
 * CPU oracle for row-wise ArgMax / ArgMin over the last axis.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, written out as the sequential scan
 * the pages describe):
 *
 *   onnxruntime PR #32092 "[CUDA] Parallelize ArgMax/ArgMin over wide last
 *   axes", Semantics: ties resolve to the lowest index (select_last_index ==
 *   0); a leading NaN still yields index 0; rows that are entirely -inf, +inf
 *   or NaN return index 0; the result must match the sequential one-thread-
 *   per-row kernel bit for bit for every input.
 *
 *   onnxruntime PR #31694 "[CUDA] Parallelize ArgMax/ArgMin over the
 *   reduction axis", Semantics: the candidate is seeded with element 0 and is
 *   only displaced by a strictly better value.
 *
 * For each row: best = (x[0], 0); for j = 1 .. cols-1, if x[j] is strictly
 * better than best (x[j] > best for ArgMax, x[j] < best for ArgMin, an IEEE
 * comparison that is false when either side is NaN) then best = (x[j], j).
 * The output is the int64 index and, optionally, the raw bits of x[r, index].
 *
 * Last-index variants (ONNX ArgMax/ArgMin attribute select_last_index = 1,
 * which #32092's Semantics section notes the CUDA provider sends to the CPU):
 * the same scan with a non-strict test, x[j] >= best (ArgMax) or x[j] <= best
 * (ArgMin), so among equal values the last one wins. The test is still false
 * when either side is NaN, so NaN handling is unchanged: a leading NaN keeps
 * index 0 and a later NaN is never chosen.
 *
 * Precision: every element is decoded exactly to binary64 and compared there.
 * Decoding binary16, bfloat16 and binary32 into binary64 is exact (including
 * subnormals, signed zeros and infinities), so each comparison decides the
 * same way as a comparison in the element's own type.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_F64 = 3 };
enum { ORACLE_MAX = 0, ORACLE_MIN = 1, ORACLE_MAX_LAST = 2, ORACLE_MIN_LAST = 3 };

/* IEEE 754 binary16: sign (1 bit), exponent (5 bits, bias 15), fraction
 * (10 bits). exponent 0 -> subnormal fraction * 2^-24; exponent 31 -> inf
 * (fraction 0) or NaN; otherwise (1024 + fraction) * 2^(exponent - 25). */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of binary32: sign (1), exponent (8, bias 127),
 * fraction (7). exponent 0 -> fraction * 2^-133; exponent 255 -> inf / NaN;
 * otherwise (128 + fraction) * 2^(exponent - 134). */
double oracle_decode_bf16(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

static size_t elem_size(int dtype) {
    switch (dtype) {
        case ORACLE_F32: return 4;
        case ORACLE_F16: return 2;
        case ORACLE_BF16: return 2;
        case ORACLE_F64: return 8;
        default: return 0;
    }
}

static double decode(const unsigned char* p, int dtype) {
    switch (dtype) {
        case ORACLE_F32: {
            float f;
            memcpy(&f, p, 4);
            return (double)f;
        }
        case ORACLE_F16: {
            uint16_t h;
            memcpy(&h, p, 2);
            return oracle_decode_f16(h);
        }
        case ORACLE_BF16: {
            uint16_t b;
            memcpy(&b, p, 2);
            return oracle_decode_bf16(b);
        }
        default: {
            double d;
            memcpy(&d, p, 8);
            return d;
        }
    }
}

/* "Strictly better": greater for ArgMax, less for ArgMin; "not worse" for
 * the last-index variants: greater or equal / less or equal. Every test is
 * false if either operand is NaN (a C relational operator on a NaN is false). */
static int better(double a, double b, int op) {
    switch (op) {
        case ORACLE_MAX: return a > b;
        case ORACLE_MIN: return a < b;
        case ORACLE_MAX_LAST: return a >= b;
        default: return a <= b;
    }
}

static int valid_op(int op) { return op >= ORACLE_MAX && op <= ORACLE_MIN_LAST; }

static void scan_rows(const unsigned char* x, int dtype, int64_t row_begin, int64_t row_end,
                      int64_t cols, int op, int64_t* out_idx, unsigned char* out_val) {
    const size_t es = elem_size(dtype);
    for (int64_t r = row_begin; r < row_end; ++r) {
        const unsigned char* row = x + (size_t)r * (size_t)cols * es;
        double best = decode(row, dtype);
        int64_t best_j = 0;
        for (int64_t j = 1; j < cols; ++j) {
            double v = decode(row + (size_t)j * es, dtype);
            if (better(v, best, op)) {
                best = v;
                best_j = j;
            }
        }
        out_idx[r] = best_j;
        if (out_val) memcpy(out_val + (size_t)r * es, row + (size_t)best_j * es, es);
    }
}

/* Returns 0 on success, -1 on invalid arguments. out_val may be NULL. */
int oracle_argreduce(const void* x, int dtype, int64_t rows, int64_t cols, int op,
                     int64_t* out_idx, void* out_val) {
    if (elem_size(dtype) == 0 || !valid_op(op)) return -1;
    if (rows < 0 || cols < 1 || (rows > 0 && (!x || !out_idx))) return -1;
    scan_rows((const unsigned char*)x, dtype, 0, rows, cols, op, out_idx, (unsigned char*)out_val);
    return 0;
}

/* Reduction over the middle axis of x[outer][R][inner] (row-major): for each
 * (o, i), the same sequential scan over r = 0 .. R-1 of x[o][r][i] (elements
 * `inner` apart). out_idx[o*inner + i] = the chosen r; out_val the raw bits of
 * that element. With inner == 1 this is the last-axis reduction above. */
int oracle_argreduce_axis(const void* x, int dtype, int64_t outer, int64_t R, int64_t inner, int op,
                          int64_t* out_idx, void* out_val) {
    if (elem_size(dtype) == 0 || !valid_op(op)) return -1;
    if (outer < 0 || R < 1 || inner < 1 || (outer > 0 && (!x || !out_idx))) return -1;
    const size_t es = elem_size(dtype);
    const unsigned char* base = (const unsigned char*)x;
    unsigned char* ov = (unsigned char*)out_val;
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t i = 0; i < inner; ++i) {
            const unsigned char* col = base + ((size_t)o * (size_t)R * (size_t)inner + (size_t)i) * es;
            const size_t stride = (size_t)inner * es;
            double best = decode(col, dtype);
            int64_t best_r = 0;
            for (int64_t r = 1; r < R; ++r) {
                double v = decode(col + (size_t)r * stride, dtype);
                if (better(v, best, op)) {
                    best = v;
                    best_r = r;
                }
            }
            out_idx[o * inner + i] = best_r;
            if (ov) memcpy(ov + (size_t)(o * inner + i) * es, col + (size_t)best_r * stride, es);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* cummax / cummin with indices (Paddle issue #79670, "Possible fixes": a   */
/* scan with argmax semantics where ties take the earlier index). For each  */
/* row and every position j, out[j] is the row's ArgMax (ArgMin) over       */
/* x[0..j] by the scan above: seed (x[0], 0), replace on a strictly better  */
/* element, so out[cols-1] equals oracle_argreduce(). Element types: the    */
/* four floating types and, compared exactly as integers, int32 (code 4)    */
/* and int64 (code 5). Ops 0 (max) and 1 (min).                             */
/* ------------------------------------------------------------------------ */
enum { ORACLE_I32 = 4, ORACLE_I64 = 5 };

static size_t cum_elem_size(int dtype) {
    if (dtype == ORACLE_I32) return 4;
    if (dtype == ORACLE_I64) return 8;
    return elem_size(dtype);
}

static int64_t read_int(const unsigned char* p, int dtype) {
    if (dtype == ORACLE_I32) {
        int32_t v;
        memcpy(&v, p, 4);
        return v;
    }
    int64_t v;
    memcpy(&v, p, 8);
    return v;
}

int oracle_cumreduce(const void* x, int dtype, int64_t rows, int64_t cols, int op, int64_t* out_idx,
                     void* out_val) {
    const size_t es = cum_elem_size(dtype);
    if (es == 0 || (op != ORACLE_MAX && op != ORACLE_MIN)) return -1;
    if (rows < 0 || cols < 1 || (rows > 0 && (!x || !out_idx))) return -1;
    const int is_int = dtype == ORACLE_I32 || dtype == ORACLE_I64;
    unsigned char* ov = (unsigned char*)out_val;
    for (int64_t r = 0; r < rows; ++r) {
        const unsigned char* row = (const unsigned char*)x + (size_t)r * (size_t)cols * es;
        int64_t best_j = 0;
        double best_f = is_int ? 0.0 : decode(row, dtype);
        int64_t best_i = is_int ? read_int(row, dtype) : 0;
        for (int64_t j = 0; j < cols; ++j) {
            if (j > 0) {
                int take;
                if (is_int) {
                    const int64_t v = read_int(row + (size_t)j * es, dtype);
                    take = op == ORACLE_MAX ? v > best_i : v < best_i;
                    if (take) best_i = v;
                } else {
                    const double v = decode(row + (size_t)j * es, dtype);
                    take = better(v, best_f, op);
                    if (take) best_f = v;
                }
                if (take) best_j = j;
            }
            out_idx[(size_t)r * (size_t)cols + (size_t)j] = best_j;
            if (ov) memcpy(ov + ((size_t)r * (size_t)cols + (size_t)j) * es, row + (size_t)best_j * es, es);
        }
    }
    return 0;
}

/* Row-parallel wrapper for timing on several host cores: rows are cut into
 * contiguous, independent ranges, one per thread, each scanned exactly as
 * above. Returns the number of threads used (>= 1), or -1 on error. */
typedef struct {
    const unsigned char* x;
    int dtype, op;
    int64_t r0, r1, cols;
    int64_t* out_idx;
    unsigned char* out_val;
} oracle_job;

static void* run_job(void* arg) {
    oracle_job* j = (oracle_job*)arg;
    scan_rows(j->x, j->dtype, j->r0, j->r1, j->cols, j->op, j->out_idx, j->out_val);
    return NULL;
}

int oracle_argreduce_mt(const void* x, int dtype, int64_t rows, int64_t cols, int op,
                        int64_t* out_idx, void* out_val, int nthreads) {
    if (elem_size(dtype) == 0 || !valid_op(op)) return -1;
    if (rows < 0 || cols < 1 || (rows > 0 && (!x || !out_idx))) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
    if (nthreads == 1) {
        scan_rows((const unsigned char*)x, dtype, 0, rows, cols, op, out_idx, (unsigned char*)out_val);
        return 1;
    }
    pthread_t th[256];
    int live[256];
    oracle_job jobs[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].x = (const unsigned char*)x;
        jobs[t].dtype = dtype;
        jobs[t].op = op;
        jobs[t].r0 = rows * t / nthreads;
        jobs[t].r1 = rows * (t + 1) / nthreads;
        jobs[t].cols = cols;
        jobs[t].out_idx = out_idx;
        jobs[t].out_val = (unsigned char*)out_val;
        live[t] = pthread_create(&th[t], NULL, run_job, &jobs[t]) == 0;
        if (live[t])
            ++started;
        else
            run_job(&jobs[t]); /* no thread available: scan this range here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (live[t]) pthread_join(th[t], NULL);
    return started > 0 ? nthreads : 1;
}
