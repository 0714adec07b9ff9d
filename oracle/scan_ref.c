/*
 * oracle/scan_ref.c -- plain, sequential CPU reference for device-wide prefix
 * sums and order-preserving stream compaction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this code.  It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Every function is the textbook definition written out as one sequential
 * loop, with no blocking, reordering or fusion:
 *
 *   inclusive  y_i = sum_{j <= i} x_j      exclusive  y_i = sum_{j < i} x_j
 *
 * ("Prefix sum and other parallel patterns", Definitions and self-test
 * answer 1; "CUDA prefix sum, the Hillis-Steele scan", Two scans, and which
 * one hands you the total.)  The running-sum loop is the CPU reference the
 * pages themselves use ("Prefix sum and other parallel patterns", scan.cu
 * main: acc loop).
 *
 * Readings where the pages are silent:
 *   - int32 sums wrap in two's complement.  The exact integer sum is carried
 *     in 64 bits (modulo 2^64, which contains the wanted modulo 2^32) and
 *     only the low 32 bits are stored.
 *   - fp32 inputs are summed in float64 and returned in float64; the fp32
 *     GPU result is compared to that with a normalised error bound.
 *   - compaction keeps element i when flags[i] != 0, in index order; the
 *     number kept is the count ("Prefix sum and other parallel patterns",
 *     Stream compaction and Exercise 1: out[pos[i]] = in[i] where pos is the
 *     exclusive scan of the flags, total = pos[n-1] + flags[n-1]); the
 *     predicate form keeps element i when x[i] > 0 in the element's type.
 *   - MoE offsets: each expert's segment is rounded up to a whole number of
 *     `align`-element GEMM tiles, and ids outside [0, E) are not counted.
 *
 * Parity pins: every function here is checked in tests/ against the pages'
 * worked examples (tests/golden/), closed forms, invariants and brute force;
 * see the test files for which pin covers which function.
 */
#include <stddef.h>
#include <stdint.h>

/* int32 scan with two's-complement wraparound. */
void oracle_scan_i32(const int32_t *x, int32_t *y, size_t n, int inclusive)
{
    uint64_t acc = 0; /* exact sum modulo 2^64 */
    for (size_t i = 0; i < n; ++i) {
        uint64_t xi = (uint64_t)(int64_t)x[i];
        if (inclusive) {
            acc += xi;
            y[i] = (int32_t)(uint32_t)acc;
        } else {
            y[i] = (int32_t)(uint32_t)acc;
            acc += xi;
        }
    }
}

/* uint32 scan modulo 2^32. */
void oracle_scan_u32(const uint32_t *x, uint32_t *y, size_t n, int inclusive)
{
    uint64_t acc = 0;
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc += x[i];
            y[i] = (uint32_t)acc;
        } else {
            y[i] = (uint32_t)acc;
            acc += x[i];
        }
    }
}

/* fp32 inputs, float64 running sum and float64 outputs. */
void oracle_scan_f32(const float *x, double *y, size_t n, int inclusive)
{
    double acc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc += (double)x[i];
            y[i] = acc;
        } else {
            y[i] = acc;
            acc += (double)x[i];
        }
    }
}

/*
 * Widened and 64-bit scans ("Parallel Prefix Sum (Scan) for NVIDIA T4
 * (sm_75)", Key Features: 64-bit indexing for large arrays; a 32-bit sum of
 * many 32-bit counts wraps, so the sum is carried in 64 bits).
 *   u32 -> u64: the exact sum (it cannot exceed 2^64 for n < 2^32).
 *   i32 -> i64: the exact signed sum.
 *   i64 (and u64, the same bits): two's-complement wraparound modulo 2^64,
 *       carried in uint64 arithmetic.
 */
void oracle_scan_u32_u64(const uint32_t *x, uint64_t *y, size_t n, int inclusive)
{
    uint64_t acc = 0;
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc += x[i];
            y[i] = acc;
        } else {
            y[i] = acc;
            acc += x[i];
        }
    }
}

void oracle_scan_i32_i64(const int32_t *x, int64_t *y, size_t n, int inclusive)
{
    int64_t acc = 0;
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc += x[i];
            y[i] = acc;
        } else {
            y[i] = acc;
            acc += x[i];
        }
    }
}

void oracle_scan_i64(const int64_t *x, int64_t *y, size_t n, int inclusive)
{
    uint64_t acc = 0;
    for (size_t i = 0; i < n; ++i) {
        if (inclusive) {
            acc += (uint64_t)x[i];
            y[i] = (int64_t)acc;
        } else {
            y[i] = (int64_t)acc;
            acc += (uint64_t)x[i];
        }
    }
}

/*
 * fp64 scan.  A float64 running sum would carry the same order of rounding
 * error as the GPU result it is meant to judge, so the running sum is kept
 * compensated: Neumaier's variant of Kahan summation (A. Neumaier,
 * "Rundungsfehleranalyse einiger Verfahren zur Summation endlicher Summen",
 * ZAMM 54, 1974) carries the rounding error of every add in `comp` and adds
 * it back when an output is taken.  Each output is then within about one
 * rounding of the exact prefix, whatever n is.
 */
void oracle_scan_f64(const double *x, double *y, size_t n, int inclusive)
{
    double sum = 0.0, comp = 0.0;
    for (size_t i = 0; i < n; ++i) {
        if (!inclusive)
            y[i] = sum + comp;
        double v = x[i];
        double t = sum + v;
        double av = v < 0.0 ? -v : v, as = sum < 0.0 ? -sum : sum;
        if (as >= av)
            comp += (sum - t) + v;
        else
            comp += (v - t) + sum;
        sum = t;
        if (inclusive)
            y[i] = sum + comp;
    }
}

/* Error normaliser for fp64 parity: a_i = sum_{j <= i} |x_j|, compensated. */
void oracle_abs_prefix_f64(const double *x, double *y, size_t n)
{
    double sum = 0.0, comp = 0.0;
    for (size_t i = 0; i < n; ++i) {
        double v = x[i] < 0.0 ? -x[i] : x[i];
        double t = sum + v;
        if (sum >= v)
            comp += (sum - t) + v;
        else
            comp += (v - t) + sum;
        sum = t;
        y[i] = sum + comp;
    }
}

/* Error normaliser for fp32 parity: a_i = sum_{j <= i} |x_j| in float64. */
void oracle_abs_prefix_f32(const float *x, double *y, size_t n)
{
    double acc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        double v = (double)x[i];
        acc += v < 0.0 ? -v : v;
        y[i] = acc;
    }
}

/*
 * Batched scans: a row-major rows x cols matrix, every row scanned on its
 * own, the running sum starting again from zero at each row (the per-row
 * cumulative sum of top-p sampling, "Prefix sum and other parallel
 * patterns", In LLMs: MoE token dispatch, last paragraph).  Each row is the
 * one-dimensional scan above, applied to that row's elements.
 */
void oracle_scan_i32(const int32_t *x, int32_t *y, size_t n, int inclusive);
void oracle_scan_u32(const uint32_t *x, uint32_t *y, size_t n, int inclusive);
void oracle_scan_f32(const float *x, double *y, size_t n, int inclusive);
void oracle_abs_prefix_f32(const float *x, double *y, size_t n);

void oracle_scan_rows_i32(const int32_t *x, int32_t *y, size_t rows, size_t cols, int inclusive)
{
    for (size_t r = 0; r < rows; ++r)
        oracle_scan_i32(x + r * cols, y + r * cols, cols, inclusive);
}

void oracle_scan_rows_u32(const uint32_t *x, uint32_t *y, size_t rows, size_t cols, int inclusive)
{
    for (size_t r = 0; r < rows; ++r)
        oracle_scan_u32(x + r * cols, y + r * cols, cols, inclusive);
}

void oracle_scan_rows_f32(const float *x, double *y, size_t rows, size_t cols, int inclusive)
{
    for (size_t r = 0; r < rows; ++r)
        oracle_scan_f32(x + r * cols, y + r * cols, cols, inclusive);
}

void oracle_abs_prefix_rows_f32(const float *x, double *y, size_t rows, size_t cols)
{
    for (size_t r = 0; r < rows; ++r)
        oracle_abs_prefix_f32(x + r * cols, y + r * cols, cols);
}

/*
 * Segmented scans: segment s is [offsets[s], offsets[s+1]) for s < S, with
 * offsets[0] = 0, offsets[S] = n and offsets non-decreasing (empty segments
 * allowed); every segment is scanned on its own, from zero.  Batched rows are
 * the case offsets[s] = s * cols.
 */
void oracle_scan_segments_i32(const int32_t *x, int32_t *y, size_t n, const uint64_t *offsets, size_t S,
                              int inclusive)
{
    (void)n;
    for (size_t s = 0; s < S; ++s)
        oracle_scan_i32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]), inclusive);
}

void oracle_scan_segments_u32(const uint32_t *x, uint32_t *y, size_t n, const uint64_t *offsets, size_t S,
                              int inclusive)
{
    (void)n;
    for (size_t s = 0; s < S; ++s)
        oracle_scan_u32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]), inclusive);
}

void oracle_scan_segments_f32(const float *x, double *y, size_t n, const uint64_t *offsets, size_t S,
                              int inclusive)
{
    (void)n;
    for (size_t s = 0; s < S; ++s)
        oracle_scan_f32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]), inclusive);
}

void oracle_abs_prefix_segments_f32(const float *x, double *y, size_t n, const uint64_t *offsets, size_t S)
{
    (void)n;
    for (size_t s = 0; s < S; ++s)
        oracle_abs_prefix_f32(x + offsets[s], y + offsets[s], (size_t)(offsets[s + 1] - offsets[s]));
}


/*
 * Order-preserving compaction: copy keys[i] for every i with flags[i] != 0,
 * in index order.  Returns the number kept.  `out` must hold n elements.
 */
uint64_t oracle_compact_u32(const uint32_t *keys, const uint8_t *flags,
                            uint32_t *out, size_t n)
{
    uint64_t count = 0;
    for (size_t i = 0; i < n; ++i) {
        if (flags[i] != 0) {
            out[count] = keys[i];
            count += 1;
        }
    }
    return count;
}

/*
 * Predicate form of the same compaction: keep keys[i] when keys[i] > 0
 * (the predicate of "Prefix sum and other parallel patterns", compact.cu and
 * Exercise 1), order preserved.  Returns the number kept.
 */
uint64_t oracle_compact_positive_f32(const float *x, float *out, size_t n)
{
    uint64_t count = 0;
    for (size_t i = 0; i < n; ++i) {
        if (x[i] > 0.0f) {
            out[count] = x[i];
            count += 1;
        }
    }
    return count;
}

/* The same predicate in the other element types: signed for int32, and
 * "nonzero" for uint32 (an unsigned value is > 0 exactly when it is not 0). */
uint64_t oracle_compact_positive_i32(const int32_t *x, int32_t *out, size_t n)
{
    uint64_t count = 0;
    for (size_t i = 0; i < n; ++i) {
        if (x[i] > 0) {
            out[count] = x[i];
            count += 1;
        }
    }
    return count;
}

uint64_t oracle_compact_positive_u32(const uint32_t *x, uint32_t *out, size_t n)
{
    uint64_t count = 0;
    for (size_t i = 0; i < n; ++i) {
        if (x[i] > 0u) {
            out[count] = x[i];
            count += 1;
        }
    }
    return count;
}

/*
 * MoE token counts and aligned offsets ("Prefix sum and other parallel
 * patterns", In LLMs: MoE token dispatch, steps 1-2, and Exercise 2):
 *   counts[e]    = number of i < m with ids[i] == e        (the histogram)
 *   offsets[0]   = 0
 *   offsets[e+1] = offsets[e] + align * ceil(counts[e] / align)
 * i.e. the exclusive prefix sum of the counts, each expert's segment rounded
 * up to a multiple of the GEMM tile size `align`, so that offsets[e] is where
 * expert e's tokens start and offsets[E] the padded total.  An id outside
 * [0, E) belongs to no expert here and is not counted.  `offsets` holds E+1
 * entries.
 */
void oracle_moe_counts_offsets(const int32_t *ids, size_t m, int32_t num_experts, uint32_t align,
                               uint32_t *counts, uint64_t *offsets)
{
    for (int32_t e = 0; e < num_experts; ++e)
        counts[e] = 0;
    for (size_t i = 0; i < m; ++i) {
        if (ids[i] >= 0 && ids[i] < num_experts)
            counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < num_experts; ++e) {
        uint64_t blocks = ((uint64_t)counts[e] + align - 1) / align;
        offsets[e + 1] = offsets[e] + blocks * align;
    }
}
