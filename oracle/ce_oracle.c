/*
 * ce_oracle.c -- the plain, slow CPU oracle of the row-wise softmax
 * cross-entropy path: per-row loss, mean loss, gradient and row argmax;
 * beside them, the rows a language model's step reads from the same logits:
 * softmax and log-softmax rows, sampling candidates, and split sums.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline call this file. The CUDA library shares no code, header, table
 * or constant with it, and neither includes nor links the other.
 *
 * Everything is computed in f64 from the f32 inputs (each input is widened
 * once), one row at a time, one column at a time, in column order, with no
 * blocking, vectorisation or fast-math -- but for one diagnostic,
 * oracle_ce_rows_page_f32, which is f32 on purpose and graded by no test.
 * Build with plain gcc, e.g.
 *     gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared ce_oracle.c -lm
 *
 * Source of every definition: the API reference page "gizml:netops"
 * (gizstack.com/docs/reference/gizml/netops.md), section Functions:
 * crossEntropyLoss, crossEntropyRows, crossEntropyGrad, argmaxInto,
 * candidatesInto, splitSumInto; section Methods: Tensor.argmax; section
 * Constants: TOP_EACH, CANDIDATE_ROW. The softmax and log-softmax rows also
 * cite the gpukit API page (dev.nu, gkd_softmax_rows) and the guide
 * "Tensors, GPU kernels and AI models" (Step 5, a request's logprobs).
 *
 * Layout: row i of the logits starts at logits + i * stride; only its first
 * `vocab` columns are read. Labels are int64, one per row. The gradient is
 * written dense, [rows, vocab].
 */
#include <math.h>
#include <stdint.h>

#define ORACLE_VERSION 3

int oracle_version(void) { return ORACLE_VERSION; }

/*
 * Statistics of one row, as the crossEntropyLoss entry defines them:
 *   m  = max_j x_j                    (the row max)
 *   s  = sum_j exp(x_j - m)           (the row's exp-sum)
 *   loss = m + log(s) - x[label].
 * s is split as s = 1 + t: the 1 is the term of the first column j* that
 * holds m (exp(0) = 1) and t sums the other columns. Then
 *   loss = (m - x[label]) + log1p(t),
 * which is the entry's expression rearranged; it is exact in real arithmetic
 * and keeps the value of a loss far below 1e-16 (a label at the row max with
 * every other logit far below), where m + log(s) - x[label] cancels in any
 * floating point format.
 *
 * The IEEE evaluation of the entry's expression is NaN for a row that holds a
 * NaN, that holds +inf (x_j* - m = inf - inf), or whose entries are all -inf
 * (every x_j - m = -inf - (-inf)). The rearranged form never forms those
 * differences, so it flags the three cases explicitly (`degenerate`).
 */
typedef struct {
    double m;     /* row max */
    int64_t jmax; /* first column holding m */
    double t;     /* sum of exp(x_j - m) over j != jmax */
    int degenerate;
} row_stats;

static row_stats stats_of_row(const float *x, int64_t vocab)
{
    row_stats r;
    r.m = -INFINITY;
    r.jmax = 0;
    r.t = 0.0;
    r.degenerate = 0;

    int any_nan = 0;
    int seen = 0;
    for (int64_t j = 0; j < vocab; ++j) {
        double v = (double)x[j];
        if (isnan(v)) {
            any_nan = 1;
            continue;
        }
        if (!seen || v > r.m) {
            r.m = v;
            r.jmax = j;
            seen = 1;
        }
    }
    if (any_nan || !seen || isinf(r.m)) {
        /* NaN present, all NaN, +inf max, or every entry -inf */
        r.degenerate = 1;
        r.t = NAN;
        return r;
    }
    double t = 0.0;
    for (int64_t j = 0; j < vocab; ++j) {
        if (j == r.jmax)
            continue;
        t += exp((double)x[j] - r.m);
    }
    r.t = t;
    return r;
}

/*
 * crossEntropyRows: each row's loss m + log(sum exp(x - m)) - x[label].
 * A label outside [0, vocab) gives a NaN loss for its row.
 * loss_out: rows doubles. Returns 0, or -1 on a bad argument.
 */
int oracle_ce_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                   const int64_t *labels, double *loss_out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        int64_t label = labels[i];
        row_stats st = stats_of_row(x, vocab);
        if (st.degenerate || label < 0 || label >= vocab) {
            loss_out[i] = NAN;
            continue;
        }
        loss_out[i] = (st.m - (double)x[label]) + log1p(st.t);
    }
    return 0;
}

/*
 * Diagnostic, not a reference (parity unpinned): crossEntropyRows computed
 * the way the entry of crossEntropyLoss ("gizml:netops", Functions) writes
 * it, in f32: m + log(sum exp(x - m)) - x[label] with "the sum in 16 lanes".
 * The entry fixes neither which column goes to which lane nor how the lanes
 * are joined; this reads them as 16 f32 partial sums, lane = column mod 16,
 * joined pairwise in a tree of fixed shape (the join the page "Compute: all
 * of the hardware from one program", section Parts, gives its strict sums).
 * The max skips NaN (a compare with NaN is false); a NaN entry then makes
 * the sum NaN. Every operation is f32: expf, logf, adds in the order above.
 * It shows what the literal f32 form loses where the label holds a dominant
 * max (m + log(s) with s just above 1 rounds the loss away).
 * loss_out: rows floats. Returns 0, or -1 on a bad argument.
 */
int oracle_ce_rows_page_f32(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                            const int64_t *labels, float *loss_out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        const int64_t label = labels[i];
        float m = -INFINITY;
        for (int64_t j = 0; j < vocab; ++j)
            if (x[j] > m)
                m = x[j];
        float lane[16];
        for (int k = 0; k < 16; ++k)
            lane[k] = 0.0f;
        for (int64_t j = 0; j < vocab; ++j)
            lane[j % 16] += expf(x[j] - m);
        for (int w = 8; w >= 1; w /= 2)
            for (int k = 0; k < w; ++k)
                lane[k] = lane[k] + lane[k + w];
        if (label < 0 || label >= vocab) {
            loss_out[i] = NAN;
            continue;
        }
        const float ms = m + logf(lane[0]);
        loss_out[i] = ms - x[label];
    }
    return 0;
}

/*
 * crossEntropyGrad: (softmax - onehot) * scale, softmax_j = exp(x_j - m) / s.
 * The entry's "f32 of 1/sum" is a statement about the f32 arithmetic of a
 * device; here 1/s is taken in f64 (the mathematical softmax).
 * A degenerate row (NaN, +inf, or all -inf) gives a NaN gradient row.
 * A label outside [0, vocab) gets no one-hot term (and a NaN loss).
 * grad_out: rows * vocab doubles, dense. loss_out (nullable): rows doubles.
 */
int oracle_ce_grad(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                   const int64_t *labels, double scale, double *grad_out, double *loss_out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        double *g = grad_out + i * vocab;
        int64_t label = labels[i];
        int label_ok = (label >= 0 && label < vocab);
        row_stats st = stats_of_row(x, vocab);
        if (st.degenerate) {
            for (int64_t j = 0; j < vocab; ++j)
                g[j] = NAN;
            if (loss_out)
                loss_out[i] = NAN;
            continue;
        }
        double s = 1.0 + st.t;
        for (int64_t j = 0; j < vocab; ++j) {
            double p = exp((double)x[j] - st.m) / s;
            double onehot = (label_ok && j == label) ? 1.0 : 0.0;
            g[j] = (p - onehot) * scale;
        }
        if (loss_out)
            loss_out[i] = label_ok ? (st.m - (double)x[label]) + log1p(st.t) : NAN;
    }
    return 0;
}

/*
 * crossEntropyLoss: the mean of the row losses, summed in f64 in row order.
 * The mean of no rows is NaN (0/0).
 */
double oracle_ce_mean(const double *loss_rows, int64_t rows)
{
    double sum = 0.0;
    for (int64_t i = 0; i < rows; ++i)
        sum += loss_rows[i];
    return sum / (double)rows;
}

/*
 * argmaxInto / Tensor.argmax: the index of each row's largest element among
 * its first `vocab` columns; the first of equals wins and NaN never wins. A
 * row with no non-NaN entry gives 0. -0 and +0 are equal (the first wins).
 * idx_out: rows int64.
 */
int oracle_argmax(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                  int64_t *idx_out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        int64_t best = 0;
        double best_v = 0.0;
        int seen = 0;
        for (int64_t j = 0; j < vocab; ++j) {
            double v = (double)x[j];
            if (isnan(v))
                continue;
            if (!seen || v > best_v) {
                best = j;
                best_v = v;
                seen = 1;
            }
        }
        idx_out[i] = best;
    }
    return 0;
}

/*
 * Softmax rows: p_j = exp(x_j - m) / s, the softmax of the crossEntropyGrad
 * entry without its one-hot term and scale (also the "row softmax" of the
 * ready-made device kernels, gkd_softmax_rows, on the gpukit API page,
 * dev.nu). 1/s is taken in f64 (the mathematical softmax). A degenerate row
 * (NaN, +inf, or all -inf) gives a NaN row. out: rows * vocab doubles, dense.
 */
int oracle_softmax(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                   double *out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        double *o = out + i * vocab;
        row_stats st = stats_of_row(x, vocab);
        for (int64_t j = 0; j < vocab; ++j)
            o[j] = st.degenerate ? NAN : exp((double)x[j] - st.m) / (1.0 + st.t);
    }
    return 0;
}

/*
 * Log-softmax rows: log p_j = x_j - m - log(s), the log probabilities of the
 * tokens (the `logprobs` of a request's Sampling, "Tensors, GPU kernels and
 * AI models", Step 5). With s = 1 + t as in stats_of_row:
 *   log p_j = (x_j - m) - log1p(t),
 * which keeps a log probability near 0 (a dominant token) to full relative
 * precision. A degenerate row gives a NaN row; a -inf entry of a finite row
 * gives -inf. out: rows * vocab doubles, dense.
 */
int oracle_log_softmax(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                       double *out)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        double *o = out + i * vocab;
        row_stats st = stats_of_row(x, vocab);
        for (int64_t j = 0; j < vocab; ++j)
            o[j] = st.degenerate ? NAN : ((double)x[j] - st.m) - log1p(st.t);
    }
    return 0;
}

/*
 * candidatesInto (netops, Functions) with the constants TOP_EACH and
 * CANDIDATE_ROW (netops, Constants): a workgroup of 256 threads reads a row;
 * each thread keeps the TOP_EACH = 4 largest logits of the values it reads;
 * a row's candidates are the 256 * 4 kept (value, token) pairs, 2048 floats.
 * The entries leave open which columns a thread reads, the order of a
 * thread's kept values and what fills a slot for which a thread read too
 * few values. This oracle takes the plainest readings:
 *   - thread t reads columns t, t + 256, t + 512, ... below vocab;
 *   - values rank by value, larger first, and among equal values the lower
 *     column first (the first of equals, as argmaxInto); NaN is never kept;
 *   - pair 4t + k holds thread t's rank-k value: float 2(4t + k) is the value,
 *     float 2(4t + k) + 1 the column as f32;
 *   - a slot with no value holds (-inf, -1).
 * cand: rows * 2048 floats (the values are copies of the logits, so nothing
 * here is rounded).
 */
#define CAND_THREADS 256
#define CAND_KEEP 4

int oracle_candidates(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                      float *cand)
{
    if (rows < 0 || vocab < 1 || stride < vocab)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        float *out = cand + i * (int64_t)(2 * CAND_THREADS * CAND_KEEP);
        for (int t = 0; t < CAND_THREADS; ++t) {
            float kv[CAND_KEEP];
            int64_t kc[CAND_KEEP];
            int kept = 0;
            for (int64_t j = t; j < vocab; j += CAND_THREADS) {
                float v = x[j];
                if (isnan(v))
                    continue;
                /* where v ranks among the kept values: below every kept value
                   that is larger or equal (equal ones have lower columns) */
                int pos = 0;
                while (pos < kept && kv[pos] >= v)
                    ++pos;
                if (pos >= CAND_KEEP)
                    continue;
                int last = kept < CAND_KEEP ? kept : CAND_KEEP - 1;
                for (int q = last; q > pos; --q) {
                    kv[q] = kv[q - 1];
                    kc[q] = kc[q - 1];
                }
                kv[pos] = v;
                kc[pos] = j;
                if (kept < CAND_KEEP)
                    ++kept;
            }
            for (int k = 0; k < CAND_KEEP; ++k) {
                float *slot = out + 2 * (CAND_KEEP * t + k);
                slot[0] = k < kept ? kv[k] : -INFINITY;
                slot[1] = k < kept ? (float)kc[k] : -1.0f;
            }
        }
    }
    return 0;
}

/*
 * splitSumInto (netops, Functions): the `total` values at y and `splits`
 * parts at p. Reading: part s is the `total` f32 values at p + s * total;
 *   y[i] = (add ? y[i] : 0) + sum_{s = 0 .. splits-1} p[s * total + i],
 * summed in f64 in split order. With add = 0 the old y is never read.
 * y_out: total doubles (y_in is read only when add != 0).
 */
int oracle_split_sum(const float *y_in, const float *p, int64_t total, int64_t splits, int add,
                     double *y_out)
{
    if (total < 0 || splits < 1)
        return -1;
    for (int64_t i = 0; i < total; ++i) {
        double acc = add ? (double)y_in[i] : 0.0;
        for (int64_t s = 0; s < splits; ++s)
            acc += (double)p[s * total + i];
        y_out[i] = acc;
    }
    return 0;
}

/*
 * Vocab-sharded cross-entropy: the row statistics of one column slice of the
 * rows, and their combination over the slices. crossEntropyLoss (netops,
 * Functions) defines the loss through the row max m and the row's exp-sum
 * s = sum_j exp(x_j - m); both decompose over any split of the columns:
 *   m = max_s m_s,  s = sum_s exp(m_s - m) * s_s,
 * so a row split over slices (e.g. a language-model head whose vocabulary is
 * split over several devices) needs only each slice's (m_s, s_s), its first
 * max column and, from the slice that holds it, x[label].
 *
 * oracle_ce_stats: for the slice [col0, col0 + vocab) of each row, whose
 * columns are at logits + i * stride (so `logits` points at column col0),
 * four doubles per row:
 *   [0] m   the max of the slice's non-NaN values (-inf if none);
 *   [1] t   sum of exp(x_j - m) over the slice but its first column holding
 *           m; NaN if the slice holds a NaN or m = +inf; 0 if m = -inf;
 *   [2] top the global column (col0 + j) of the first element holding m, or
 *           -1 if the slice has no non-NaN value;
 *   [3] xl  x[label] if col0 <= label < col0 + vocab, else 0.
 */
int oracle_ce_stats(const float *logits, int64_t rows, int64_t vocab, int64_t stride, int64_t col0,
                    const int64_t *labels, double *stats_out)
{
    if (rows < 0 || vocab < 1 || stride < vocab || col0 < 0)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const float *x = logits + i * stride;
        double *o = stats_out + 4 * i;
        double m = -INFINITY;
        int64_t jmax = -1;
        int any_nan = 0;
        for (int64_t j = 0; j < vocab; ++j) {
            double v = (double)x[j];
            if (isnan(v)) {
                any_nan = 1;
                continue;
            }
            if (jmax < 0 || v > m) {
                m = v;
                jmax = j;
            }
        }
        double t = 0.0;
        if (any_nan || m == INFINITY) {
            t = NAN;
        } else if (m != -INFINITY) {
            for (int64_t j = 0; j < vocab; ++j)
                if (j != jmax)
                    t += exp((double)x[j] - m);
        }
        int64_t local = labels[i] - col0;
        o[0] = m;
        o[1] = t;
        o[2] = jmax < 0 ? -1.0 : (double)(col0 + jmax);
        o[3] = (local >= 0 && local < vocab) ? (double)x[local] : 0.0;
    }
    return 0;
}

/*
 * The combination of `shards` slices' statistics (stats: shards * rows * 4
 * doubles, slice-major, as oracle_ce_stats writes them) into each whole row's
 *   M = max_s m_s, and the first column holding it: the lowest top among the
 *       slices with m_s = M (0 if no slice has a non-NaN value);
 *   T = the row's exp-sum relative to M less the one term of that column:
 *       t_s of its slice s*, plus (1 + t_s) exp(m_s - M) of every other slice
 *       (0 for a slice with m_s = -inf);
 *   loss = (M - x[label]) + log1p(T), x[label] the sum of the slices' xl (0
 *       from every slice but the label's); NaN if the label is outside
 *       [0, vocab_total), or if the row holds a NaN (some t_s is NaN) or M is
 *       infinite, as crossEntropyRows' value on the whole row.
 * loss_out, top_out (int64), m_out, t_out: rows each; any may be NULL.
 */
int oracle_ce_stats_combine(const double *stats, int64_t shards, int64_t rows, int64_t vocab_total,
                            const int64_t *labels, double *loss_out, int64_t *top_out, double *m_out,
                            double *t_out)
{
    if (shards < 1 || rows < 0 || vocab_total < 1)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        double M = -INFINITY, xl = 0.0;
        int any_nan_t = 0;
        for (int64_t s = 0; s < shards; ++s) {
            const double *st = stats + 4 * (s * rows + i);
            if (st[0] > M)
                M = st[0];
            if (isnan(st[1]))
                any_nan_t = 1;
            xl += st[3];
        }
        int64_t star = -1;
        double top = -1.0;
        for (int64_t s = 0; s < shards; ++s) {
            const double *st = stats + 4 * (s * rows + i);
            if (st[0] == M && st[2] >= 0.0 && (top < 0.0 || st[2] < top)) {
                top = st[2];
                star = s;
            }
        }
        int degenerate = any_nan_t || isinf(M) || star < 0;
        double T = NAN;
        if (!degenerate) {
            T = 0.0;
            for (int64_t s = 0; s < shards; ++s) {
                const double *st = stats + 4 * (s * rows + i);
                if (s == star)
                    T += st[1];
                else if (st[0] != -INFINITY)
                    T += (1.0 + st[1]) * exp(st[0] - M);
            }
        }
        int label_ok = labels[i] >= 0 && labels[i] < vocab_total;
        if (loss_out)
            loss_out[i] = (degenerate || !label_ok) ? NAN : (M - xl) + log1p(T);
        if (top_out)
            top_out[i] = top < 0.0 ? 0 : (int64_t)top;
        if (m_out)
            m_out[i] = M;
        if (t_out)
            t_out[i] = T;
    }
    return 0;
}
