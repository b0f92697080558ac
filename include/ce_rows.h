/*
 * ce_rows.h -- C ABI of the row-wise softmax cross-entropy library for
 * NVIDIA GB300 (sm_103a): per-row loss, mean loss, fused loss + gradient,
 * and the row argmax that closes a decode step; beside them, the rows a
 * language model's step reads from the same logits (softmax, log-softmax,
 * sampling candidates) and the join of split partial sums.
 *
 * Definitions follow the API reference page "gizml:netops"
 * (gizstack.com/docs/reference/gizml/netops.md), section Functions:
 * crossEntropyRows, crossEntropyLoss, crossEntropyGrad, argmaxInto,
 * candidatesInto, splitSumInto; section Methods: Tensor.argmax; section
 * Constants: TOP_EACH, CANDIDATE_ROW.
 *
 * Common conventions of every entry point:
 *  - Logits are f32, row-major: row i starts at logits + i * stride
 *    (elements); only its first `vocab` columns are read, the padding
 *    columns vocab..stride-1 never are.
 *  - Labels are int64, one per row. Outputs are written per row; the
 *    gradient is written dense, [rows, vocab] (row i at grad + i * vocab).
 *  - All pointers are DEVICE pointers on the current CUDA device, owned by
 *    the caller; the library keeps none of them after the call returns and
 *    allocates no memory per call.
 *  - Every call only enqueues work on `stream` (NULL: the legacy default
 *    stream) and returns; nothing waits for the GPU. A result is ready once
 *    the stream has reached it.
 *  - Arguments are checked on the host before anything is launched; a
 *    rejected call returns a negative status and launches nothing:
 *      CE_EINVAL: a required pointer is NULL (while rows > 0), rows < 0,
 *                 vocab < 1, stride < vocab, vocab > 2^24 (the token
 *                 written as f32 must be exact), or a non-finite scale;
 *      CE_EALIGN: a pointer is not aligned to its element size;
 *      CE_ECUDA:  the CUDA runtime reported an error at launch
 *                 (ce_last_cuda_error() gives its code).
 *  - rows == 0 is valid and launches nothing, except that ce_loss, ce_mean
 *    and ce_grad_step (given a loss_mean) still write their mean (NaN: the
 *    mean of no rows).
 *  - A label outside [0, vocab) is found on the device: that row's loss
 *    is NaN, its gradient row gets no one-hot term, and a device counter
 *    (read by ce_device_error_count) is incremented. Nothing traps.
 *  - A row holding a NaN or +inf, or whose entries are all -inf, has a NaN
 *    loss and a NaN gradient row (the IEEE value of the definition). Its
 *    argmax still follows Tensor.argmax: NaN never wins, first of equals.
 */
#ifndef CE_ROWS_H
#define CE_ROWS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of this ABI are the library's only exported ones. */
#if defined(__GNUC__)
#define CE_API __attribute__((visibility("default")))
#else
#define CE_API
#endif

/* The CUDA runtime's cudaStream_t, without requiring CUDA headers. */
typedef struct CUstream_st *ce_stream_t;

enum ce_status {
    CE_OK = 0,
    CE_EINVAL = -1,
    CE_EALIGN = -2,
    CE_ECUDA = -3,
    CE_EDEVICE = -4, /* no CUDA device, or not an sm_103 device */
    CE_ERANGE = -5,  /* argmax_rows_noalloc: more rows than its fixed scratch holds */
};

/*
 * crossEntropyRows (gizml:netops, Functions): each row's loss
 *     m + log(sum_j exp(x_j - m)) - x[label],   m = max_j x_j,
 * as f32 into loss_rows[rows], computed on the device without a host wait.
 * The kernel evaluates the equal form (m - x[label]) + log1p(t), where t
 * sums exp(x_j - m) over all columns but one holding m, so a loss far below
 * the f32 resolution of m keeps its relative accuracy.
 *   logits:    [rows, stride] f32, read only.
 *   labels:    [rows] int64, read only.
 *   loss_rows: [rows] f32, written; must not overlap the inputs.
 */
CE_API int ce_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
            const int64_t *labels, float *loss_rows, ce_stream_t stream);

/*
 * The mean step of crossEntropyLoss (gizml:netops, Functions): the mean of
 * `rows` f32 row losses, accumulated in f64, written as one double to
 * *loss_mean (a device pointer; the value stays on the device, so a
 * recorded step never waits for it). The sum is a fixed-shape tree over a
 * cluster of CTAs that does not depend on the device: the same inputs give
 * the same bits on every run. The kernel is launched as a programmatic
 * dependent of the kernel before it on `stream` (it waits for that kernel to
 * complete before reading anything), so after this library's row kernels it
 * starts without a launch gap.
 *   loss_rows: [rows] f32, read only.   loss_mean: 1 double, written.
 */
CE_API int ce_mean(const float *loss_rows, int64_t rows, double *loss_mean, ce_stream_t stream);

/*
 * crossEntropyLoss (gizml:netops, Functions): ce_rows followed by ce_mean,
 * both enqueued on `stream`. loss_rows ([rows] f32) is required: it holds
 * the row losses (an output) that the mean reads.
 */
CE_API int ce_loss(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
            const int64_t *labels, float *loss_rows, double *loss_mean, ce_stream_t stream);

/*
 * crossEntropyGrad (gizml:netops, Functions): the gradient
 *     grad[i, j] = (softmax_ij - [j == label_i]) * scale,
 *     softmax_ij = exp(x_ij - m_i) * f32(1 / sum_i),
 * with `scale` (e.g. 1/rows, the gradient of the mean over rows) rounded to
 * f32. One kernel reads each logit once from HBM and writes each gradient
 * once; from the same read it can also write each row's loss (as ce_rows).
 *   logits:    [rows, stride] f32, read only, unless grad == logits.
 *   labels:    [rows] int64, read only.
 *   grad:      [rows, vocab] f32 dense, written. grad == logits (in place)
 *              is allowed when stride == vocab; any other overlap is not.
 *   loss_rows: [rows] f32, or NULL.
 */
CE_API int ce_grad(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
            const int64_t *labels, double scale, float *grad, float *loss_rows, ce_stream_t stream);

/*
 * The whole training-step path from one read of the logits: ce_grad's
 * gradient and row losses, each row's argmax token (argmaxInto's rule, as
 * argmax_rows writes it) and the mean loss (crossEntropyLoss, as ce_mean
 * writes it). Arguments as ce_grad, and:
 *   top:       [rows] f32, or NULL.
 *   loss_mean: 1 double on the device, or NULL; needs loss_rows (CE_EINVAL
 *              otherwise). The mean kernel is launched as a programmatic
 *              dependent of the fused kernel: it is scheduled while the fused
 *              kernel finishes and reads the row losses only once that kernel
 *              has completed, so the step costs no separate launch gap.
 */
CE_API int ce_grad_step(const float *logits, int64_t rows, int64_t vocab, int64_t stride,
                        const int64_t *labels, double scale, float *grad, float *loss_rows, float *top,
                        double *loss_mean, ce_stream_t stream);

/*
 * crossEntropyGrad and crossEntropyLoss of a batch that is in HOST memory:
 * the training step fed from the host, with the host-to-device copy
 * overlapped with the kernels. The labels, then the logits in chunks of
 * rows, are copied into caller-owned device buffers on a copy stream the
 * library keeps per device; the fused kernel (as ce_grad_step, with the
 * tokens) runs on each chunk on `stream` as soon as that chunk has landed, so
 * chunk c is computed while chunk c + 1 is copied. Then ce_mean over all the
 * rows, and the mean and tokens back to the host. Everything is enqueued: the call returns at once, and the host and
 * device buffers must stay valid, and the host outputs unread, until
 * `stream` has reached this point. Host inputs in page-locked memory copy
 * asynchronously; pageable ones work but the copies may block the caller.
 *   logits_h:    [rows, stride_h] f32, host, read only.
 *   labels_h:    [rows] int64, host, read only.
 *   logits_d:    [rows, vocab] f32 dense, device, written (the staged copy).
 *   labels_d:    [rows] int64, device, written.
 *   grad:        [rows, vocab] f32 dense, device, written; grad == logits_d
 *                (the gradient over the staged copy) is allowed.
 *   loss_rows:   [rows] f32, device, written.   top: [rows] f32 device or NULL.
 *   loss_mean:   1 double, device, written.
 *   loss_mean_h: 1 double, host, or NULL.    top_h: [rows] f32 host or NULL
 *                (needs top).
 *   chunk_rows:  rows per copied chunk; 0 picks 16 chunks (at most 64).
 * Calls that share device buffers must be ordered by their streams. The
 * same argument checks as ce_grad apply (CE_EINVAL / CE_EALIGN before any
 * copy); rows == 0 writes a NaN mean.
 */
CE_API int ce_grad_host(const float *logits_h, int64_t rows, int64_t vocab, int64_t stride_h,
                        const int64_t *labels_h, double scale, float *logits_d, int64_t *labels_d,
                        float *grad, float *loss_rows, float *top, double *loss_mean,
                        double *loss_mean_h, float *top_h, int64_t chunk_rows, ce_stream_t stream);

/*
 * argmaxInto (gizml:netops, Functions) with Tensor.argmax's rule (Methods):
 * over `rows` rows of `stride` elements, the index of the largest of the
 * first `vocab` entries -- the first of equals; NaN never wins; a row with
 * no non-NaN entry gives 0 -- written as f32 (exact, since vocab <= 2^24)
 * into top[rows]. The direct form (rows at logits + i * stride); for rows
 * given by a table of addresses see argmax_rows_indirect.
 *   logits:    [rows, stride] f32, read only.   top: [rows] f32, written.
 */
CE_API int argmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *top,
                       ce_stream_t stream);

/*
 * argmax_rows_noalloc -- the tokens of argmax_rows (same rule, same f32
 * output) for callers that must not allocate device memory: code running
 * inside another runtime that owns and pre-plans every byte of device memory
 * (an inference server's memory planner, a plugin handed only its inputs
 * and outputs), and latency-critical decode loops where a cudaMalloc -- which
 * can synchronise the whole device -- is not acceptable. The pages have no
 * counterpart: argmaxInto takes no workspace.
 *
 * It allocates nothing: its scratch is a fixed 64 KiB array in the library's
 * own device memory (one 64-bit key per segment of the rows' even split over
 * the GPU), held on every device that loads the library until the process
 * exits. The caller still passes the logits and `top` as in argmax_rows.
 *   - A call with rows + 2 * (SMs of the device) <= 8192 always fits (7888
 *     rows on a 152-SM GB300); a call that does not fit returns CE_ERANGE
 *     and launches nothing.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, no allocation); make that first call
 *     before capturing any stream.
 *   - Every call uses the same array and leaves its contents there. Nothing
 *     in it needs to start at zero (each call reads only keys it wrote), but
 *     two calls that run at the same time on the GPU -- on different streams,
 *     or from different host threads -- race on it and may return wrong
 *     tokens; order them on one stream.
 */
CE_API int argmax_rows_noalloc(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *top,
                               ce_stream_t stream);

/*
 * Softmax rows: out[i, j] = exp(x_ij - m_i) * f32(1 / sum_i), the softmax of
 * crossEntropyGrad (gizml:netops, Functions) without its one-hot term and
 * scale -- the row softmax among the gpukit API page's device kernels
 * (dev.nu, gkd_softmax_rows). Same kernel, same single HBM read of each
 * logit and single write of each output as ce_grad.
 *   logits: [rows, stride] f32, read only, unless out == logits.
 *   out:    [rows, vocab] f32 dense, written. out == logits (in place) is
 *           allowed when stride == vocab; any other overlap is not.
 * A row holding a NaN or +inf, or all -inf, gives a NaN row; a -inf entry of
 * a finite row gives 0.
 */
CE_API int softmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *out,
                        ce_stream_t stream);

/*
 * Log-softmax rows: out[i, j] = (x_ij - m_i) - log(sum_i), the log
 * probabilities of the tokens (a request's `logprobs`, guide "Tensors, GPU
 * kernels and AI models", Step 5). log(sum) is taken as log1p(t), t the sum
 * over all columns but one holding the max, so the log probability of a
 * dominant token keeps its relative accuracy. Layout, aliasing and
 * non-finite rows as softmax_rows; a -inf entry of a finite row gives -inf.
 */
CE_API int log_softmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *out,
                            ce_stream_t stream);

/* candidatesInto's workgroup, TOP_EACH and CANDIDATE_ROW (gizml:netops, Constants). */
#define CE_CANDIDATE_THREADS 256
#define CE_TOP_EACH 4
#define CE_CANDIDATE_ROW 2048

/*
 * candidatesInto (gizml:netops, Functions; Constants TOP_EACH, CANDIDATE_ROW):
 * each row's sampling candidates. A workgroup of CE_CANDIDATE_THREADS = 256
 * threads reads the row; thread t reads columns t, t + 256, t + 512, ...
 * below vocab and keeps its CE_TOP_EACH = 4 largest values, ranked by value
 * and, among equal values, by the lower column (NaN is never kept). Row i's
 * candidates are the CE_CANDIDATE_ROW = 2048 floats at cand + 2048 * i:
 * float 2(4t + k) is thread t's rank-k value and float 2(4t + k) + 1 its
 * column as f32 (exact, vocab <= 2^24); a slot for which thread t read no
 * value holds (-inf, -1). Bit-exact: the values are copies of the logits.
 * The direct form (rows at logits + i * stride); for rows given by a table of
 * addresses see candidates_rows_indirect.
 *   logits: [rows, stride] f32, read only.
 *   cand:   [rows, 2048] f32, written; must not overlap the logits.
 */
CE_API int candidates_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *cand,
                           ce_stream_t stream);

/*
 * argmaxInto and candidatesInto in their indirect form (gizml:netops,
 * Functions): the entries read "rows of `stride`, of the head blocks in
 * `blocks` when `indirect`"; the extracted sentence is garbled, and this
 * library takes its plainest reading -- row i is read at the device address
 * row_addrs[i] instead of at logits + i * stride (rows picked in place, e.g.
 * each sequence's last position, without gathering them first). Same rules,
 * outputs and kernels as argmax_rows / candidates_rows.
 *   row_addrs: [rows] uint64 device addresses of f32 rows, each with `vocab`
 *              readable floats; 8-byte aligned table, read only. Rows may
 *              repeat and may sit anywhere (4-byte aligned).
 *   top:  [rows] f32, written.   cand: [rows, 2048] f32, written.
 * An address that is null or not 4-byte aligned is detected on the device and
 * never read: that row's token is NaN, its candidates all (-inf, -1). The
 * outputs must not overlap any row.
 */
CE_API int argmax_rows_indirect(const uint64_t *row_addrs, int64_t rows, int64_t vocab, float *top,
                                ce_stream_t stream);
CE_API int candidates_rows_indirect(const uint64_t *row_addrs, int64_t rows, int64_t vocab, float *cand,
                                    ce_stream_t stream);

/*
 * splitSumInto (gizml:netops, Functions): joins `splits` partial results of
 * `total` f32 values each (part s at parts + s * total, e.g. the partial
 * products of a split reduction):
 *     y[i] = (add ? y[i] : 0) + parts[0][i] + ... + parts[splits-1][i],
 * added in f32 in split order. With add == 0 the old y is never read.
 *   y:     [total] f32, written (read first when add != 0).
 *   parts: [splits, total] f32, read only. y may be parts itself (part 0),
 *          any other overlap is rejected (CE_EINVAL).
 * total == 0 launches nothing; splits < 1 is CE_EINVAL.
 */
CE_API int split_sum(float *y, const float *parts, int64_t total, int64_t splits, int add, ce_stream_t stream);

/*
 * Vocab-sharded cross-entropy: the loss, token and gradient of rows whose
 * columns are split over slices (e.g. a language-model head whose vocabulary
 * is split over devices), with one exchange of 16 bytes per row and slice.
 * crossEntropyLoss (gizml:netops, Functions) defines the loss by the row max
 * m and exp-sum s = sum_j exp(x_j - m); both decompose over any split of the
 * columns (m = max_s m_s, s = sum_s exp(m_s - m) s_s), so:
 *   1. ce_stats on each slice            -> [rows] float4 per slice;
 *   2. gather the slices' stats in column order (the caller's exchange);
 *   3. ce_stats_combine                  -> each row's loss, token and the
 *                                           combined float4;
 *   4. ce_grad_from_stats on each slice  -> the slice of crossEntropyGrad.
 * The results equal ce_grad's on the whole rows (same rules for ties, NaN,
 * infinities and bad labels), up to f32 rounding order.
 *
 * ce_stats: per row of the slice [col0, col0 + vocab) -- `logits` points at
 * column col0 of row 0, rows `stride` apart -- the float4 (m, t, top, xl):
 *   m   the max of the slice's non-NaN values (-inf if none);
 *   t   sum of exp(x_j - m) over the slice but one element holding m; NaN if
 *       the slice holds a NaN; not meaningful when m is +-inf;
 *   top the global column of the first element holding m as f32, or -1 if
 *       the slice has no non-NaN value;
 *   xl  x[label] if col0 <= label < col0 + vocab, else 0.
 *   labels: [rows] int64 GLOBAL columns.   stats: [rows] x 4 f32, 16-byte
 *   aligned, written. col0 + vocab <= 2^24. No label is checked here.
 */
CE_API int ce_stats(const float *logits, int64_t rows, int64_t vocab, int64_t stride, int64_t col0,
                    const int64_t *labels, float *stats, ce_stream_t stream);

/*
 * ce_stats_combine: merges `shards` slices' stats (stats: [shards][rows] x 4
 * f32, slices in column order, 16-byte aligned) into each whole row's
 *   loss_rows (f32, or NULL): crossEntropyRows of the whole row;
 *   top       (f32, or NULL): the whole row's argmax token;
 *   combined  ([rows] x 4 f32, 16-byte aligned, or NULL): (M, T, top, x[label])
 *             of the whole row, the input of ce_grad_from_stats.
 * A label outside [0, vocab_total) gives a NaN loss and increments the
 * device counter, as ce_rows does.
 */
CE_API int ce_stats_combine(const float *stats, int64_t shards, int64_t rows, int64_t vocab_total,
                            const int64_t *labels, float *loss_rows, float *top, float *combined,
                            ce_stream_t stream);

/*
 * ce_grad_from_stats: the slice [col0, col0 + vocab) of crossEntropyGrad,
 *     grad[i, j] = (exp(x_ij - M_i) * f32(1 / (1 + T_i)) - [col0 + j == label_i]) * scale,
 * from the combined (M, T) of ce_stats_combine; dense [rows, vocab]. A row
 * whose M is infinite or T is NaN gives a NaN gradient row. grad == logits is
 * allowed when stride == vocab; any other overlap is not.
 */
CE_API int ce_grad_from_stats(const float *logits, int64_t rows, int64_t vocab, int64_t stride, int64_t col0,
                              const int64_t *labels, const float *combined, double scale, float *grad,
                              ce_stream_t stream);

/* Human-readable text of a status code (a static string). */
CE_API const char *ce_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
CE_API int ce_version(void);

/* The cudaError_t code behind the calling thread's last CE_ECUDA. */
CE_API int ce_last_cuda_error(void);

/*
 * Device-side error counter of the current device, for tests and
 * diagnostics: *out = rows seen with a label outside [0, vocab) since the
 * last reset. This call WAITS for `stream` to finish.
 */
CE_API int ce_device_error_count(ce_stream_t stream, int64_t *out);

/*
 * The second device counter: waits on an asynchronous copy or a peer CTA
 * that gave up after their time limit (the output of such a call is then
 * undefined; the kernel still ran to its end). WAITS for `stream`.
 * ce_device_error_reset zeroes both counters (enqueued on `stream`).
 */
CE_API int ce_device_wait_timeouts(ce_stream_t stream, int64_t *out);
CE_API int ce_device_error_reset(ce_stream_t stream);

/*
 * Launch-plan override, for tests and tuning: forces the kernel family
 * (path: 0 automatic, 1 shared-memory-staged (persistent), 2 streaming from
 * global, 3 refused (formerly a ring-of-copies kernel), 4
 * shared-memory-staged with one row per cluster, 5 refused (the argmax split
 * evenly over the GPU is argmax_rows_noalloc's own plan), 6 one warp per row -- ce_rows, ce_loss,
 * argmax_rows and ce_stats only, 7 argmax through a ring of bulk-copied row
 * chunks -- argmax_rows and argmax_rows_indirect only), the CTAs that share
 * one row (cluster: 0 automatic, else 1..16; candidates_rows and path 7 take
 * at most 8) and the threads of a CTA (threads: 0 automatic, else 128 or
 * 256; 512 is rejected by every kernel family; candidates_rows and path 7
 * take 256 only).
 * Applies to every later call in the process. A forced plan that cannot
 * launch on this device makes the calls return CE_EINVAL.
 */
CE_API int ce_debug_force(int path, int cluster, int threads);

/*
 * Grid override, for tests: at most `clusters` clusters (0: no cap) in every
 * later launch of a row kernel (not argmax_rows_noalloc's), so that each
 * cluster loops over several rows even when the rows are few. Results are
 * the same; only the schedule changes. Returns CE_EINVAL for clusters < 0.
 */
CE_API int ce_debug_grid_cap(int64_t clusters);

/*
 * Read probe, for measurement: reads `bytes` bytes at device address p (16-byte
 * aligned, bytes a multiple of 16) once -- one CTA per SM, 32 KB chunks by
 * bulk asynchronous copies through four shared-memory stages, the fastest
 * plain read of a large buffer measured on this device -- and XORs every word
 * read into *out (4 bytes on the device, not cleared first). No page defines
 * it: it gives the ceiling of a plain read of a buffer of that size on this
 * device, to time beside a row kernel that reads the same bytes.
 */
CE_API int ce_debug_read(const void *p, int64_t bytes, uint32_t *out, ce_stream_t stream);

/*
 * The plan the library would pick (host only, launches nothing) for
 * op (0 ce_rows, 1 ce_grad, 2 argmax_rows, 3 softmax_rows, 4
 * log_softmax_rows, 5 candidates_rows) on the current device:
 * out[0] path, out[1] cluster, out[2] threads, out[3] dynamic shared bytes
 * per CTA, out[4] columns per CTA, out[5] CTAs in the grid.
 */
CE_API int ce_plan(int op, int64_t rows, int64_t vocab, int64_t stride, int64_t out[6]);

#ifdef __cplusplus
}
#endif

#endif /* CE_ROWS_H */
