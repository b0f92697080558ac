// ce_kernels.cu -- sm_103a kernels of the row-wise softmax cross-entropy
// path and of the rows a language model's step reads beside it, and their
// launchers.
//
// What they compute is defined on the API reference page "gizml:netops"
// (gizstack.com/docs/reference/gizml/netops.md), section Functions:
//   crossEntropyRows  each row's loss m + log(sum exp(x - m)) - x[label]
//   crossEntropyLoss  the mean of the row losses in f64
//   crossEntropyGrad  (softmax - onehot) * scale, softmax = exp(x - m) * f32(1/sum)
//   argmaxInto        each row's token (first of equals, NaN never wins) as f32
//   candidatesInto    each row's sampling candidates (TOP_EACH per thread of 256)
//   splitSumInto      the join of split partial sums
// and section Methods: Tensor.argmax (the tie and NaN rules).
//
// Kernel families (every one HBM-bound by design; none uses tensor cores):
//   k_rows_stream   one read of each logit: the online (m, t, idx) state of
//                   each thread's columns, merged over the CTA and then over
//                   the CTAs of a thread-block cluster that share one row
//                   through distributed shared memory. Writes the row loss,
//                   the argmax token, or a vocab slice's statistics.
//   k_rows_warp     the same for many moderate rows, one warp per row.
//   k_grad_staged   fused loss + gradient (or softmax / log-softmax rows): the
//                   cluster's CTAs bulk-copy (TMA engine) their slices of a
//                   row into shared memory, compute the state from there,
//                   exchange it over DSMEM, then write from shared memory. HBM
//                   sees each logit read once and each output written once.
//   k_grad_stream   the same for rows too long to stage: two reads.
//   k_argmax_flat   argmax of few long rows split evenly over the GPU, with
//                   k_argmax_combine (forced, and the no-allocation call).
//   k_candidates    sampling candidates, one list per thread, the row's chunks
//                   bulk-copied into a shared-memory ring.
//   k_split_sum     split sums in one resident wave.
//   k_stats_combine / k_grad_from_stats  the vocab-sharded loss and gradient.
//   k_read_probe    a plain read of a buffer (measurement only).
//   k_mean          the mean of the row losses, an f64 fixed-shape tree over a
//                   cluster, launched as a programmatic dependent of the row
//                   kernel that wrote them.
//
// The row kernels loop over rows (row = cluster id, + number of clusters), so
// any row count fits one launch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <utility>

#include "ce_device.cuh"
#include "ce_internal.h"

namespace cerows {

// [0] rows seen with a label outside [0, vocab); [1] bounded waits that gave up.
__device__ unsigned long long g_status[2];

namespace {

constexpr int kUnroll = 4;      // 16-byte loads in flight per thread (streaming)
// the same for the argmax scan, whose state is two registers: eight in flight
// (256 x 151936, L2 flushed: 32.9 -> 30.6 us on one box, with a plain read of
// the same bytes at 28.7 us; clusters of 2: 36.9 -> 32.7 us)
constexpr int kArgmaxUnroll = 8;
// the same for a warp alone on its row (4096 x 32000, L2 flushed: argmax
// 90 -> 80 us, row losses 97 -> 90 us against 4; 12 for the losses needs 76
// registers and leaves rows unscheduled, 16 for the argmax gains nothing)
constexpr int kWarpUnroll = 8;

struct alignas(16) StagedHeader {
    PushXchg xg;  // row states pushed by the cluster's CTAs
    uint64_t bar;  // the slice's bulk copy
    RowState red[32];
    float bc[4];
};
static_assert(sizeof(StagedHeader) <= kStagedHeaderBytes, "staged header too large");

__device__ __forceinline__ bool label_valid(int64_t label, int vocab) { return label >= 0 && label < vocab; }

// Row `row`'s first column: logits + row * stride, or, when the rows are given
// by a table of addresses, that address -- null when the address is null or
// not 4-byte aligned, a row that is then never read.
__device__ __forceinline__ const float *row_start(const Args &a, int64_t row) {
    if (!a.row_at) return a.logits + row * a.stride;
    const uint64_t v = a.row_at[row];
    return (v == 0 || (v & 3)) ? nullptr : reinterpret_cast<const float *>(v);
}

// The row loss from the merged state: (m - x[label]) + log1p(t); NaN for a
// bad label, or a row whose max is +-inf (a +inf entry, or all -inf / NaN),
// or whose t is NaN (a NaN entry).
__device__ __forceinline__ float row_loss(const RowState &g, float xl, bool lab_ok) {
    if (!lab_ok || !isfinite(g.m) || isnan(g.t)) return __int_as_float(0x7fffffff);
    return (g.m - xl) + log1pf(g.t);
}

// A 16-byte vector of shared-memory grid index q holding columns
// c0 - off + 4q ... +3 of the row: the slice's columns, -inf elsewhere.
__device__ __forceinline__ float4 load_edge(const float *p, int off, int n, int q) {
    float v[4];
#pragma unroll
    for (int l = 0; l < 4; ++l) {
        const int i = 4 * q + l - off;  // column - c0
        v[l] = (i >= 0 && i < n) ? p[i] : -INFINITY;
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ float row_token(const RowState &g) {
    return static_cast<float>(g.idx == kNoIndex ? 0 : g.idx);
}

// The argmax state (max, first column) of columns [j0, j0 + n) read from
// global memory at p, without the exp-sum: per 16-byte vector one max4 and one
// compare, and selects keep the best value, its vector and the vector itself
// -- no branch, so a warp never serialises on a lane that found a new max.
// The first lane holding the best value is found once at the end; strict
// compares keep the first vector of equals, and NaN never wins (fmaxf drops
// it). A thread whose vectors hold nothing above -inf rescans them exactly
// (only rows of -inf and NaN get there).
//
// The thread takes the body vectors q0, q0 + S, q0 + 2S, ... (in increasing
// column order); `edge` is its index among the threads that read the at most
// three columns before the first 16-byte boundary and after the last (-1:
// none). One thread set reading [j0, j0 + n) alone: q0 = edge = tid, S = T.
template <int kU>
__device__ __forceinline__ RowState scan_argmax(const float *__restrict__ p, int j0, int n, int q0, int S, int edge) {
    RowState st = empty_state();
    const int off = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
    const int head = min(n, (4 - off) & 3);
    const int nvec = (n - head) >> 2;
    const int tail = n - head - 4 * nvec;
    const float4 *pv = reinterpret_cast<const float4 *>(p + head);
    const int jv = j0 + head;
    if (edge >= 0 && edge < head) push<false>(st, ld_stream_f1(p + edge), j0 + edge);
    float best = -INFINITY;
    int bk = -1;
    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
    int k = q0;
    for (; k + (kU - 1) * S < nvec; k += kU * S) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = ld_stream_f4(pv + k + u * S);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const float mv = max4(v[u]);
            const bool gt = mv > best;
            best = gt ? mv : best;
            bk = gt ? k + u * S : bk;
            bv = gt ? v[u] : bv;
        }
    }
    for (; k < nvec; k += S) {
        const float4 v = ld_stream_f4(pv + k);
        const float mv = max4(v);
        const bool gt = mv > best;
        best = gt ? mv : best;
        bk = gt ? k : bk;
        bv = gt ? v : bv;
    }
    if (bk >= 0) {
        const int l = bv.x == best ? 0 : bv.y == best ? 1 : bv.z == best ? 2 : 3;
        push<false>(st, best, jv + 4 * bk + l);
    } else {
        for (k = q0; k < nvec; k += S) push4<false>(st, ld_stream_f4(pv + k), jv + 4 * k);
    }
    if (edge >= 0 && edge < tail) push<false>(st, ld_stream_f1(p + head + 4 * nvec + edge), jv + 4 * nvec + edge);
    return st;
}

// Push the columns [j0, j0 + n) of one row, read from global memory at p
// (p -> column j0): a scalar head up to the first 16-byte boundary, 16-byte
// vectors, a scalar tail. Each thread sees its columns in increasing order.
template <bool kStats, int kU = kUnroll>
__device__ __forceinline__ RowState scan_global(const float *__restrict__ p, int j0, int n, int tid, int T) {
    if constexpr (!kStats) return scan_argmax<kU>(p, j0, n, tid, T, tid);
    RowState st = empty_state();
    const int off = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
    const int head = min(n, (4 - off) & 3);
    const int nvec = (n - head) >> 2;
    const int tail = n - head - 4 * nvec;
    const float4 *pv = reinterpret_cast<const float4 *>(p + head);
    const int jv = j0 + head;
    if (tid < head) push<kStats>(st, ld_stream_f1(p + tid), j0 + tid);
    int k = tid;
    for (; k + (kU - 1) * T < nvec; k += kU * T) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = ld_stream_f4(pv + k + u * T);
#pragma unroll
        for (int u = 0; u < kU; ++u) push_vec<kStats>(st, v[u], jv + 4 * (k + u * T));
    }
    for (; k < nvec; k += T) push_vec<kStats>(st, ld_stream_f4(pv + k), jv + 4 * k);
    if (tid < tail) push<kStats>(st, ld_stream_f1(p + head + 4 * nvec + tid), jv + 4 * nvec + tid);
    return st;
}

// the CTA's threads over one slice
template <bool kStats, int kU = kUnroll>
__device__ __forceinline__ RowState scan_global(const float *__restrict__ p, int j0, int n) {
    return scan_global<kStats, kU>(p, j0, n, static_cast<int>(threadIdx.x), static_cast<int>(blockDim.x));
}

// ---------------------------------------------------------------------------
// k_rows_stream: row loss (kStats) and/or argmax token; one read per logit.
// The C CTAs of a cluster split a row -- the loss in C contiguous slices of
// `cols` columns, the argmax by taking the row's blocks of T vectors in turn
// -- and their states meet by pushes.
template <bool kStats>
__global__ void __launch_bounds__(kStreamMaxThreads, 6) k_rows_stream(Args a, int cols) {
    __shared__ RowState red[32];
    __shared__ PushXchg xg;
    launch_dependents();  // a mean of the row losses may be scheduled now; it waits for this grid's end
    const uint32_t rank = cluster_rank(), C = cluster_size();
    const int tid = threadIdx.x;
    const int c0 = static_cast<int>(rank) * cols;
    const int n = max(0, min(a.vocab, c0 + cols) - c0);
    const int64_t cid = cluster_id_x(), G = cluster_count_x();
    const int64_t K = cid < a.rows ? (a.rows - 1 - cid) / G + 1 : 0;  // rows of this cluster
    if (tid == 0) push_xchg_init(xg, K, C);
    __syncthreads();
    // every CTA's slot barriers exist before a peer pushes to them: the wait
    // that matches this arrive comes just before the first push, so the
    // barrier's latency hides under the first row's scan
    cluster_arrive();
    bool failed = false;
    int64_t k = 0;
    for (int64_t row = cid; row < a.rows; row += G, ++k) {
        // the label and x[label], fetched early by the thread that writes the loss
        const float *rp = row_start(a, row);  // the same for every CTA of the cluster
        int64_t label = 0;
        float xl = 0.0f;
        bool lab_ok = true;
        if (kStats && rank == 0 && tid == 0) {
            label = a.labels[row] - a.col0;  // col0: 0 but for a vocab slice
            lab_ok = label_valid(label, a.vocab);
            if (lab_ok && rp) xl = rp[label];
        }
        RowState st = empty_state();
        if constexpr (kStats) {
            if (n > 0 && rp) st = scan_global<true>(rp + c0, c0, n);
        } else if (rp) {
            // the cluster's CTAs take the row's 4 KB blocks of vectors in turn
            // (256 x 151936, L2 flushed: 30.3-30.6 -> 29.2 us against one
            // contiguous third each; the loss scan, one more register short,
            // spills with it and stays contiguous)
            const int T = static_cast<int>(blockDim.x);
            st = scan_argmax<kArgmaxUnroll>(rp, 0, a.vocab, static_cast<int>(rank) * T + tid, static_cast<int>(C) * T,
                                            rank == 0 ? tid : -1);
        }
        st = block_reduce_w0<kStats>(st, red);
        if (k == 0) cluster_wait();
        if (tid == 0) push_xchg_publish(xg, k, rank, C, st, 0.0f);
        if (tid < 32) {
            float unused;
            const RowState g = push_xchg_merge<kStats>(xg, k, K, C, 0u, &unused, &failed);
            if (rank == 0 && tid == 0) {
                if (kStats && a.stats) {
                    // a vocab slice's statistics; x[label] is 0 unless the slice holds the label
                    const float top = g.idx == kNoIndex ? -1.0f : static_cast<float>(a.col0 + g.idx);
                    reinterpret_cast<float4 *>(a.stats)[row] = make_float4(g.m, g.t, top, xl);
                } else if (kStats && a.loss) {
                    a.loss[row] = row_loss(g, xl, lab_ok);
                    if (!lab_ok) atomicAdd(&g_status[0], 1ull);
                }
                if (a.top) a.top[row] = rp ? row_token(g) : __int_as_float(0x7fffffff);
            }
        }
        __syncthreads();  // red is rewritten for the next row
    }
    if (K == 0) cluster_wait();  // the first arrive's match, for a cluster without rows
    cluster_arrive();  // no CTA leaves while a peer may still push to it
    cluster_wait();
    if (__syncthreads_or(failed) && tid == 0) atomicAdd(&g_status[1], 1ull);
}

// ---------------------------------------------------------------------------
// k_rows_warp: the outputs of k_rows_stream (row loss, token, or a vocab
// slice's statistics) for many short rows: one warp per row, looping over
// rows, the state merged by shuffles alone -- no CTA barrier, no exchange.
// Each warp keeps 2 KB of loads in flight; tens of warps per SM cover HBM's
// latency where a CTA per row would spend most of its time starting, merging
// and ending.
template <bool kStats>
__global__ void __launch_bounds__(256) k_rows_warp(Args a) {
    launch_dependents();  // a mean of the row losses may be scheduled now; it waits for this grid's end
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < a.rows;
         row += nwarps) {
        const float *rp = row_start(a, row);
        int64_t label = 0;
        float xl = 0.0f;
        bool lab_ok = true;
        if (kStats && lane == 0) {
            label = a.labels[row] - a.col0;  // col0: 0 but for a vocab slice
            lab_ok = label_valid(label, a.vocab);
            if (lab_ok && rp) xl = rp[label];
        }
        RowState g = rp ? scan_global<kStats, kWarpUnroll>(rp, 0, a.vocab, lane, 32) : empty_state();
        g = warp_reduce<kStats>(g);
        if (lane == 0) {
            if (kStats && a.stats) {
                const float top = g.idx == kNoIndex ? -1.0f : static_cast<float>(a.col0 + g.idx);
                reinterpret_cast<float4 *>(a.stats)[row] = make_float4(g.m, g.t, top, xl);
            } else if (kStats && a.loss) {
                a.loss[row] = row_loss(g, xl, lab_ok);
                if (!lab_ok) atomicAdd(&g_status[0], 1ull);
            }
            if (a.top) a.top[row] = rp ? row_token(g) : __int_as_float(0x7fffffff);
        }
    }
}

// ---------------------------------------------------------------------------
// k_grad_staged: fused loss + gradient (+ token) from shared-memory slices,
// persistent, each CTA's next slice copied in as soon as this one is written.
//
// CTA `rank` of a cluster owns columns [c0, c0 + n), c0 = rank * cols, of the
// cluster's rows (cluster cid of G takes rows cid, cid + G, ...). A row's
// slice sits in shared memory on the 16-byte grid of the logits: float i of
// buf holds column c0 - off + i, off = the slice's start modulo 16 bytes (in
// floats). Its aligned body arrives by one bulk copy (mbarrier bar, one phase
// per row); the at most two partial end vectors are loaded by the threads
// that own them, with -inf outside the slice. Thread t owns, in every pass,
// the vectors t + T*i. Per row:
//   sweep 1  each thread's max m over its vectors, and the first vector
//            holding it;
//   sweep 2  t = the sum of exp(x - m) but for the first element holding m
//            (x stays in shared memory: storing e back measured slower);
//   merge    over the CTA; then each CTA pushes its state into every CTA of
//            the cluster (st.async, completing bytes on their mbarrier) and
//            merges the C states in rank order, so every CTA holds the same
//            row state -- no cluster barrier per row;
//   write    grad = exp(x - M) * f32(1/(1 + T)) * scale (the label column
//            less scale); once the slice is written, the bulk copy of the
//            CTA's next row starts. The copy's latency hides behind the other
//            CTAs of the SM (four per SM): handing the slice over in two or
//            four ranges, each behind its own CTA barrier, measured slower
//            (16384 x 50257: 1.010 / 1.024 ms against 0.992 ms).
//
// The same kernel writes two other rows of the same statistics (kMode):
//   kModeSoftmax     out = exp(x - M) * f32(1/(1 + T)): no label, no scale;
//   kModeLogSoftmax  out = (x - M) - log1p(T).
template <int kMode>
__global__ void __launch_bounds__(kStagedMaxThreads, 3) k_grad_staged(Args a, int cols) {
    constexpr bool kCE = kMode == kModeGrad;
    constexpr bool kLog = kMode == kModeLogSoftmax;
    extern __shared__ __align__(128) unsigned char smem[];
    launch_dependents();  // a mean of the row losses may be scheduled now; it waits for this grid's end
    StagedHeader &h = *reinterpret_cast<StagedHeader *>(smem);
    float *buf = reinterpret_cast<float *>(smem + kStagedHeaderBytes);
    float4 *buf4 = reinterpret_cast<float4 *>(buf);
    const uint32_t rank = cluster_rank(), C = cluster_size();
    const int tid = threadIdx.x, T = blockDim.x;
    const int c0 = static_cast<int>(rank) * cols;
    const int n = max(0, min(a.vocab, c0 + cols) - c0);
    const float scale = a.scale;
    const int64_t G = cluster_count_x();

    // the bulk copy of the aligned body of `row`'s slice
    auto issue = [&](int64_t row, uint64_t policy) {
        const float *p = a.logits + row * a.stride + c0;
        const int off = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
        const int head = min(n, (4 - off) & 3);
        const int nvec = (n - head) >> 2;
        const int qa = (off + head) >> 2;
        const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
        mbar_arrive_expect_tx(&h.bar, bytes);
        if (bytes) bulk_copy_g2s(buf4 + qa, p - off + 4 * qa, bytes, &h.bar, policy);
    };

    const int64_t cid = cluster_id_x();
    const int64_t K = cid < a.rows ? (a.rows - 1 - cid) / G + 1 : 0;  // rows of this cluster
    uint64_t policy = 0;
    if (tid == 0) {
        mbar_init(&h.bar, 1);
        fence_mbar_init();
        push_xchg_init(h.xg, K, C);
        policy = l2_policy_evict_first();
        if (K > 0) issue(cid, policy);
    }
    __syncthreads();
    // every CTA's barriers exist before a peer pushes to them: the matching
    // wait comes just before the first push, under the first row's sweeps
    cluster_arrive();

    bool failed = false;
    uint32_t parity = 0;
    int64_t k = 0;  // this cluster's row count so far
    // each row's label is loaded one row ahead, off the row's critical path
    int64_t label_next = (kCE && K > 0) ? a.labels[cid] : 0;
    for (int64_t row = cid; row < a.rows; row += G, parity ^= 1u, ++k) {
        const float *p = a.logits + row * a.stride + c0;
        const int off = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
        const int head = min(n, (4 - off) & 3);
        const int nvec = (n - head) >> 2;       // whole body vectors
        const int qa = (off + head) >> 2;       // first body vector (0 or 1)
        const int nq = (off + n + 3) >> 2;      // vectors covering the slice
        const int jbase = c0 - off;             // column of float 0 of buf
        const bool more = row + G < a.rows;

        // the partial end vectors (at most two), loaded by their owners and
        // stored straight into the buffer: they lie outside the bulk copy's
        // bytes, and the previous row's reads of them ended at its last barrier
        const int qe0 = qa == 1 ? 0 : -1;
        const int qe1 = qa + nvec < nq ? qa + nvec : -1;
        auto owner = [&](int q) { return q & (T - 1); };  // T is a power of 2
        if (qe0 >= 0 && owner(qe0) == tid) buf4[qe0] = load_edge(p, off, n, qe0);
        if (qe1 >= 0 && owner(qe1) == tid) buf4[qe1] = load_edge(p, off, n, qe1);
        const int64_t label = label_next;
        if (kCE && more) label_next = a.labels[row + G];
        const bool lab_ok = !kCE || label_valid(label, a.vocab);
        const int lab_local = (kCE && lab_ok && label >= c0 && label < c0 + n) ? static_cast<int>(label - c0) : -1;
        const int lab_f = lab_local >= 0 ? off + lab_local : -1;  // float index of the label
        const int lab_q = lab_f >> 2;

        // sweep 1: max and its first vector
        float m = -INFINITY;
        int qm = -1;
        if (tid < nq && !failed) failed = !mbar_wait_bounded(&h.bar, parity);
        for (int q = tid; q < nq; q += T) {
            const float mv = max4(buf4[q]);
            if (mv > m) {
                m = mv;
                qm = q;
            }
        }
        // x[label]: read by the thread that owns its vector, before it
        // overwrites anything below (only that thread touches that vector)
        if (lab_q >= 0 && owner(lab_q) == tid) h.bc[2] = buf[lab_f];

        // sweep 2: t sums exp(x - m) over all but the first element holding
        // m (masked to -inf for the sweep, then restored)
        RowState st;
        if (m != -INFINITY) {
            const float4 vm = buf4[qm];
            const int lm = vm.x == m ? 0 : vm.y == m ? 1 : vm.z == m ? 2 : 3;
            buf[4 * qm + lm] = -INFINITY;
            float2 acc = make_float2(0.0f, 0.0f);
            for (int q = tid; q < nq; q += T) {
                const float4 e = exp4_sub(buf4[q], m);
                acc = __fadd2_rn(acc, __fadd2_rn(make_float2(e.x, e.y), make_float2(e.z, e.w)));
            }
            const float t = acc.x + acc.y;
            buf[4 * qm + lm] = m;
            st = RowState{m, t, jbase + 4 * qm + lm};
        } else {
            // no value above -inf among this thread's columns: the exact
            // update; e is 0 for -inf and NaN for NaN
            st = empty_state();
            for (int q = tid; q < nq; q += T) {
                for (int l = 0; l < 4; ++l) {
                    const int i = 4 * q + l;
                    const float x = buf[i];
                    if (i >= off && i - off < n) push<true>(st, x, jbase + i);
                }
            }
        }
        st = block_reduce_w0<true>(st, h.red);
        if (k == 0) cluster_wait();

        // exchange over the cluster: push this CTA's state into slot k % 2 of
        // every CTA (st.async, completing bytes on their slot barrier); warp 0
        // waits for the C states of its own slot and merges them in rank order
        if (tid == 0) push_xchg_publish(h.xg, k, rank, C, st, lab_local >= 0 ? h.bc[2] : 0.0f);
        if (tid < 32) {
            float xl;
            // a valid label is below 2^24: a 32-bit division
            const uint32_t own = lab_ok ? static_cast<uint32_t>(label) / static_cast<uint32_t>(cols) : 0u;
            const RowState g = push_xchg_merge<true>(h.xg, k, K, C, own, &xl, &failed);
            if (tid == 0) {
                const bool bad = !isfinite(g.m) || isnan(g.t);
                h.bc[0] = g.m;
                // f32(1/sum), or for log-softmax log(sum) = log1p(T)
                h.bc[1] = bad ? __int_as_float(0x7fffffff) : kLog ? log1pf(g.t) : 1.0f / (1.0f + g.t);
                if (kCE && rank == 0) {
                    if (a.loss) a.loss[row] = row_loss(g, xl, lab_ok);
                    if (!lab_ok) atomicAdd(&g_status[0], 1ull);
                    if (a.top) a.top[row] = row_token(g);
                }
            }
        }
        __syncthreads();

        // the output
        const float M = h.bc[0], rcp = h.bc[1];
        const float cm = rcp * scale;
        float *gp = a.grad + row * static_cast<int64_t>(a.vocab) + c0;  // column c0
        const bool vec_store = ((reinterpret_cast<uintptr_t>(gp) >> 2) & 3) == static_cast<uintptr_t>(off);
        for (int q = tid; q < nq; q += T) {
            const float4 g = kLog ? sub2_4(buf4[q], M, rcp) : mul4(exp4_sub(buf4[q], M), cm);
            if (vec_store && static_cast<unsigned>(q - qa) < static_cast<unsigned>(nvec)) {
                __stcs(reinterpret_cast<float4 *>(gp - off) + q, g);
            } else {
                const int i = 4 * q - off;  // column - c0 of lane 0
                if (i >= 0 && i < n) __stcs(gp + i, g.x);
                if (i + 1 >= 0 && i + 1 < n) __stcs(gp + i + 1, g.y);
                if (i + 2 >= 0 && i + 2 < n) __stcs(gp + i + 2, g.z);
                if (i + 3 >= 0 && i + 3 < n) __stcs(gp + i + 3, g.w);
            }
        }
        // the label column: its owner stored e * c there above; this later
        // store by the same thread replaces it
        if (lab_q >= 0 && owner(lab_q) == tid) __stcs(gp + lab_local, (exp_le0(buf[lab_f] - M) * rcp - 1.0f) * scale);
        // the slice, the edge vectors and bc are free: the next row's copy
        // starts, and they are rewritten for the next row
        __syncthreads();
        if (more && tid == 0) {
            fence_proxy_async_smem();
            issue(row + G, policy);
        }
    }
    if (K == 0) cluster_wait();  // the first arrive's match, for a cluster without rows
    cluster_arrive();  // no CTA leaves while a peer may still push to it
    cluster_wait();
    if (__syncthreads_or(failed) && tid == 0) {
        atomicAdd(&g_status[1], 1ull);
        // give a copy still in flight a last bounded chance to land
        (void)mbar_wait_bounded(&h.bar, parity ^ 1u, 10000000ull);
    }
}

// ---------------------------------------------------------------------------
// k_grad_stream: fused loss + gradient for rows too long to stage; the
// cluster's CTAs read their slices twice (state, then gradient) and meet by
// pushes.
template <int kMode>
__global__ void __launch_bounds__(kStreamMaxThreads, 6) k_grad_stream(Args a, int cols) {
    constexpr bool kCE = kMode == kModeGrad;
    constexpr bool kLog = kMode == kModeLogSoftmax;
    launch_dependents();  // a mean of the row losses may be scheduled now; it waits for this grid's end
    __shared__ RowState red[32];
    __shared__ PushXchg xg;
    __shared__ float bc[2];
    const uint32_t rank = cluster_rank(), C = cluster_size();
    const int tid = threadIdx.x, T = blockDim.x;
    const int c0 = static_cast<int>(rank) * cols;
    const int n = max(0, min(a.vocab, c0 + cols) - c0);
    const float scale = a.scale;
    const int64_t cid = cluster_id_x(), G = cluster_count_x();
    const int64_t K = cid < a.rows ? (a.rows - 1 - cid) / G + 1 : 0;  // rows of this cluster
    if (tid == 0) push_xchg_init(xg, K, C);
    __syncthreads();
    cluster_arrive();  // slot barriers exist before a peer pushes: the wait comes before the first push
    bool failed = false;
    int64_t k = 0;
    for (int64_t row = cid; row < a.rows; row += G, ++k) {
        const float *p = a.logits + row * a.stride + c0;
        const int64_t label = kCE ? a.labels[row] : 0;
        const bool lab_ok = !kCE || label_valid(label, a.vocab);
        const int lab_local = (kCE && lab_ok && label >= c0 && label < c0 + n) ? static_cast<int>(label - c0) : -1;
        // x[label] is read before any CTA of the cluster writes (grad may alias logits)
        const float xl_own = (tid == 0 && lab_local >= 0) ? p[lab_local] : 0.0f;
        RowState st = empty_state();
        if (n > 0) st = scan_global<true>(p, c0, n);
        st = block_reduce_w0<true>(st, red);
        if (k == 0) cluster_wait();
        if (tid == 0) push_xchg_publish(xg, k, rank, C, st, xl_own);
        if (tid < 32) {
            float xl;
            const uint32_t owner = lab_ok ? static_cast<uint32_t>(label / cols) : 0u;
            const RowState g = push_xchg_merge<true>(xg, k, K, C, owner, &xl, &failed);
            if (tid == 0) {
                const bool bad = !isfinite(g.m) || isnan(g.t);
                bc[0] = g.m;
                bc[1] = bad ? __int_as_float(0x7fffffff) : kLog ? log1pf(g.t) : 1.0f / (1.0f + g.t);
                if (kCE && rank == 0) {
                    if (a.loss) a.loss[row] = row_loss(g, xl, lab_ok);
                    if (!lab_ok) atomicAdd(&g_status[0], 1ull);
                    if (a.top) a.top[row] = row_token(g);
                }
            }
        }
        __syncthreads();
        const float M = bc[0], rcp = bc[1];
        float *gp = a.grad + row * static_cast<int64_t>(a.vocab) + c0;
        // coherent loads: with grad == logits this thread writes what it read
        for (int kk = tid; kk < n; kk += T) {
            const float x = __ldcs(p + kk);
            if (kLog) {
                __stcs(gp + kk, (x - M) - rcp);
            } else {
                const float pr = exp_le0(x - M) * rcp;
                __stcs(gp + kk, (kk == lab_local ? pr - 1.0f : pr) * scale);
            }
        }
        __syncthreads();  // bc and red are rewritten for the next row
    }
    if (K == 0) cluster_wait();  // the first arrive's match, for a cluster without rows
    cluster_arrive();  // no CTA leaves while a peer may still push to it
    cluster_wait();
    if (__syncthreads_or(failed) && tid == 0) atomicAdd(&g_status[1], 1ull);
}

// ---------------------------------------------------------------------------
// Argmax of few long rows, split evenly over one wave of CTAs.
//
// k_argmax_flat: CTA j of P scans elements [e_j, e_{j+1}), e_j = floor(j E / P),
// of the rows read as one sequence of E = rows * vocab elements (the first
// vocab columns of each row). For each row r its range meets, it writes the
// segment's key into ws[j + r] -- segments are ordered by position, so before
// (j, r) come exactly j range starts and r row starts: the index is unique.
// A key orders (value, then lower column first): the value's bits made
// monotone above, the column's complement below; a segment without a
// non-NaN value keys as value 0 (below -inf), column first.
// k_argmax_combine: each row's token is the largest key among the CTAs that
// met the row.
constexpr int kFlatThreads = 512;
constexpr int kFlatUnroll = 8;

__device__ __forceinline__ uint64_t argmax_key(const RowState &st, int first_col) {
    if (st.idx == kNoIndex) return 0xFFFFFFFFull - static_cast<uint32_t>(first_col);
    const uint32_t u = __float_as_uint(st.m + 0.0f);  // -0 -> +0
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<uint64_t>(ord) << 32) | (0xFFFFFFFFull - static_cast<uint32_t>(st.idx));
}

__device__ __forceinline__ int64_t flat_split(int64_t E, int64_t P, int64_t j) { return (E * j) / P; }

__global__ void __launch_bounds__(kFlatThreads, 2) k_argmax_flat(Args a, uint64_t *__restrict__ ws) {
    __shared__ RowState red[32];
    launch_dependents();  // the combine may be scheduled now; it waits for this grid's end
    const int64_t E = a.rows * static_cast<int64_t>(a.vocab), P = gridDim.x, j = blockIdx.x;
    const int64_t e0 = flat_split(E, P, j), e1 = flat_split(E, P, j + 1);
    for (int64_t r = e0 / a.vocab; r < a.rows && r * a.vocab < e1; ++r) {
        const int64_t ra = max(e0, r * a.vocab), rb = min(e1, (r + 1) * a.vocab);
        const int ca = static_cast<int>(ra - r * a.vocab);
        RowState st = scan_global<false, kFlatUnroll>(a.logits + r * a.stride + ca, ca, static_cast<int>(rb - ra));
        st = block_reduce_w0<false>(st, red);
        if (threadIdx.x == 0) ws[j + r] = argmax_key(st, ca);
        __syncthreads();  // red is rewritten for the next segment
    }
}

__global__ void k_argmax_combine(Args a, const uint64_t *__restrict__ ws, int P) {
    wait_prerequisites();  // every segment's key is written and visible
    const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (r >= a.rows) return;
    const int64_t E = a.rows * static_cast<int64_t>(a.vocab);
    // the CTA holding element x: the largest j with e_j <= x
    auto cta_of = [&](int64_t x) {
        int lo = 0, hi = P - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (flat_split(E, P, mid) <= x) lo = mid; else hi = mid - 1;
        }
        return lo;
    };
    const int jf = cta_of(r * a.vocab), jl = cta_of((r + 1) * a.vocab - 1);
    uint64_t key = 0;
    for (int jj = jf; jj <= jl; ++jj) key = max(key, ws[jj + r]);
    a.top[r] = static_cast<float>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
}

// ---------------------------------------------------------------------------
// Sampling candidates (candidatesInto; constants TOP_EACH and CANDIDATE_ROW).
//
// What is computed: a workgroup of 256 threads reads each row; thread t reads
// columns t, t + 256, t + 512, ... and keeps its 4 largest values, ranked by
// value and then by the lower column (NaN is never kept). Row i's output is
// 2048 floats at cand + 2048 i: pair 4t + k is thread t's rank-k (value,
// column as f32), (-inf, -1) where the thread read fewer than 4 values.
//
// How: see k_candidates below; the helpers here keep a thread's sorted list.
namespace cand {

constexpr int kEmptyCol = 0x7fffffff;  // a slot without a value ranks last

struct TopList {
    float v[kTopEach];
    int c[kTopEach];
};

__device__ __forceinline__ void top_init(TopList &L) {
#pragma unroll
    for (int k = 0; k < kTopEach; ++k) {
        L.v[k] = -INFINITY;
        L.c[k] = kEmptyCol;
    }
}

// (v1, c1) ranks above (v2, c2): a larger value, or an equal one at a lower
// column. Any comparison with a NaN value is false.
__device__ __forceinline__ bool ranks_above(float v1, int c1, float v2, int c2) {
    return v1 > v2 || (v1 == v2 && c1 < c2);
}

// Keep (x, col) if it ranks above the list's last slot; the list stays sorted.
__device__ __forceinline__ void top_push(TopList &L, float x, int col) {
    if (!ranks_above(x, col, L.v[3], L.c[3])) return;
    const bool a0 = ranks_above(L.v[0], L.c[0], x, col);
    const bool a1 = ranks_above(L.v[1], L.c[1], x, col);
    const bool a2 = ranks_above(L.v[2], L.c[2], x, col);
    const float v0 = L.v[0], v1 = L.v[1], v2 = L.v[2];
    const int c0 = L.c[0], c1 = L.c[1], c2 = L.c[2];
    L.v[3] = a2 ? x : v2;
    L.c[3] = a2 ? col : c2;
    L.v[2] = a2 ? v2 : (a1 ? x : v1);
    L.c[2] = a2 ? c2 : (a1 ? col : c1);
    L.v[1] = a1 ? v1 : (a0 ? x : v0);
    L.c[1] = a1 ? c1 : (a0 ? col : c0);
    L.v[0] = a0 ? v0 : x;
    L.c[0] = a0 ? c0 : col;
}

// The scan's insertion: x at column col, later than every column the list
// holds, so an equal value never displaces a kept one (four compares, then
// selects; the caller has seen x > the list's 4th value). Strict compares keep
// out NaN, and also -inf (it ties an empty slot's -inf): a list left with
// empty slots takes its -inf columns after the scan.
__device__ __forceinline__ void stream_push(TopList &L, float x, int col) {
    const bool p0 = x > L.v[0], p1 = x > L.v[1], p2 = x > L.v[2], p3 = x > L.v[3];
    const float v0 = L.v[0], v1 = L.v[1], v2 = L.v[2];
    const int c0 = L.c[0], c1 = L.c[1], c2 = L.c[2];
    L.v[3] = p2 ? v2 : (p3 ? x : L.v[3]);
    L.c[3] = p2 ? c2 : (p3 ? col : L.c[3]);
    L.v[2] = p1 ? v1 : (p2 ? x : v2);
    L.c[2] = p1 ? c1 : (p2 ? col : c2);
    L.v[1] = p0 ? v0 : (p1 ? x : v1);
    L.c[1] = p0 ? c0 : (p1 ? col : c1);
    L.v[0] = p0 ? x : v0;
    L.c[0] = p0 ? col : c0;
}

__device__ __forceinline__ float2 slot_of(const TopList &L, int k) {
    return make_float2(L.v[k], __int_as_float(L.c[k]));
}

__device__ __forceinline__ void push_slot(TopList &L, float2 e) { top_push(L, e.x, __float_as_int(e.y)); }

__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// Insert the values whose bits are set in `mask` (bit u: the value of the
// thread's column col0 + 256 u, read by val(u, col)), in column order: each is
// later in column order than every pair the list holds, as stream_push needs.
// The warp runs as many steps as its busiest lane has marks; a lane out of
// marks inserts -inf, which changes nothing (nor does a marked value that is
// no longer above the list's 4th). Each step reads the next marked value
// before it inserts the current one, so the read's latency overlaps the
// insertion.
template <typename Val>
__device__ __forceinline__ void insert_marked(TopList &L, uint32_t mask, int col0, Val val) {
    const int steps = static_cast<int>(__reduce_max_sync(kFullMask, static_cast<unsigned>(__popc(mask))));
    int u = __ffs(mask) - 1;  // -1 once the lane's marks are used
    mask &= mask - 1;
    float x = u >= 0 ? val(u, col0 + kCandThreads * u) : -INFINITY;
    for (int i = 0; i < steps; ++i) {
        const int col = col0 + kCandThreads * u;
        const int un = __ffs(mask) - 1;
        mask &= mask - 1;
        const float xn = un >= 0 ? val(un, col0 + kCandThreads * un) : -INFINITY;
        stream_push(L, x, col);
        u = un;
        x = xn;
    }
}

}  // namespace cand

// ChunkRing: a CTA's even share [jr0, jr1) of the blocks of 256 columns of
// each of its cluster's rows (cluster cid of G takes rows cid, cid + G, ...),
// streamed chunk by chunk: kBlocks blocks arrive by one bulk copy
// into a ring of kCandStages shared-memory stages (mbarrier full[s]), up to
// kCandStages chunks ahead, across rows. Each warp counts itself done with a
// stage (an acq_rel atomic on used[s]); the warp that finishes a chunk last
// issues the copy of the chunk kCandStages ahead into its stage. A chunk sits
// on the 16-byte grid of the logits (float i of a stage holds column
// cs - off + i), so any row phase is one aligned copy; the at most 3 columns
// of a row before its first 16-byte boundary and after its last are not
// copied (their threads read them from global memory).
struct RowGeom {
    int off, h, e;  // 16-byte phase (floats); columns [0, h) and [e, vocab) outside the copied grid
};

template <int kBlocks>
struct ChunkRing {
    static constexpr int kStageFloats = cand_stage_floats(kBlocks);
    const Args *a;
    int vocab;     // a->vocab and a->rows, held in registers: read every chunk
    int64_t rows;
    uint64_t *full;
    uint32_t *used;
    float *stages;
    int jr0, jr1, nk;  // blocks [jr0, jr1) of every row, in nk chunks
    int64_t cid, G;
    uint64_t policy;

    __device__ __forceinline__ ChunkRing(const Args &args, unsigned char *smem)
        : a(&args), vocab(args.vocab), rows(args.rows) {
        full = reinterpret_cast<uint64_t *>(smem);
        used = reinterpret_cast<uint32_t *>(full + kCandStages);
        stages = reinterpret_cast<float *>(smem + kCandHeaderBytes);
        const uint32_t rank = cluster_rank(), C = cluster_size();
        const int nb = (args.vocab + kCandThreads - 1) / kCandThreads;
        jr0 = static_cast<int>(static_cast<int64_t>(nb) * rank / C);
        jr1 = static_cast<int>(static_cast<int64_t>(nb) * (rank + 1) / C);
        nk = (jr1 - jr0 + kBlocks - 1) / kBlocks;
        cid = cluster_id_x();
        G = cluster_count_x();
        policy = l2_policy_evict_first();
    }
    __device__ __forceinline__ RowGeom geom(const float *p) const {
        const int off = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
        const int h = min(vocab, (4 - off) & 3);
        return RowGeom{off, h, h + ((vocab - h) & ~3)};
    }
    // the columns [cs, ce) of chunk k
    __device__ __forceinline__ int chunk_begin(int k) const { return kCandThreads * (jr0 + kBlocks * k); }
    __device__ __forceinline__ int chunk_end(int k) const {
        return min(vocab, kCandThreads * min(jr0 + kBlocks * (k + 1), jr1));
    }
    __device__ __forceinline__ float *stage(int s) const { return stages + s * kStageFloats; }
    // chunk k of `row` into stage s: the grid-aligned body of its columns
    __device__ __forceinline__ void issue(int64_t row, int k, int s) const {
        const float *p = row_start(*a, row);
        uint32_t bytes = 0;
        int dst = 0, c_lo = 0;
        if (p) {
            const RowGeom r = geom(p);
            const int cs = chunk_begin(k), ce = chunk_end(k);
            c_lo = max(cs - r.off, r.h);
            const int c_hi = min(cs - r.off + ((ce - cs + r.off + 3) & ~3), r.e);
            if (c_hi > c_lo) {
                bytes = 4u * static_cast<uint32_t>(c_hi - c_lo);
                dst = c_lo - (cs - r.off);
            }
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        if (bytes) bulk_copy_g2s(stage(s) + dst, p + c_lo, bytes, &full[s], policy);
    }
    // thread 0, once, before a __syncthreads: the barriers and the first chunks
    __device__ __forceinline__ void start() const {
        for (int s = 0; s < kCandStages; ++s) {
            mbar_init(&full[s], 1);
            used[s] = 0;
        }
        fence_mbar_init();
        int64_t row = cid;
        for (int k = 0, s = 0; s < kCandStages && row < rows && nk > 0; ++s) {
            issue(row, k, s);
            if (++k == nk) k = 0, row += G;
        }
    }
    // a warp is done with chunk k of `row` in stage s: the warp that finishes
    // it last refills the stage with the chunk kCandStages ahead
    __device__ __forceinline__ void release(int64_t row, int k, int s, int lane) const {
        constexpr uint32_t kWarps = kCandThreads / 32;
        int kn = k + kCandStages;
        int64_t rn = row;
        while (kn >= nk) kn -= nk, rn += G;
        __syncwarp();
        if (lane == 0 && rn < rows && atom_add_acq_rel_smem(&used[s], 1u) % kWarps == kWarps - 1)
            issue(rn, kn, s);
    }
    // after a wait gave up: a last bounded wait for the copies still in flight
    __device__ __forceinline__ void settle() const {
        const int64_t K = cid < rows ? (rows - 1 - cid) / G + 1 : 0;
        const int64_t total = K * nk;
        for (int64_t gl = total > kCandStages ? total - kCandStages : 0; gl < total; ++gl)
            (void)mbar_wait_bounded(&full[gl % kCandStages], static_cast<uint32_t>(gl / kCandStages) & 1u,
                                    10000000ull);
    }
};

// k_candidates: thread t of a 256-thread CTA is the pages' logical thread t
// itself and keeps one sorted list in registers, over the columns t + 256 j of
// its CTA's share of the row, streamed through a ChunkRing. Per chunk a thread
// marks, in a 15-bit mask, its values above the list's 4th value as of the
// chunk's start (never above the current one, so no value that belongs in the
// list is left out) and then inserts the marked ones: a warp runs the
// insertion once per value that some lane keeps, not once per value read.
// For C > 1, CTAs 1..C-1 leave their lists in shared memory and CTA 0 pulls
// and merges them through distributed shared memory and writes the row.
template <int kBlocks>
__global__ void __launch_bounds__(kCandThreads, 4) k_candidates(Args a, float *__restrict__ out) {
    using namespace cand;
    extern __shared__ __align__(128) unsigned char smem[];
    const ChunkRing<kBlocks> R(a, smem);
    float2 *lt = reinterpret_cast<float2 *>(smem + cand_ring_bytes(kBlocks)) + threadIdx.x;  // list slots (split rows)
    const int t = threadIdx.x, lane = t & 31;
    const uint32_t rank = cluster_rank(), C = cluster_size();
    const bool vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    constexpr int kChunkCols = kBlocks * kCandThreads;
    if (t == 0) R.start();
    __syncthreads();

    bool failed = false;
    int s = 0;        // stage of the next chunk
    uint32_t ph = 0;  // and the parity of its phase
    // Cluster barrier phases, per row: a wait before the list slots are
    // written (CTA 0 has pulled the previous row's lists), an arrive once they
    // are, a wait before the pull, an arrive after it.
    if (C > 1) cluster_arrive();
    for (int64_t row = R.cid; row < a.rows; row += R.G) {
        const float *p = row_start(a, row);  // null: a row without values
        const RowGeom r = p ? R.geom(p) : RowGeom{0, 0, 0};
        TopList L;
        top_init(L);
        for (int k = 0; k < R.nk; ++k) {
            if (!mbar_wait_bounded(&R.full[s], ph)) failed = true;
            if (p) {
                const int cs = R.chunk_begin(k), ce = R.chunk_end(k);
                const float *sv = R.stage(s) + r.off + t;  // sv[256 u]: column cs + t + 256 u
                auto fast = [&](int u, int) { return sv[kCandThreads * u]; };
                if (ce - cs == kChunkCols && cs >= r.h && ce <= r.e) {
                    if (k == 0) {
                        // the list starts empty: mark in groups of 8 blocks, each
                        // against the list's 4th value after the group before, so
                        // fewer of the chunk's values reach an insertion step
#pragma unroll
                        for (int u0 = 0; u0 < kBlocks; u0 += 8) {
                            const float thr = L.v[3];
                            uint32_t mask = 0;
#pragma unroll
                            for (int u = u0; u < u0 + 8 && u < kBlocks; ++u)
                                mask |= sv[kCandThreads * u] > thr ? 1u << u : 0u;
                            insert_marked(L, mask, cs + t, fast);
                        }
                    } else {
                        const float thr = L.v[3];
                        uint32_t mask = 0;
#pragma unroll
                        for (int u = 0; u < kBlocks; ++u) mask |= sv[kCandThreads * u] > thr ? 1u << u : 0u;
                        insert_marked(L, mask, cs + t, fast);
                    }
                } else {
                    // a chunk at the row's ends or cut short: its whole blocks
                    // inside the 16-byte grid body [h, e) are read from the
                    // stage as above; the at most two others column by column
                    // (columns past ce skipped, those outside the body read
                    // from global memory)
                    auto val = [&](int u, int col) {
                        return (col >= r.h && col < r.e) ? sv[kCandThreads * u] : ld_stream_f1(p + col);
                    };
                    const int u_lo = cs < r.h ? 1 : 0;                                 // block 0 of a misaligned row
                    const int u_hi = max(u_lo, (min(ce, r.e) - cs) / kCandThreads);    // whole blocks in [h, e)
                    const int u_end = (ce - cs + kCandThreads - 1) / kCandThreads;     // blocks with columns
                    const float thr = L.v[3];
                    uint32_t mask = 0;
#pragma unroll 8
                    for (int u = u_lo; u < u_hi; ++u) mask |= sv[kCandThreads * u] > thr ? 1u << u : 0u;
                    for (int u = 0; u < u_end; ++u) {
                        if (u >= u_lo && u < u_hi) continue;
                        const int col = cs + t + kCandThreads * u;
                        if (col < ce && val(u, col) > thr) mask |= 1u << u;
                    }
                    insert_marked(L, mask, cs + t, val);
                }
            }
            R.release(row, k, s, lane);
            if (++s == kCandStages) s = 0, ph ^= 1u;
        }
        // a list with an empty slot takes, in column order, its columns that
        // hold -inf (the scan kept every larger value already)
        if (p && L.c[3] == kEmptyCol) {
            int q = 0;
#pragma unroll
            for (int k = 0; k < kTopEach; ++k) q += L.c[k] != kEmptyCol;
            for (int jj = R.jr0; jj < R.jr1 && q < kTopEach; ++jj) {
                const int col = t + kCandThreads * jj;
                if (col >= a.vocab || p[col] != -INFINITY) continue;
#pragma unroll
                for (int k = 0; k < kTopEach; ++k)
                    if (k == q) L.c[k] = col;  // its value is already -inf
                ++q;
            }
        }
        if (C > 1) {
            cluster_wait();  // CTA 0 has pulled the previous row's lists
            if (rank != 0)
#pragma unroll
                for (int k = 0; k < kTopEach; ++k) lt[k * kCandThreads] = slot_of(L, k);
            cluster_arrive_release();
            cluster_wait();
            if (rank == 0)
                for (uint32_t q = 1; q < C; ++q) {
                    const uint32_t src = peer_smem(lt, q);
                    float2 e[kTopEach];
#pragma unroll
                    for (int k = 0; k < kTopEach; ++k)
                        e[k] = ld_dsmem_f2(src + 8u * static_cast<uint32_t>(k * kCandThreads));
#pragma unroll
                    for (int k = 0; k < kTopEach; ++k) push_slot(L, e[k]);
                }
            cluster_arrive_release();  // the peers' list slots may be rewritten once CTA 0 is past here
        }
        if (rank == 0) {
            float o[8];
#pragma unroll
            for (int k = 0; k < kTopEach; ++k) {
                const bool empty_slot = L.c[k] == kEmptyCol;
                o[2 * k] = empty_slot ? -INFINITY : L.v[k];
                o[2 * k + 1] = empty_slot ? -1.0f : static_cast<float>(L.c[k]);
            }
            float *dst = out + row * static_cast<int64_t>(kCandRow) + 8 * t;
            if (vec_out) {
                __stcs(reinterpret_cast<float4 *>(dst), make_float4(o[0], o[1], o[2], o[3]));
                __stcs(reinterpret_cast<float4 *>(dst) + 1, make_float4(o[4], o[5], o[6], o[7]));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) __stcs(dst + i, o[i]);
            }
        }
    }
    if (C > 1) cluster_wait();  // the last arrive's match: no CTA leaves while CTA 0 may still pull
    if (__syncthreads_or(failed) && t == 0) {
        atomicAdd(&g_status[1], 1ull);
        R.settle();
    }
}

// k_argmax_ring: argmaxInto through the same ChunkRing, for few long rows.
// Thread t keeps the first largest value of its columns t + 256 j (a strict
// compare from -inf, so NaN never wins; a thread left without a value above
// -inf takes its first -inf afterwards); for C > 1 CTA 0 pulls the peers'
// thread-t states over distributed shared memory, then reduces its 256
// states (larger value, then lower column) and writes the token, 0 for a row
// of NaN only.
template <int kBlocks>
__global__ void __launch_bounds__(kCandThreads, 4) k_argmax_ring(Args a) {
    using namespace cand;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 red[kCandThreads / 32];
    const ChunkRing<kBlocks> R(a, smem);
    float2 *lt = reinterpret_cast<float2 *>(smem + cand_ring_bytes(kBlocks)) + threadIdx.x;  // state slot (split rows)
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t rank = cluster_rank(), C = cluster_size();
    constexpr int kChunkCols = kBlocks * kCandThreads;
    if (t == 0) R.start();
    __syncthreads();

    bool failed = false;
    int s = 0;
    uint32_t ph = 0;
    if (C > 1) cluster_arrive();
    for (int64_t row = R.cid; row < a.rows; row += R.G) {
        const float *p = row_start(a, row);
        const RowGeom r = p ? R.geom(p) : RowGeom{0, 0, 0};
        float best = -INFINITY;
        int bcol = kNoIndex;
        for (int k = 0; k < R.nk; ++k) {
            if (!mbar_wait_bounded(&R.full[s], ph)) failed = true;
            if (p) {
                const int cs = R.chunk_begin(k), ce = R.chunk_end(k);
                const float *sv = R.stage(s) + r.off + t;
                if (ce - cs == kChunkCols && cs >= r.h && ce <= r.e) {
#pragma unroll
                    for (int u = 0; u < kBlocks; ++u) {
                        const float x = sv[kCandThreads * u];
                        const bool gt = x > best;
                        best = gt ? x : best;
                        bcol = gt ? cs + t + kCandThreads * u : bcol;
                    }
                } else {
#pragma unroll 4
                    for (int u = 0; u < kBlocks; ++u) {
                        const int col = cs + t + kCandThreads * u;
                        if (col < ce) {
                            const float x = (col >= r.h && col < r.e) ? sv[kCandThreads * u] : ld_stream_f1(p + col);
                            const bool gt = x > best;
                            best = gt ? x : best;
                            bcol = gt ? col : bcol;
                        }
                    }
                }
            }
            R.release(row, k, s, lane);
            if (++s == kCandStages) s = 0, ph ^= 1u;
        }
        // nothing above -inf among this thread's columns: its first -inf, if
        // any, is its first value that is not NaN (rows of -inf and NaN only)
        if (p && bcol == kNoIndex)
            for (int jj = R.jr0; jj < R.jr1; ++jj) {
                const int col = t + kCandThreads * jj;
                if (col < a.vocab && p[col] == -INFINITY) {
                    bcol = col;
                    break;
                }
            }
        if (C > 1) {
            cluster_wait();  // CTA 0 has pulled the previous row's states
            if (rank != 0) *lt = make_float2(best, __int_as_float(bcol));
            cluster_arrive_release();
            cluster_wait();
            if (rank == 0)
                for (uint32_t q = 1; q < C; ++q) {
                    const float2 e = ld_dsmem_f2(peer_smem(lt, q));
                    const int ec = __float_as_int(e.y);
                    if (ranks_above(e.x, ec, best, bcol)) best = e.x, bcol = ec;
                }
            cluster_arrive_release();
        }
        if (rank == 0) {
            // over the CTA: the larger value, then the lower column
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float ob = __shfl_xor_sync(kFullMask, best, d);
                const int oc = __shfl_xor_sync(kFullMask, bcol, d);
                if (ranks_above(ob, oc, best, bcol)) best = ob, bcol = oc;
            }
            if (lane == 0) red[warp] = make_float2(best, __int_as_float(bcol));
            __syncthreads();
            if (t == 0) {
                for (int w = 1; w < kCandThreads / 32; ++w) {
                    const int oc = __float_as_int(red[w].y);
                    if (ranks_above(red[w].x, oc, best, bcol)) best = red[w].x, bcol = oc;
                }
                if (a.top) a.top[row] = !p ? __int_as_float(0x7fffffff) : static_cast<float>(bcol != kNoIndex ? bcol : 0);
            }
            __syncthreads();  // red is rewritten for the next row
        }
    }
    if (C > 1) cluster_wait();
    if (__syncthreads_or(failed) && t == 0) {
        atomicAdd(&g_status[1], 1ull);
        R.settle();
    }
}

// ---------------------------------------------------------------------------
// Split sums (splitSumInto): y[i] = (add ? y[i] : 0) + parts[0][i] + ... +
// parts[splits - 1][i], part s at parts + s * total, added in f32 in split
// order. One resident wave of CTAs in a grid-stride loop over 16-byte
// vectors (kVec) or single floats; each thread sums two units per step, and
// keeps their loads of several parts in flight. Loads and stores are
// coherent: y may be parts[0] itself.
constexpr int kSplitUnroll = 4;

__device__ __forceinline__ void acc_add(float &a, float b) { a += b; }
__device__ __forceinline__ void acc_add(float4 &a, const float4 &b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

template <typename T>
__device__ __forceinline__ T zero_of() {
    return T{};
}
template <>
__device__ __forceinline__ float4 zero_of<float4>() {
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// y[i] and y[j] (j = i + blockDim, when j < n) from their `splits` parts
template <typename T>
__device__ __forceinline__ void split_pair(T *__restrict__ y, const T *p, int64_t n, int64_t splits, bool add,
                                           int64_t i, int64_t j) {
    const bool two = j < n;
    T a = add ? __ldcs(y + i) : zero_of<T>();
    T b = (add && two) ? __ldcs(y + j) : zero_of<T>();
    int64_t sp = 0;
    for (; sp + kSplitUnroll <= splits; sp += kSplitUnroll) {
        T va[kSplitUnroll], vb[kSplitUnroll];
#pragma unroll
        for (int k = 0; k < kSplitUnroll; ++k) {
            va[k] = __ldcs(p + (sp + k) * n + i);
            vb[k] = two ? __ldcs(p + (sp + k) * n + j) : zero_of<T>();
        }
#pragma unroll
        for (int k = 0; k < kSplitUnroll; ++k) {
            acc_add(a, va[k]);
            acc_add(b, vb[k]);
        }
    }
    // the last splits % 4 parts, all loads first
    const int rest = static_cast<int>(splits - sp);
    T va[kSplitUnroll - 1], vb[kSplitUnroll - 1];
#pragma unroll
    for (int k = 0; k < kSplitUnroll - 1; ++k) {
        va[k] = k < rest ? __ldcs(p + (sp + k) * n + i) : zero_of<T>();
        vb[k] = (k < rest && two) ? __ldcs(p + (sp + k) * n + j) : zero_of<T>();
    }
#pragma unroll
    for (int k = 0; k < kSplitUnroll - 1; ++k) {
        if (k < rest) {
            acc_add(a, va[k]);
            acc_add(b, vb[k]);
        }
    }
    __stcs(y + i, a);
    if (two) __stcs(y + j, b);
}

template <bool kVec>
__global__ void __launch_bounds__(kSplitThreads) k_split_sum(float *__restrict__ y, const float *parts, int64_t total,
                                                            int64_t splits, bool add) {
    // CTA b takes units [2 T b, 2 T b + 2 T) of each grid step: i and i + T
    const int64_t T = blockDim.x, step = 2 * T * gridDim.x;
    if (kVec) {
        const int64_t n = total / 4;
        for (int64_t i = 2 * T * blockIdx.x + threadIdx.x; i < n; i += step)
            split_pair(reinterpret_cast<float4 *>(y), reinterpret_cast<const float4 *>(parts), n, splits, add, i,
                       i + T);
    } else {
        for (int64_t i = 2 * T * blockIdx.x + threadIdx.x; i < total; i += step)
            split_pair(y, parts, total, splits, add, i, i + T);
    }
}

// ---------------------------------------------------------------------------
// Vocab-sharded rows. A row split over column slices (k_rows_stream writes
// each slice's float4 (m, t, top, x[label] or 0)) is put back together here:
// k_stats_combine merges the slices' states in slice order with the same
// symmetric merge the CTAs of a cluster use for one row, and writes the whole
// row's loss, token and combined state (M, T, top, x[label]); then
// k_grad_from_stats writes one slice's gradient from the combined (M, T).
__global__ void __launch_bounds__(256) k_stats_combine(const float4 *__restrict__ stats, int64_t shards,
                                                       int64_t rows, int64_t vocab_total,
                                                       const int64_t *__restrict__ labels, float *__restrict__ loss,
                                                       float *__restrict__ top, float4 *__restrict__ combined) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; row < rows; row += step) {
        RowState g = empty_state();
        float xl = 0.0f;
        for (int64_t sh = 0; sh < shards; ++sh) {
            const float4 v = stats[sh * rows + row];
            const RowState q{v.x, v.y, v.z < 0.0f ? kNoIndex : static_cast<int>(v.z)};
            g = sh == 0 ? q : merge<true>(g, q);
            xl += v.w;  // every slice but the label's adds an exact 0
        }
        const int64_t label = labels[row];
        const bool lab_ok = label >= 0 && label < vocab_total;
        if (loss) loss[row] = row_loss(g, xl, lab_ok);
        if (!lab_ok) atomicAdd(&g_status[0], 1ull);
        if (top) top[row] = row_token(g);
        if (combined)
            combined[row] = make_float4(g.m, g.t, g.idx == kNoIndex ? -1.0f : static_cast<float>(g.idx), xl);
    }
}

// One CTA per row (looping): grad[j] = (exp(x_j - M) * f32(1/(1 + T)) - [col0
// + j == label]) * scale over the slice, dense [rows, vocab]; NaN rows where
// the whole row is degenerate. 16-byte loads and stores when the row and its
// gradient row share their 16-byte phase (a scalar head, vectors, a scalar
// tail), single floats otherwise. Loads and stores are coherent (grad may be
// the slice itself when the slice is dense).
constexpr int kGradStatsUnroll = 4;

__global__ void __launch_bounds__(256) k_grad_from_stats(Args a, const float4 *__restrict__ combined) {
    const int T = blockDim.x, tid = threadIdx.x;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const float4 st = combined[row];
        const float M = st.x;
        const bool bad = !isfinite(M) || isnan(st.y);
        const float rcp = bad ? __int_as_float(0x7fffffff) : 1.0f / (1.0f + st.y);
        const float cm = rcp * a.scale;
        const int64_t local = a.labels[row] - a.col0;
        const int lab = (local >= 0 && local < a.vocab) ? static_cast<int>(local) : -1;
        const float *p = a.logits + row * a.stride;
        float *g = a.grad + row * static_cast<int64_t>(a.vocab);
        auto one = [&](int j, float x) {
            const float e = exp_le0(x - M);
            return j == lab ? (e * rcp - 1.0f) * a.scale : e * cm;
        };
        const int offp = static_cast<int>((reinterpret_cast<uintptr_t>(p) >> 2) & 3);
        const int offg = static_cast<int>((reinterpret_cast<uintptr_t>(g) >> 2) & 3);
        int head = a.vocab, nvec = 0;
        if (offp == offg) {
            head = min(a.vocab, (4 - offp) & 3);
            nvec = (a.vocab - head) >> 2;
        }
        // the scalar head (or the whole row when the phases differ)
        for (int j = tid; j < head; j += T) __stcs(g + j, one(j, __ldcs(p + j)));
        const float4 *pv = reinterpret_cast<const float4 *>(p + head);
        float4 *gv = reinterpret_cast<float4 *>(g + head);
        int q = tid;
        for (; q + (kGradStatsUnroll - 1) * T < nvec; q += kGradStatsUnroll * T) {
            float4 x[kGradStatsUnroll];
#pragma unroll
            for (int u = 0; u < kGradStatsUnroll; ++u) x[u] = __ldcs(pv + q + u * T);
#pragma unroll
            for (int u = 0; u < kGradStatsUnroll; ++u) {
                const int j = head + 4 * (q + u * T);
                __stcs(gv + q + u * T, make_float4(one(j, x[u].x), one(j + 1, x[u].y), one(j + 2, x[u].z),
                                                   one(j + 3, x[u].w)));
            }
        }
        for (; q < nvec; q += T) {
            const float4 x = __ldcs(pv + q);
            const int j = head + 4 * q;
            __stcs(gv + q, make_float4(one(j, x.x), one(j + 1, x.y), one(j + 2, x.z), one(j + 3, x.w)));
        }
        // the scalar tail
        for (int j = head + 4 * nvec + tid; j < a.vocab; j += T) __stcs(g + j, one(j, __ldcs(p + j)));
    }
}

// ---------------------------------------------------------------------------
// k_mean: one cluster of kMeanCtas CTAs, launched as a programmatic dependent
// of the row kernel before it on the stream (so it is already resident when
// that kernel ends). Thread g of the cluster's kMeanCtas * kMeanThreads sums
// rows g, g + kMeanCtas * kMeanThreads, ... in f64; a butterfly over each
// warp, then over the CTA's warps; the CTAs' sums meet in CTA 0's shared
// memory (distributed shared memory) and are added by a butterfly in rank
// order. The shape does not depend on the device: the same bits every run.
// 8 CTAs of 256 threads: GB300 adds f64 at about two lanes per clock per SM,
// so fewer butterfly lanes end sooner (4096 x 32000 ce_loss less ce_rows:
// 4.7 us at 512 threads, 4.1 at 256; 1024 threads x 4 CTAs: 7.7)
constexpr int kMeanCtas = 8;
constexpr int kMeanThreads = 256;

__global__ void __launch_bounds__(kMeanThreads) k_mean(const float *__restrict__ loss, int64_t rows,
                                                       double *__restrict__ out) {
    __shared__ double warp_sum[kMeanThreads / 32];
    __shared__ double cta_sum[kMeanCtas];
    cluster_arrive();      // every CTA has started before CTA 0's shared memory is written
    wait_prerequisites();  // the row losses are complete and visible
    const uint32_t rank = cluster_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int64_t kAll = static_cast<int64_t>(kMeanCtas) * kMeanThreads;
    double s = 0.0;
    for (int64_t i = static_cast<int64_t>(rank) * kMeanThreads + tid; i < rows; i += kAll)
        s += static_cast<double>(loss[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFullMask, s, o);
    if (lane == 0) warp_sum[warp] = s;
    __syncthreads();
    cluster_wait();
    if (warp == 0) {
        double r = lane < kMeanThreads / 32 ? warp_sum[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(kFullMask, r, o);
        if (lane == 0) st_dsmem_f64(peer_smem(&cta_sum[rank], 0), r);
    }
    cluster_arrive_release();
    cluster_wait();
    if (rank == 0 && warp == 0) {
        double r = lane < kMeanCtas ? cta_sum[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(kFullMask, r, o);
        if (lane == 0) *out = r / static_cast<double>(rows);
    }
}

// ---------------------------------------------------------------------------
// k_read_probe: a plain read of `bytes` bytes, the ceiling of a read of that
// size on this device, for measurement beside the row kernels. One CTA per SM
// streams chunks c = blockIdx.x, blockIdx.x + gridDim.x, ... of 32 KB through
// four shared-memory stages by bulk copies (the TMA engine); every thread
// folds its 16-byte vectors of each chunk by XOR into one word. Measured on
// GB300, 155.7 MB with L2 flushed: 27.6 us against 28.7-28.9 us for 16-byte
// loads, eight in flight per thread over one resident wave of 512-thread CTAs.
constexpr int kProbeThreads = 256;
constexpr int kProbeStages = 4;
constexpr int kProbeChunk = 32768;
constexpr int kProbeSmem = 128 + kProbeStages * kProbeChunk;

__global__ void __launch_bounds__(kProbeThreads, 1) k_read_probe(const char *__restrict__ p, int64_t bytes,
                                                                 uint32_t *__restrict__ out) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    const float4 *stage = reinterpret_cast<const float4 *>(smem + 128);
    const int tid = threadIdx.x;
    const int64_t nch = (bytes + kProbeChunk - 1) / kProbeChunk;
    const int64_t K = blockIdx.x < nch ? (nch - 1 - blockIdx.x) / gridDim.x + 1 : 0;  // chunks of this CTA
    const uint64_t policy = l2_policy_evict_first();
    auto chunk_bytes = [&](int64_t k) {
        const int64_t rest = bytes - (blockIdx.x + k * gridDim.x) * static_cast<int64_t>(kProbeChunk);
        return static_cast<uint32_t>(rest < kProbeChunk ? rest : kProbeChunk);
    };
    auto issue = [&](int64_t k) {
        const int s = static_cast<int>(k % kProbeStages);
        const uint32_t nb = chunk_bytes(k);
        mbar_arrive_expect_tx(&bar[s], nb);
        bulk_copy_g2s(smem + 128 + s * kProbeChunk, p + (blockIdx.x + k * gridDim.x) * static_cast<int64_t>(kProbeChunk),
                      nb, &bar[s], policy);
    };
    if (tid == 0) {
        for (int s = 0; s < kProbeStages; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int64_t k = 0; k < K && k < kProbeStages; ++k) issue(k);
    }
    __syncthreads();
    uint32_t acc = 0;
    bool failed = false;
    for (int64_t k = 0; k < K; ++k) {
        const int s = static_cast<int>(k % kProbeStages);
        if (!failed && !mbar_wait_bounded(&bar[s], static_cast<uint32_t>(k / kProbeStages) & 1u)) failed = true;
        const int nv = static_cast<int>(chunk_bytes(k) / 16);
        const float4 *sv = stage + s * (kProbeChunk / 16);
#pragma unroll 4
        for (int q = tid; q < nv; q += kProbeThreads) {
            const float4 v = sv[q];
            acc ^= __float_as_uint(v.x) ^ __float_as_uint(v.y) ^ __float_as_uint(v.z) ^ __float_as_uint(v.w);
        }
        __syncthreads();  // stage s is free
        if (tid == 0 && k + kProbeStages < K) {
            fence_proxy_async_smem();
            issue(k + kProbeStages);
        }
    }
    acc = __reduce_xor_sync(kFullMask, acc);
    if ((tid & 31) == 0) atomicXor(out, acc);
    if (__syncthreads_or(failed) && tid == 0) {
        atomicAdd(&g_status[1], 1ull);
        // a last bounded wait for the copies still in flight
        for (int64_t k = K > kProbeStages ? K - kProbeStages : 0; k < K; ++k)
            (void)mbar_wait_bounded(&bar[k % kProbeStages], static_cast<uint32_t>(k / kProbeStages) & 1u, 10000000ull);
    }
}

cudaError_t launch_clustered(const void *fn, const Plan &p, void **args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.clusters * p.cluster), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int kMode>
const void *fused_kernel(int path) {
    return path == kPathStaged ? reinterpret_cast<const void *>(&k_grad_staged<kMode>)
                               : reinterpret_cast<const void *>(&k_grad_stream<kMode>);
}

const void *kernel_of(const Plan &p, Op op) {
    if (op == kOpGrad) {
        return fused_kernel<kModeGrad>(p.path);
    }
    if (op == kOpSoftmax) return fused_kernel<kModeSoftmax>(p.path);
    if (op == kOpLogSoftmax) return fused_kernel<kModeLogSoftmax>(p.path);
    if (op == kOpCandidates)
        return p.chunk == kCandChunkLarge ? reinterpret_cast<const void *>(&k_candidates<kCandChunkLarge>)
                                          : reinterpret_cast<const void *>(&k_candidates<kCandChunkSmall>);
    if (p.path == kPathRing)
        return p.chunk == kCandChunkLarge ? reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkLarge>)
                                          : reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkSmall>);
    if (p.path == kPathWarp)
        return op == kOpRows ? reinterpret_cast<const void *>(&k_rows_warp<true>)
                             : reinterpret_cast<const void *>(&k_rows_warp<false>);
    if (op == kOpRows) return reinterpret_cast<const void *>(&k_rows_stream<true>);
    return reinterpret_cast<const void *>(&k_rows_stream<false>);
}

}  // namespace

cudaError_t set_kernel_attributes(const DeviceInfo &dev) {
    const void *fns[] = {reinterpret_cast<const void *>(&k_rows_stream<true>),
                         reinterpret_cast<const void *>(&k_rows_stream<false>),
                         reinterpret_cast<const void *>(&k_grad_staged<kModeGrad>),
                         reinterpret_cast<const void *>(&k_grad_staged<kModeSoftmax>),
                         reinterpret_cast<const void *>(&k_grad_staged<kModeLogSoftmax>),
                         reinterpret_cast<const void *>(&k_grad_stream<kModeGrad>),
                         reinterpret_cast<const void *>(&k_grad_stream<kModeSoftmax>),
                         reinterpret_cast<const void *>(&k_grad_stream<kModeLogSoftmax>),
                         reinterpret_cast<const void *>(&k_candidates<kCandChunkSmall>),
                         reinterpret_cast<const void *>(&k_candidates<kCandChunkLarge>),
                         reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkSmall>),
                         reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkLarge>)};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const void *staged[] = {reinterpret_cast<const void *>(&k_grad_staged<kModeGrad>),
                            reinterpret_cast<const void *>(&k_grad_staged<kModeSoftmax>),
                            reinterpret_cast<const void *>(&k_grad_staged<kModeLogSoftmax>)};
    for (const void *f : staged) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.max_smem_optin);
        if (e != cudaSuccess) return e;
    }
    const std::pair<const void *, int> rings[] = {
        {reinterpret_cast<const void *>(&k_candidates<kCandChunkSmall>), cand_max_smem_bytes(kCandChunkSmall)},
        {reinterpret_cast<const void *>(&k_candidates<kCandChunkLarge>), cand_max_smem_bytes(kCandChunkLarge)},
        {reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkSmall>), cand_max_smem_bytes(kCandChunkSmall)},
        {reinterpret_cast<const void *>(&k_argmax_ring<kCandChunkLarge>), cand_max_smem_bytes(kCandChunkLarge)}};
    for (const auto &r : rings) {
        cudaError_t e = cudaFuncSetAttribute(r.first, cudaFuncAttributeMaxDynamicSharedMemorySize, r.second);
        if (e != cudaSuccess) return e;
    }
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(&k_read_probe), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kProbeSmem);
}

cudaError_t max_active_clusters(const Plan &p, Op op, int *n) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.cluster), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, kernel_of(p, op), &cfg);
}

cudaError_t launch_rows_stream(const Plan &p, const Args &a, bool stats, cudaStream_t s) {
    if (p.path == kPathRing) {
        if (stats) return cudaErrorInvalidValue;  // the ring serves the argmax only
        Args aa = a;
        void *args[] = {&aa};
        return launch_clustered(kernel_of(p, kOpArgmax), p, args, s);
    }
    if (p.path == kPathWarp) {
        if (stats)
            k_rows_warp<true><<<static_cast<unsigned>(p.clusters), p.threads, 0, s>>>(a);
        else
            k_rows_warp<false><<<static_cast<unsigned>(p.clusters), p.threads, 0, s>>>(a);
        return cudaGetLastError();
    }
    Args aa = a;
    int cols = p.cols;
    void *args[] = {&aa, &cols};
    return launch_clustered(kernel_of(p, stats ? kOpRows : kOpArgmax), p, args, s);
}

cudaError_t launch_fused(const Plan &p, Op op, const Args &a, cudaStream_t s) {
    Args aa = a;
    int cols = p.cols;
    void *args[] = {&aa, &cols};
    return launch_clustered(kernel_of(p, op), p, args, s);
}

cudaError_t launch_candidates(const Plan &p, const Args &a, float *cand, cudaStream_t s) {
    Args aa = a;
    float *cc = cand;
    void *args[] = {&aa, &cc};
    return launch_clustered(kernel_of(p, kOpCandidates), p, args, s);
}

cudaError_t launch_split_sum(float *y, const float *parts, int64_t total, int64_t splits, bool add, int sms,
                             cudaStream_t s) {
    const bool vec = total % 4 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(parts) & 15) == 0;
    const void *fn = vec ? reinterpret_cast<const void *>(&k_split_sum<true>)
                         : reinterpret_cast<const void *>(&k_split_sum<false>);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kSplitThreads, 0);
    if (e != cudaSuccess) return e;
    // one resident wave, and no more CTAs than there are pairs of units
    const int64_t units = vec ? total / 4 : total;
    const int64_t pair_ctas = (units + 2 * kSplitThreads - 1) / (2 * kSplitThreads);
    const int ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(pair_ctas, int64_t(per_sm) * sms)));
    if (vec)
        k_split_sum<true><<<ctas, kSplitThreads, 0, s>>>(y, parts, total, splits, add);
    else
        k_split_sum<false><<<ctas, kSplitThreads, 0, s>>>(y, parts, total, splits, add);
    return cudaGetLastError();
}

cudaError_t launch_argmax_flat(const Args &a, int ctas, void *ws, cudaStream_t s) {
    k_argmax_flat<<<ctas, kFlatThreads, 0, s>>>(a, static_cast<uint64_t *>(ws));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int threads = 256;
    const unsigned blocks = static_cast<unsigned>((a.rows + threads - 1) / threads);
    // a programmatic dependent of the scan: no launch gap between the two
    // (64 x 151936, L2 flushed: 23.6 -> 21.0 us; 1024 rows 104 -> 101 us)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_argmax_combine, a, static_cast<const uint64_t *>(ws), ctas);
}

cudaError_t launch_stats_combine(const float *stats, int64_t shards, int64_t rows, int64_t vocab_total,
                                 const int64_t *labels, float *loss, float *top, float *combined, int sms,
                                 cudaStream_t s) {
    const int64_t blocks = std::min<int64_t>((rows + 255) / 256, 8 * int64_t(sms));
    k_stats_combine<<<static_cast<unsigned>(std::max<int64_t>(1, blocks)), 256, 0, s>>>(
        reinterpret_cast<const float4 *>(stats), shards, rows, vocab_total, labels, loss, top,
        reinterpret_cast<float4 *>(combined));
    return cudaGetLastError();
}

cudaError_t launch_grad_from_stats(const Args &a, const float *combined, int sms, cudaStream_t s) {
    (void)sms;
    const int64_t blocks = std::min<int64_t>(a.rows, int64_t(1) << 20);
    k_grad_from_stats<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a, reinterpret_cast<const float4 *>(combined));
    return cudaGetLastError();
}

cudaError_t launch_mean(const float *loss, int64_t rows, double *out, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMeanCtas, 1, 1);
    cfg.blockDim = dim3(kMeanThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMeanCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_mean, loss, rows, out);
}

cudaError_t launch_read_probe(const void *p, int64_t bytes, uint32_t *out, int sms, cudaStream_t s) {
    const int64_t nch = (bytes + kProbeChunk - 1) / kProbeChunk;
    const int ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(nch, sms)));
    k_read_probe<<<ctas, kProbeThreads, kProbeSmem, s>>>(static_cast<const char *>(p), bytes, out);
    return cudaGetLastError();
}

cudaError_t read_status(unsigned long long out[2], cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(unsigned long long) * 2, 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
}

cudaError_t reset_status(cudaStream_t s) {
    static const unsigned long long zero[2] = {0ull, 0ull};
    return cudaMemcpyToSymbolAsync(g_status, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
}

}  // namespace cerows
