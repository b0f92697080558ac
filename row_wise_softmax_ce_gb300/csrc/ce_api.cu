// ce_api.cu -- the C ABI declared in include/ce_rows.h: host-side argument
// checks, the choice of kernel and launch shape, and status codes.
//
// Conventions follow the pages this library implements: the operations of
// "gizml:netops" (crossEntropyRows, crossEntropyLoss, crossEntropyGrad,
// argmaxInto, candidatesInto, splitSumInto) run where the data is and do not wait for the GPU; and, as the
// "gpukit" API page's device-op wrappers do, every entry point checks its
// buffers and sizes first and fails closed -- a wrong size never reaches
// the device.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "ce_internal.h"
#include "ce_rows.h"

using namespace cerows;

namespace {

constexpr int kVersion = 10000;            // 1.0.0
constexpr int64_t kMaxVocab = 1ll << 24;   // tokens are written exactly as f32
constexpr int kMaxDevices = 64;
constexpr int kStagedTargetCols = 16384;   // 64 KB of f32 per CTA: 3 CTAs per SM
constexpr int kStagedTargetCols4 = 13816;  // the widest slice of which 4 CTAs fit an SM's 228 KB
                                           // (2 KB header, 16-byte grid, 1 KB reserved per CTA)
constexpr int kStreamMinCols = 2048;       // columns per CTA, at least, when a row is split
constexpr int64_t kMaxClusters = 1ll << 20;

thread_local int t_last_cuda_error = 0;

// Scratch of argmax_rows_noalloc: one 64-bit key per (CTA, row) segment of the
// even split, 8192 keys = 64 KiB, resident on every device that loads this
// library until the process exits. Host code never names it directly: its
// device address comes from cudaGetSymbolAddress (noalloc_scratch below).
constexpr int64_t kNoAllocKeys = 8192;
static __device__ __align__(256) uint64_t g_noalloc_keys[kNoAllocKeys];
uint64_t *g_noalloc_ptr[kMaxDevices] = {};

struct Force {
    int path = 0, cluster = 0, threads = 0;
    int64_t grid_cap = 0;  // at most this many clusters (0: no cap)
};
Force g_force;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_ready[kMaxDevices] = {};

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return CE_OK;
    t_last_cuda_error = static_cast<int>(e);
    return CE_ECUDA;
}

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int round_up4(int64_t v) { return static_cast<int>((v + 3) & ~int64_t(3)); }

// The current device, its properties, and the kernels' attributes (set once).
int current_device(DeviceInfo *out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return CE_EDEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return CE_EDEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[dev]) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(e);
            return CE_EDEVICE;
        }
        if (d.cc_major != 10 || d.cc_minor != 3) return CE_EDEVICE;  // built for sm_103a only
        if ((e = set_kernel_attributes(d)) != cudaSuccess) return cuda_status(e);
        g_dev[dev] = d;
        g_ready[dev] = true;
    }
    *out = g_dev[dev];
    return CE_OK;
}

// Launch shape of a streaming kernel (ce_rows, argmax_rows, and the fused
// path for rows too long to stage): split a row over C CTAs when there are
// too few rows to give every SM several CTAs.
void plan_stream(Plan &p, int64_t rows, int64_t vocab, const DeviceInfo &dev, int threads, int cluster) {
    p.path = kPathStream;
    p.threads = threads ? threads : kStreamMaxThreads;
    if (cluster) {
        p.cluster = cluster;
    } else {
        // split rows until about four and a half CTAs per SM; none from three
        // rows per SM up. Measured on GB300, rows x 151936, L2 flushed (us, by
        // CTAs per row 1 / 2 / 3 / 4 / 5 / 6). Argmax (branch-free scan, eight
        // loads in flight): 256 rows 37.3 / 31.5 / 30.8 / 37.0 / 34.7 / 31.2;
        // 128 rows 33.1 / 23.2 / 20.9 / 22.4 / 20.8 / 18.9; 512 rows 53.9 /
        // 59.9 / 53.2 / 59.9 / 57.3 / 56.1. Row losses: 256 rows 45.2 / 37.0 /
        // 35.2 / 41.1 / 37.3 / 36.9; 128 rows 41.1 / 28.7 / 24.6 / - / 24.1 /
        // 22.5; 512 rows 59.1 / 69.2 / 59.3 / - / 61.9 / -; 64 rows 16.7 at 5,
        // 15.9 at 8 and 11; 200 rows 30.8 at 2, 28.4 at 4.
        int64_t c = rows >= 3 * static_cast<int64_t>(dev.sms) ? 1 : ceil_div(9 * static_cast<int64_t>(dev.sms), 2 * rows);
        c = std::min<int64_t>(c, std::min<int64_t>(kMaxCluster, ceil_div(vocab, kStreamMinCols)));
        p.cluster = static_cast<int>(std::max<int64_t>(1, c));
    }
    p.cols = round_up4(ceil_div(vocab, p.cluster));
    p.smem = 0;
    p.clusters = std::min<int64_t>(rows, kMaxClusters);
}

// Launch shape of the warp-per-row kernel: 256-thread CTAs (8 rows at a
// time each), as many as are resident at once and no more than the rows need.
bool plan_warp(Plan &p, Op op, int64_t rows) {
    p.path = kPathWarp;
    p.threads = 256;
    p.cluster = 1;
    p.smem = 0;
    p.cols = 0;
    p.clusters = 1;
    int active = 0;
    if (max_active_clusters(p, op, &active) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (active < 1) return false;
    p.clusters = std::max<int64_t>(1, std::min<int64_t>(ceil_div(rows, 8), active));
    return true;
}

// Launch shape of the staged fused kernel: the fewest CTAs per row whose
// slices are at most kStagedTargetCols columns (at most 16 CTAs).
// The staged kernel's geometry for `c` CTAs per row: columns per CTA and the
// shared memory that covers any row misalignment ((cols + 9) / 4 vectors);
// false when it does not fit. *active: the clusters resident at once.
bool staged_shape(Plan &p, Op op, int64_t vocab, const DeviceInfo &dev, int64_t c, int *active) {
    if (c > kMaxCluster) c = kMaxCluster;
    p.cluster = static_cast<int>(c);
    p.cols = round_up4(ceil_div(vocab, c));
    p.smem = kStagedHeaderBytes + 16 * ((p.cols + 9) / 4);
    if (p.smem > dev.max_smem_optin) return false;
    *active = 0;
    if (max_active_clusters(p, op, active) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return *active >= 1;
}

bool plan_staged(Plan &p, Op op, int64_t rows, int64_t vocab, const DeviceInfo &dev, int threads, int cluster,
                 bool per_row, bool auto_form) {
    p.path = kPathStaged;
    p.threads = threads ? threads : 256;
    // the kernel maps vectors to threads modulo T: 128 or 256
    if (p.threads > kStagedMaxThreads || (p.threads & (p.threads - 1)) != 0) return false;
    int active = 0;
    const int64_t c = cluster ? cluster : std::max<int64_t>(1, ceil_div(vocab, kStagedTargetCols));
    if (!staged_shape(p, op, vocab, dev, c, &active)) return false;
    // persistent (every cluster resident at once, looping over rows), or one
    // row per cluster with the hardware scheduling clusters as others finish.
    // Measured on GB300: persistent is ahead when each cluster loops over
    // many rows (8192 x 128256: 160 rows per cluster, 93% vs 89% of copy
    // bandwidth), one row per cluster when it would loop over few (4096 x
    // 32000: 18 rows per cluster, 93% vs 89%).
    if (auto_form) per_row = rows < 32 * static_cast<int64_t>(active);
    if (auto_form && !cluster && !threads) {
        // slices small enough for four CTAs per SM. Persistent: they pay when
        // they put more CTAs on the GPU at once. Measured on GB300, 8192 x
        // 128256 (8 CTAs of 66 KB per row, 408 resident: 94.8% of copy
        // bandwidth; 10 of 53 KB, 580 resident: 98.9%; 9, 11: 87.8%, 96.3%).
        // One row per cluster: they pay on rows of three slices or more (L2
        // flushed, softmax rows x 151936, 10 CTAs per row (3 per SM) vs 12 vs
        // 11 (4 per SM): 128 rows 33.0 / 31.2 / - us, 256 rows 57.3 / 54.8 /
        // 53.4 us, 1024 rows 203.6 / 190.7 / 185.0 us; the gradient of 256
        // rows 59.1 / 55.8 / 55.2 us; 13 per row: 57.9 us), not on two (4096 x
        // 32000, 2 vs 3: softmax 155.9 vs 158.3 us, gradient 156.6 vs 154.3 us).
        Plan q = p;
        int active4 = 0;
        const int64_t c4 = std::max<int64_t>(1, ceil_div(vocab, kStagedTargetCols4));
        if (c4 != c && staged_shape(q, op, vocab, dev, c4, &active4)) {
            const bool take = per_row ? c >= 3
                                      : rows >= 32 * static_cast<int64_t>(active4) &&
                                            static_cast<int64_t>(active4) * q.cluster >
                                                static_cast<int64_t>(active) * p.cluster;
            if (take) {
                p = q;
                active = active4;
            }
        }
    }
    p.clusters = per_row ? std::min<int64_t>(rows, kMaxClusters) : std::min<int64_t>(rows, active);
    return true;
}

// Launch shape of the candidates kernel: 256 threads (the pages' workgroup);
// a row split over C = 2 x SMs / rows CTAs (about two per SM), 1 <= C <= 8,
// each with at least 2048 columns. Measured on GB300, rows x 151936, L2
// flushed (us, C = 1 / 2 / 3 / 4 / 8): 256 rows 40.6 / 41.0 / 46.5 / 47.1 /
// 67.6; 128 rows 32.8 / 28.2 / 28.9 / 30.9 / 39.2; 64 rows 33.2 / 22.5 / 24.6
// / 22.5 / 26.6; 32 rows 32.7 / 22.8 / 20.0 / 18.8 / 18.4.
void plan_candidates(Plan &p, int64_t rows, int64_t vocab, const DeviceInfo &dev, int cluster) {
    p.path = kPathStream;
    p.threads = kCandThreads;
    int64_t c = cluster;
    if (!c) {
        const int64_t target = 2 * static_cast<int64_t>(dev.sms);
        c = std::max<int64_t>(1, std::min<int64_t>(kCandMaxCluster, target / std::max<int64_t>(1, rows)));
        c = std::min<int64_t>(c, std::min<int64_t>(kCandMaxCluster, ceil_div(vocab, kStreamMinCols)));
    }
    p.cluster = static_cast<int>(std::max<int64_t>(1, c));
    p.cols = round_up4(ceil_div(vocab, p.cluster));
    // chunks of 32 blocks where the grid has at most two CTAs per SM (their
    // ring allows two per SM), else of 15 (four per SM). Measured on GB300, L2
    // flushed (us, 15 / 30 / 36 blocks): 256 x 151936 39.1 / 33.2 / 32.7;
    // 4096 x 32000 114 / 125 / 127; 16384 x 50257 588 / 711 / 702.
    p.chunk = rows * static_cast<int64_t>(p.cluster) <= 2 * static_cast<int64_t>(dev.sms) ? kCandChunkLarge
                                                                                          : kCandChunkSmall;
    p.smem = cand_ring_bytes(p.chunk) + (p.cluster > 1 ? kCandListBytes : 0);
    p.clusters = std::min<int64_t>(rows, kMaxClusters);
}

// Where the ring argmax beats the streaming one (both measured on GB300,
// where one warp per row does not apply): from four rows per SM up -- 1024 x
// 151936 (L2 flushed) 93.7 vs 105.0 us, 16384 x 50257 447 vs 462 us, 8192 x
// 128256 568 vs 571 us; 256 x 151936 31.4 vs 30.7 us and 64 rows 14.8 vs 14.6
// us stay with the streaming kernel.
bool ring_argmax_applies(int64_t rows, const DeviceInfo &dev) { return rows >= 4 * static_cast<int64_t>(dev.sms); }

// Launch shape of the ring argmax: the candidates kernel's chunk ring, one
// (value, column) state per thread; the row split like the candidates'.
void plan_argmax_ring(Plan &p, int64_t rows, int64_t vocab, const DeviceInfo &dev, int cluster) {
    plan_candidates(p, rows, vocab, dev, cluster);
    p.path = kPathRing;
    p.smem = cand_ring_bytes(p.chunk) + (p.cluster > 1 ? kRingArgmaxSlotBytes : 0);
}

// Where one warp per row beats a CTA (or cluster) per row, measured on GB300
// with L2 flushed: ce_rows 4096 x 32000 81% vs 66% of copy bandwidth, 16384 x
// 50257 97% vs 83%, slices of 16032 columns x 8192 rows 2.24 vs 2.49 ms for
// eight; argmax 4096 x 32000 96% vs 90%, but 16384 x 50257 97% vs 105%. Long
// rows (128256) and few rows stay with the CTA per row.
bool warp_applies(Op op, int64_t rows, int64_t vocab, const DeviceInfo &dev) {
    if (rows < 8 * static_cast<int64_t>(dev.sms)) return false;
    if (op == kOpRows) return vocab <= 65536;
    if (op == kOpArgmax) return vocab <= 32768;
    return false;
}

int make_plan(Op op, int64_t rows, int64_t vocab, const DeviceInfo &dev, Plan *out) {
    Force f;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        f = g_force;
    }
    Plan p;
    if (op == kOpGrad || op == kOpSoftmax || op == kOpLogSoftmax) {
        if (f.path == kPathRetired3) {
            return CE_EINVAL;
        } else if (f.path == kPathStaged || f.path == kPathStagedPerRow) {
            if (!plan_staged(p, op, rows, vocab, dev, f.threads, f.cluster, f.path == kPathStagedPerRow, false))
                return CE_EINVAL;
        } else if (f.path == kPathStream) {
            plan_stream(p, rows, vocab, dev, f.threads, f.cluster);
        } else if (f.path == kPathFlat || f.path == kPathWarp || f.path == kPathRing) {
            return CE_EINVAL;
        } else if (!plan_staged(p, op, rows, vocab, dev, f.threads, f.cluster, false, true)) {
            plan_stream(p, rows, vocab, dev, f.threads, f.cluster ? f.cluster : kMaxCluster);
        }
    } else if (op == kOpCandidates) {
        if (f.path != kPathAuto && f.path != kPathStream) return CE_EINVAL;
        if (f.threads && f.threads != kCandThreads) return CE_EINVAL;
        if (f.cluster > kCandMaxCluster) return CE_EINVAL;
        plan_candidates(p, rows, vocab, dev, f.cluster);
    } else if (f.path == kPathRing) {
        if (op != kOpArgmax || (f.threads && f.threads != kCandThreads) || f.cluster > kCandMaxCluster)
            return CE_EINVAL;
        plan_argmax_ring(p, rows, vocab, dev, f.cluster);
    } else if (f.path == kPathFlat) {
        // the even split needs scratch for its per-segment keys: only
        // argmax_rows_noalloc, which owns a fixed array, runs it
        return CE_EINVAL;
    } else if (f.path == kPathWarp) {
        if ((f.threads && f.threads != 256) || f.cluster > 1 || !plan_warp(p, op, rows)) return CE_EINVAL;
    } else if (f.path == kPathAuto && f.cluster == 0 && f.threads == 0 && warp_applies(op, rows, vocab, dev) &&
               plan_warp(p, op, rows)) {
        // many rows of moderate width: one warp per row
    } else if (op == kOpArgmax && f.path == kPathAuto && f.cluster == 0 && f.threads == 0 &&
               ring_argmax_applies(rows, dev)) {
        plan_argmax_ring(p, rows, vocab, dev, 0);
    } else {
        plan_stream(p, rows, vocab, dev, f.threads, f.cluster);
    }
    if (p.cluster < 1 || p.cluster > kMaxCluster) return CE_EINVAL;
    if (p.path == kPathStream && p.threads > kStreamMaxThreads) return CE_EINVAL;
    // every row kernel loops over rows with a stride of the cluster count, so
    // a smaller grid only gives each cluster more rows
    if (f.grid_cap > 0) p.clusters = std::min(p.clusters, f.grid_cap);
    *out = p;
    return CE_OK;
}

// ce_grad_host's copy stream and events, one set per device, created on
// first use and kept for the life of the process (like the error counter).
constexpr int kHostChunksMax = 64;
struct HostPipe {
    std::mutex mu;  // held while a call enqueues, so calls do not interleave their events
    bool ready = false;
    cudaStream_t copy = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t chunk[kHostChunksMax] = {};
};
HostPipe g_pipe[kMaxDevices];

// caller holds h.mu
cudaError_t host_pipe_ready(HostPipe &h) {
    if (h.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming);
    for (int i = 0; i < kHostChunksMax && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(&h.chunk[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (int i = 0; i < kHostChunksMax; ++i)
            if (h.chunk[i]) (void)cudaEventDestroy(h.chunk[i]), h.chunk[i] = nullptr;
        if (h.start) (void)cudaEventDestroy(h.start), h.start = nullptr;
        if (h.copy) (void)cudaStreamDestroy(h.copy), h.copy = nullptr;
        return e;
    }
    h.ready = true;
    return cudaSuccess;
}

int check_logits(const float *logits, int64_t rows, int64_t vocab, int64_t stride) {
    if (rows < 0 || vocab < 1 || vocab > kMaxVocab || stride < vocab) return CE_EINVAL;
    if (rows > 0 && logits == nullptr) return CE_EINVAL;
    if (rows > 0 && stride > (INT64_MAX / 4) / rows) return CE_EINVAL;  // byte offsets fit int64
    if (misaligned(logits, 4)) return CE_EALIGN;
    return CE_OK;
}

bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

Args make_args(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels) {
    Args a = {};
    a.logits = logits;
    a.rows = rows;
    a.vocab = static_cast<int>(vocab);
    a.stride = stride;
    a.labels = labels;
    return a;
}

// The checks and the fused launch behind ce_grad and ce_grad_step.
int grad_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels,
              double scale, float *grad, float *loss_rows, float *top, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (!std::isfinite(scale)) return CE_EINVAL;
    if (rows > 0 && (labels == nullptr || grad == nullptr)) return CE_EINVAL;
    if (misaligned(labels, 8) || misaligned(grad, 4) || misaligned(loss_rows, 4) || misaligned(top, 4))
        return CE_EALIGN;
    if (rows == 0) return CE_OK;
    const int64_t in_bytes = ((rows - 1) * stride + vocab) * 4;
    const int64_t out_bytes = rows * vocab * 4;
    if (grad == logits) {
        if (stride != vocab) return CE_EINVAL;  // in place needs the same layout
    } else if (ranges_overlap(grad, out_bytes, logits, in_bytes)) {
        return CE_EINVAL;
    }
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpGrad, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, labels);
    a.scale = static_cast<float>(scale);
    a.grad = grad;
    a.loss = loss_rows;
    a.top = top;
    return cuda_status(launch_fused(p, kOpGrad, a, stream));
}

}  // namespace

extern "C" {

int ce_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels,
            float *loss_rows, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (rows > 0 && (labels == nullptr || loss_rows == nullptr)) return CE_EINVAL;
    if (misaligned(labels, 8) || misaligned(loss_rows, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpRows, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, labels);
    a.loss = loss_rows;
    return cuda_status(launch_rows_stream(p, a, true, stream));
}

int ce_mean(const float *loss_rows, int64_t rows, double *loss_mean, ce_stream_t stream) {
    if (rows < 0 || loss_mean == nullptr || (rows > 0 && loss_rows == nullptr)) return CE_EINVAL;
    if (misaligned(loss_rows, 4) || misaligned(loss_mean, 8)) return CE_EALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    return cuda_status(launch_mean(loss_rows, rows, loss_mean, stream));
}

int ce_loss(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels,
            float *loss_rows, double *loss_mean, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (loss_mean == nullptr || (rows > 0 && (labels == nullptr || loss_rows == nullptr))) return CE_EINVAL;
    if (misaligned(labels, 8) || misaligned(loss_rows, 4) || misaligned(loss_mean, 8)) return CE_EALIGN;
    if ((st = ce_rows(logits, rows, vocab, stride, labels, loss_rows, stream))) return st;
    return ce_mean(loss_rows, rows, loss_mean, stream);
}

int ce_grad(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels,
            double scale, float *grad, float *loss_rows, ce_stream_t stream) {
    return grad_rows(logits, rows, vocab, stride, labels, scale, grad, loss_rows, nullptr, stream);
}

int ce_grad_step(const float *logits, int64_t rows, int64_t vocab, int64_t stride, const int64_t *labels,
                 double scale, float *grad, float *loss_rows, float *top, double *loss_mean, ce_stream_t stream) {
    // the mean reads the row losses: asking for it needs somewhere to put them
    if (loss_mean != nullptr && rows > 0 && loss_rows == nullptr) return CE_EINVAL;
    if (misaligned(loss_mean, 8)) return CE_EALIGN;
    int st = grad_rows(logits, rows, vocab, stride, labels, scale, grad, loss_rows, top, stream);
    if (st || loss_mean == nullptr) return st;
    return ce_mean(loss_rows, rows, loss_mean, stream);
}

// softmax_rows and log_softmax_rows: the fused kernels without labels.
int normalised_rows(Op op, const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *out,
                    ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (rows > 0 && out == nullptr) return CE_EINVAL;
    if (misaligned(out, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    const int64_t in_bytes = ((rows - 1) * stride + vocab) * 4;
    const int64_t out_bytes = rows * vocab * 4;
    if (out == logits) {
        if (stride != vocab) return CE_EINVAL;  // in place needs the same layout
    } else if (ranges_overlap(out, out_bytes, logits, in_bytes)) {
        return CE_EINVAL;
    }
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(op, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, nullptr);
    a.scale = 1.0f;
    a.grad = out;
    return cuda_status(launch_fused(p, op, a, stream));
}

int softmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *out, ce_stream_t stream) {
    return normalised_rows(kOpSoftmax, logits, rows, vocab, stride, out, stream);
}

int log_softmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *out,
                     ce_stream_t stream) {
    return normalised_rows(kOpLogSoftmax, logits, rows, vocab, stride, out, stream);
}

int candidates_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *cand,
                    ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (rows > 0 && cand == nullptr) return CE_EINVAL;
    if (misaligned(cand, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    if (ranges_overlap(cand, rows * int64_t(kCandRow) * 4, logits, ((rows - 1) * stride + vocab) * 4))
        return CE_EINVAL;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpCandidates, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, nullptr);
    return cuda_status(launch_candidates(p, a, cand, stream));
}

int split_sum(float *y, const float *parts, int64_t total, int64_t splits, int add, ce_stream_t stream) {
    if (total < 0 || splits < 1) return CE_EINVAL;
    if (total > 0 && (y == nullptr || parts == nullptr)) return CE_EINVAL;
    if (total > 0 && splits > (INT64_MAX / 4) / total) return CE_EINVAL;  // byte offsets fit int64
    if (misaligned(y, 4) || misaligned(parts, 4)) return CE_EALIGN;
    if (total == 0) return CE_OK;
    // y may be part 0 itself (each element is read before it is written, by
    // the same thread); any other overlap is rejected
    if (y != parts && ranges_overlap(y, total * 4, parts, splits * total * 4)) return CE_EINVAL;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    return cuda_status(launch_split_sum(y, parts, total, splits, add != 0, dev.sms, stream));
}

// argmax_rows_indirect / candidates_rows_indirect: the rows at the addresses
// of a device table (argmaxInto's indirect form); same kernels and plans as
// the direct calls, less the even split (which walks rows by their stride).
int check_row_table(const uint64_t *row_addrs, int64_t rows, int64_t vocab) {
    if (rows < 0 || vocab < 1 || vocab > kMaxVocab) return CE_EINVAL;
    if (rows > 0 && row_addrs == nullptr) return CE_EINVAL;
    if (misaligned(row_addrs, 8)) return CE_EALIGN;
    return CE_OK;
}

int argmax_rows_indirect(const uint64_t *row_addrs, int64_t rows, int64_t vocab, float *top, ce_stream_t stream) {
    int st = check_row_table(row_addrs, rows, vocab);
    if (st) return st;
    if (rows > 0 && top == nullptr) return CE_EINVAL;
    if (misaligned(top, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpArgmax, rows, vocab, dev, &p))) return st;
    Args a = make_args(nullptr, rows, vocab, vocab, nullptr);
    a.row_at = row_addrs;
    a.top = top;
    return cuda_status(launch_rows_stream(p, a, false, stream));
}

int candidates_rows_indirect(const uint64_t *row_addrs, int64_t rows, int64_t vocab, float *cand,
                             ce_stream_t stream) {
    int st = check_row_table(row_addrs, rows, vocab);
    if (st) return st;
    if (rows > 0 && cand == nullptr) return CE_EINVAL;
    if (misaligned(cand, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpCandidates, rows, vocab, dev, &p))) return st;
    Args a = make_args(nullptr, rows, vocab, vocab, nullptr);
    a.row_at = row_addrs;
    return cuda_status(launch_candidates(p, a, cand, stream));
}

int ce_stats(const float *logits, int64_t rows, int64_t vocab, int64_t stride, int64_t col0, const int64_t *labels,
             float *stats, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (col0 < 0 || col0 + vocab > kMaxVocab) return CE_EINVAL;  // global columns exact in f32
    if (rows > 0 && (labels == nullptr || stats == nullptr)) return CE_EINVAL;
    if (misaligned(labels, 8) || misaligned(stats, 16)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    if (ranges_overlap(stats, rows * 16, logits, ((rows - 1) * stride + vocab) * 4)) return CE_EINVAL;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpRows, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, labels);
    a.stats = stats;
    a.col0 = col0;
    return cuda_status(launch_rows_stream(p, a, true, stream));
}

int ce_stats_combine(const float *stats, int64_t shards, int64_t rows, int64_t vocab_total, const int64_t *labels,
                     float *loss_rows, float *top, float *combined, ce_stream_t stream) {
    if (shards < 1 || rows < 0 || vocab_total < 1 || vocab_total > kMaxVocab) return CE_EINVAL;
    if (rows > 0 && (stats == nullptr || labels == nullptr)) return CE_EINVAL;
    if (rows > 0 && shards > (INT64_MAX / 16) / rows) return CE_EINVAL;
    if (misaligned(stats, 16) || misaligned(labels, 8) || misaligned(loss_rows, 4) || misaligned(top, 4) ||
        misaligned(combined, 16))
        return CE_EALIGN;
    if (rows == 0) return CE_OK;
    if (combined && ranges_overlap(combined, rows * 16, stats, shards * rows * 16)) return CE_EINVAL;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    return cuda_status(
        launch_stats_combine(stats, shards, rows, vocab_total, labels, loss_rows, top, combined, dev.sms, stream));
}

int ce_grad_from_stats(const float *logits, int64_t rows, int64_t vocab, int64_t stride, int64_t col0,
                       const int64_t *labels, const float *combined, double scale, float *grad, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (col0 < 0 || col0 + vocab > kMaxVocab || !std::isfinite(scale)) return CE_EINVAL;
    if (rows > 0 && (labels == nullptr || combined == nullptr || grad == nullptr)) return CE_EINVAL;
    if (misaligned(labels, 8) || misaligned(combined, 16) || misaligned(grad, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    const int64_t in_bytes = ((rows - 1) * stride + vocab) * 4;
    const int64_t out_bytes = rows * vocab * 4;
    if (grad == logits) {
        if (stride != vocab) return CE_EINVAL;  // in place needs the same layout
    } else if (ranges_overlap(grad, out_bytes, logits, in_bytes)) {
        return CE_EINVAL;
    }
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Args a = make_args(logits, rows, vocab, stride, labels);
    a.scale = static_cast<float>(scale);
    a.grad = grad;
    a.col0 = col0;
    return cuda_status(launch_grad_from_stats(a, combined, dev.sms, stream));
}

int argmax_rows(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *top, ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (rows > 0 && top == nullptr) return CE_EINVAL;
    if (misaligned(top, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    Plan p;
    if ((st = make_plan(kOpArgmax, rows, vocab, dev, &p))) return st;
    Args a = make_args(logits, rows, vocab, stride, nullptr);
    a.top = top;
    return cuda_status(launch_rows_stream(p, a, false, stream));
}

// The device address of g_noalloc_keys on the current device, looked up once
// per device (with that device current) and cached.
int noalloc_scratch(const DeviceInfo &dev, uint64_t **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_noalloc_ptr[dev.device] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_keys);
        if (e != cudaSuccess || ptr == nullptr) {
            t_last_cuda_error = static_cast<int>(e);
            return CE_ECUDA;
        }
        g_noalloc_ptr[dev.device] = static_cast<uint64_t *>(ptr);
    }
    *out = g_noalloc_ptr[dev.device];
    return CE_OK;
}

int argmax_rows_noalloc(const float *logits, int64_t rows, int64_t vocab, int64_t stride, float *top,
                        ce_stream_t stream) {
    int st = check_logits(logits, rows, vocab, stride);
    if (st) return st;
    if (rows > 0 && top == nullptr) return CE_EINVAL;
    if (misaligned(top, 4)) return CE_EALIGN;
    if (rows == 0) return CE_OK;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    // the even split over at most two CTAs per SM, each at least 8192 elements
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(2 * dev.sms, rows * vocab / 8192));
    if (ctas + rows > kNoAllocKeys) return CE_ERANGE;
    uint64_t *keys = nullptr;
    if ((st = noalloc_scratch(dev, &keys))) return st;
    Args a = make_args(logits, rows, vocab, stride, nullptr);
    a.top = top;
    return cuda_status(launch_argmax_flat(a, static_cast<int>(ctas), keys, stream));
}

const char *ce_status_string(int status) {
    switch (status) {
    case CE_OK: return "ok";
    case CE_EINVAL: return "invalid argument (null pointer, size, stride, vocab > 2^24, scale or forced plan)";
    case CE_EALIGN: return "pointer not aligned to its element size";
    case CE_ECUDA: return "CUDA runtime error at launch (see ce_last_cuda_error)";
    case CE_EDEVICE: return "no usable sm_103 CUDA device";
    case CE_ERANGE: return "too many rows for argmax_rows_noalloc's fixed scratch (rows + 2 * SMs must be <= 8192)";
    default: return "unknown status";
    }
}

int ce_grad_host(const float *logits_h, int64_t rows, int64_t vocab, int64_t stride_h, const int64_t *labels_h,
                 double scale, float *logits_d, int64_t *labels_d, float *grad, float *loss_rows, float *top,
                 double *loss_mean, double *loss_mean_h, float *top_h, int64_t chunk_rows, ce_stream_t stream) {
    int st = check_logits(logits_h, rows, vocab, stride_h);
    if (st) return st;
    if (!std::isfinite(scale) || chunk_rows < 0 || loss_mean == nullptr) return CE_EINVAL;
    if (rows > 0 && (labels_h == nullptr || logits_d == nullptr || labels_d == nullptr || grad == nullptr ||
                     loss_rows == nullptr))
        return CE_EINVAL;
    if (top_h != nullptr && top == nullptr) return CE_EINVAL;
    if (misaligned(labels_h, 8) || misaligned(logits_d, 4) || misaligned(labels_d, 8) || misaligned(grad, 4) ||
        misaligned(loss_rows, 4) || misaligned(top, 4) || misaligned(loss_mean, 8) || misaligned(loss_mean_h, 8) ||
        misaligned(top_h, 4))
        return CE_EALIGN;
    const int64_t dense = rows * vocab * 4;
    if (grad != logits_d && ranges_overlap(grad, dense, logits_d, dense)) return CE_EINVAL;
    DeviceInfo dev;
    if ((st = current_device(&dev))) return st;
    HostPipe &h = g_pipe[dev.device];
    std::lock_guard<std::mutex> lock(h.mu);
    cudaError_t e = host_pipe_ready(h);
    if (e != cudaSuccess) return cuda_status(e);
    if (rows > 0) {
        int64_t n = chunk_rows > 0 ? ceil_div(rows, chunk_rows) : std::min<int64_t>(rows, 16);
        n = std::min<int64_t>(n, kHostChunksMax);
        const int64_t chunk = ceil_div(rows, n);
        n = ceil_div(rows, chunk);
        // the copies start once earlier work on the stream (which may still
        // read logits_d or labels_d) is done
        if ((e = cudaEventRecord(h.start, stream)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaStreamWaitEvent(h.copy, h.start, 0)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaMemcpyAsync(labels_d, labels_h, static_cast<size_t>(rows) * 8, cudaMemcpyHostToDevice,
                                 h.copy)) != cudaSuccess)
            return cuda_status(e);
        for (int64_t c = 0; c < n; ++c) {
            const int64_t r0 = c * chunk, r1 = std::min(rows, r0 + chunk);
            e = cudaMemcpy2DAsync(logits_d + r0 * vocab, static_cast<size_t>(vocab) * 4, logits_h + r0 * stride_h,
                                  static_cast<size_t>(stride_h) * 4, static_cast<size_t>(vocab) * 4,
                                  static_cast<size_t>(r1 - r0), cudaMemcpyHostToDevice, h.copy);
            if (e == cudaSuccess) e = cudaEventRecord(h.chunk[c], h.copy);
            if (e != cudaSuccess) return cuda_status(e);
        }
        // chunk c's kernel runs while chunk c + 1 is copied
        for (int64_t c = 0; c < n; ++c) {
            const int64_t r0 = c * chunk, r1 = std::min(rows, r0 + chunk);
            if ((e = cudaStreamWaitEvent(stream, h.chunk[c], 0)) != cudaSuccess) return cuda_status(e);
            st = grad_rows(logits_d + r0 * vocab, r1 - r0, vocab, vocab, labels_d + r0, scale, grad + r0 * vocab,
                           loss_rows + r0, top ? top + r0 : nullptr, stream);
            if (st) return st;
        }
    }
    if ((st = ce_mean(loss_rows, rows, loss_mean, stream))) return st;
    if (loss_mean_h && (e = cudaMemcpyAsync(loss_mean_h, loss_mean, 8, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
        return cuda_status(e);
    if (top_h && rows > 0 &&
        (e = cudaMemcpyAsync(top_h, top, static_cast<size_t>(rows) * 4, cudaMemcpyDeviceToHost, stream)) !=
            cudaSuccess)
        return cuda_status(e);
    return CE_OK;
}

int ce_version(void) { return kVersion; }

int ce_last_cuda_error(void) { return t_last_cuda_error; }

// Reads device counter `which` (0 bad labels, 1 waits that gave up); waits for `stream`.
static int read_counter(ce_stream_t stream, int which, int64_t *out) {
    if (out == nullptr) return CE_EINVAL;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    unsigned long long v[2] = {0ull, 0ull};
    if ((st = cuda_status(read_status(v, stream)))) return st;
    *out = static_cast<int64_t>(v[which]);
    return CE_OK;
}

int ce_device_error_count(ce_stream_t stream, int64_t *out) { return read_counter(stream, 0, out); }

int ce_device_wait_timeouts(ce_stream_t stream, int64_t *out) { return read_counter(stream, 1, out); }

int ce_device_error_reset(ce_stream_t stream) {
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    return cuda_status(reset_status(stream));
}

int ce_debug_force(int path, int cluster, int threads) {
    if (path < 0 || path > kPathRing || cluster < 0 || cluster > kMaxCluster) return CE_EINVAL;
    if (threads != 0 && threads != 128 && threads != 256 && threads != 512) return CE_EINVAL;
    std::lock_guard<std::mutex> lock(g_mu);
    g_force.path = path;
    g_force.cluster = cluster;
    g_force.threads = threads;
    return CE_OK;
}

int ce_debug_grid_cap(int64_t clusters) {
    if (clusters < 0) return CE_EINVAL;
    std::lock_guard<std::mutex> lock(g_mu);
    g_force.grid_cap = clusters;
    return CE_OK;
}

int ce_debug_read(const void *p, int64_t bytes, uint32_t *out, ce_stream_t stream) {
    if (bytes < 0 || out == nullptr || (bytes > 0 && p == nullptr)) return CE_EINVAL;
    if (bytes % 16 != 0) return CE_EINVAL;
    if (misaligned(p, 16) || misaligned(out, 4)) return CE_EALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    return cuda_status(launch_read_probe(p, bytes, out, dev.sms, stream));
}

int ce_plan(int op, int64_t rows, int64_t vocab, int64_t stride, int64_t out[6]) {
    if (out == nullptr || op < 0 || op > kOpCandidates) return CE_EINVAL;
    if (rows < 1 || vocab < 1 || vocab > kMaxVocab || stride < vocab) return CE_EINVAL;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st) return st;
    Plan p;
    if ((st = make_plan(static_cast<Op>(op), rows, vocab, dev, &p))) return st;
    out[0] = p.path;
    out[1] = p.cluster;
    out[2] = p.threads;
    out[3] = p.smem;
    out[4] = p.cols;
    out[5] = p.clusters * p.cluster;
    return CE_OK;
}

}  // extern "C"
