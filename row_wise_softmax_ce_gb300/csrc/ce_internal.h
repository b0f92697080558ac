// ce_internal.h -- launch plans and kernel launchers shared by the C ABI
// (ce_api.cu) and the kernels (ce_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace cerows {

enum Path : int {
    kPathAuto = 0,
    kPathStaged = 1,
    kPathStream = 2,
    kPathRetired3 = 3,  // once a ring-of-copies kernel; now refused
    kPathStagedPerRow = 4,
    kPathFlat = 5,
    kPathWarp = 6,  // one warp per row (ce_rows, argmax, slice statistics of many short rows)
    kPathRing = 7,  // argmax through a ring of bulk-copied row chunks (few long rows)
};
enum Op : int { kOpRows = 0, kOpGrad = 1, kOpArgmax = 2, kOpSoftmax = 3, kOpLogSoftmax = 4, kOpCandidates = 5 };
// What the fused two-pass kernels write from a row's (max, exp-sum) state.
enum Mode : int { kModeGrad = 0, kModeSoftmax = 1, kModeLogSoftmax = 2 };

// candidatesInto: a workgroup of 256 threads, each keeping its TOP_EACH = 4
// largest values; a row's candidates are 2048 floats (value, token pairs).
constexpr int kCandThreads = 256;
constexpr int kTopEach = 4;
constexpr int kCandRow = 2 * kCandThreads * kTopEach;
constexpr int kCandMaxCluster = 8;
// Shared memory of the candidates kernel: mbarriers and counters, a ring of
// kCandStages chunks of a row (B blocks of 256 columns on the 16-byte grid of
// the logits: up to 3 floats before the chunk and 1 after), and, for rows
// split over a cluster, the lists CTA 0 pulls from the others. Two chunk
// sizes: 15 blocks keep a split-row CTA at 54 KB (four per SM) for grids of
// many CTAs; 32 blocks (104 KB, two per SM) halve the per-chunk overhead where
// the grid has at most two CTAs per SM (256 decode rows of 151936: 39.1 ->
// about 33 us).
constexpr int kCandChunkSmall = 15;
constexpr int kCandChunkLarge = 32;
constexpr int kCandStages = 3;
constexpr int kCandHeaderBytes = 48;
constexpr int kCandListBytes = kCandThreads * kTopEach * 8;
constexpr int kRingArgmaxSlotBytes = kCandThreads * 8;  // one (value, column) per thread (split rows)
constexpr int cand_stage_floats(int blocks) { return blocks * kCandThreads + 4; }
constexpr int cand_ring_bytes(int blocks) { return kCandHeaderBytes + kCandStages * cand_stage_floats(blocks) * 4; }
constexpr int cand_max_smem_bytes(int blocks) { return cand_ring_bytes(blocks) + kCandListBytes; }
static_assert(kCandStages * 12 <= kCandHeaderBytes && kCandHeaderBytes % 16 == 0 &&
                  cand_stage_floats(kCandChunkSmall) % 4 == 0 && cand_stage_floats(kCandChunkLarge) % 4 == 0 &&
                  4 * (cand_max_smem_bytes(kCandChunkSmall) + 1024) <= 228 * 1024 &&
                  2 * (cand_max_smem_bytes(kCandChunkLarge) + 1024) <= 228 * 1024 && kCandChunkLarge <= 32,
              "candidates smem layout: four small-chunk or two large-chunk CTAs per SM; a 32-bit mark mask");
constexpr int kSplitThreads = 256;

// Per-CTA shared bytes the staged kernel reserves before its row buffer.
constexpr int kStagedHeaderBytes = 2048;
constexpr int kMaxCluster = 16;
// Largest CTA each kernel family is compiled for (its __launch_bounds__).
constexpr int kStagedMaxThreads = 256;
constexpr int kStreamMaxThreads = 256;
struct Plan {
    int path = kPathStream;
    int cluster = 1;       // CTAs per row (a thread-block cluster)
    int threads = 256;     // threads per CTA
    int smem = 0;          // dynamic shared bytes per CTA
    int cols = 0;          // columns per CTA (a multiple of 4)
    int chunk = 0;         // candidates and ring argmax: blocks of 256 columns per ring chunk
    int64_t clusters = 0;  // clusters in the grid (each loops over rows)
};

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int max_smem_optin = 0;  // per block
    int cc_major = 0, cc_minor = 0;
};

// Arguments of one launch; unused pointers are null.
struct Args {
    const float *logits;
    int64_t rows;
    int vocab;
    int64_t stride;
    const int64_t *labels;
    float scale;
    float *grad;
    float *loss;
    float *top;
    float *stats;   // vocab-sharded rows: [rows] float4 (m, t, top, x[label]) of the slice
    int64_t col0;   // vocab-sharded rows: global column of the slice's first column
    const uint64_t *row_at;  // rows given by address (argmaxInto's indirect form), or null
};

cudaError_t set_kernel_attributes(const DeviceInfo &dev);
cudaError_t max_active_clusters(const Plan &p, Op op, int *n);

cudaError_t launch_rows_stream(const Plan &p, const Args &a, bool stats, cudaStream_t s);
// the two-pass kernels (staged or stream, as p.path says) for kOpGrad,
// kOpSoftmax or kOpLogSoftmax; the output row goes to a.grad
cudaError_t launch_fused(const Plan &p, Op op, const Args &a, cudaStream_t s);
// cand: rows * kCandRow floats
cudaError_t launch_candidates(const Plan &p, const Args &a, float *cand, cudaStream_t s);
// one resident wave on a device of `sms` SMs
cudaError_t launch_split_sum(float *y, const float *parts, int64_t total, int64_t splits, bool add, int sms,
                             cudaStream_t s);
cudaError_t launch_mean(const float *loss, int64_t rows, double *out, cudaStream_t s);
// vocab-sharded rows: combine `shards` slices' statistics; gradient of one slice
cudaError_t launch_stats_combine(const float *stats, int64_t shards, int64_t rows, int64_t vocab_total,
                                 const int64_t *labels, float *loss, float *top, float *combined, int sms,
                                 cudaStream_t s);
cudaError_t launch_grad_from_stats(const Args &a, const float *combined, int sms, cudaStream_t s);
// argmax of few long rows split evenly over `ctas` CTAs; ws: 8 * (ctas + rows) bytes
cudaError_t launch_argmax_flat(const Args &a, int ctas, void *ws, cudaStream_t s);

// a plain read of `bytes` (a multiple of 16, 16-byte aligned) in one resident wave
cudaError_t launch_read_probe(const void *p, int64_t bytes, uint32_t *out, int sms, cudaStream_t s);

cudaError_t read_status(unsigned long long out[2], cudaStream_t s);
cudaError_t reset_status(cudaStream_t s);

}  // namespace cerows
