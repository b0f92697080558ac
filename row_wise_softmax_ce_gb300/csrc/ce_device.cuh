// ce_device.cuh -- device-side building blocks of the row-wise softmax
// cross-entropy kernels for sm_103a: inline-PTX wrappers (mbarrier, bulk
// asynchronous copies, thread-block clusters and distributed shared memory,
// streaming loads and stores) and the per-row online state.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace cerows {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kNoIndex = 0x7fffffff;  // "no column seen yet"

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// mbarrier in this CTA's shared memory
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async proxy and the cluster
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this thread's earlier generic-proxy shared accesses before later
// async-proxy (bulk copy) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// atomic add on a shared counter, acquire + release at CTA scope; returns
// the old value
__device__ __forceinline__ uint32_t atom_add_acq_rel_smem(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
    return old;
}

// One poll of the phase with the given parity. A thread whose phase has not
// completed is suspended in hardware (it issues nothing) until the phase
// completes or about `suspend_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity, uint32_t suspend_ns = 1000000u) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return done != 0;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// `limit_ns` nanoseconds and 2^20 polls. Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = 200000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < (1u << 20); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Bulk asynchronous copy (the TMA engine, no tensor map) from global memory
// into this CTA's shared memory; completion is signalled on `bar` as bytes.
// dst and src must be 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy: lines read once are the first to be evicted.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// thread-block cluster
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster calls these, in uniform control
// flow, alternating arrive and wait. The arrive is relaxed: a thread whose
// shared-memory writes peers must see calls fence_cluster() first.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// An arrive that releases this thread's earlier writes (shared memory of
// peers included) to the threads that pass the matching cluster_wait.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Programmatic dependent launch. launch_dependents: the next kernel on the
// stream, if launched with programmatic stream serialization, may be
// scheduled once every CTA of this grid has called it (or exited).
// wait_prerequisites: block until the grids this one depends on have
// completed and their memory is visible; a no-op without such a dependency.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_smem(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// 8-byte store into the shared memory of a CTA of the cluster (a
// shared::cluster address from peer_smem).
__device__ __forceinline__ void st_dsmem_f64(uint32_t addr, double v) {
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(addr), "d"(v) : "memory");
}

// 16-byte store into the shared memory of a CTA of the cluster (a
// shared::cluster address from peer_smem), completing `bytes` = 16 on that
// CTA's mbarrier (also a shared::cluster address).
__device__ __forceinline__ void st_async_peer(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile("st.async.weak.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                 "r"(__float_as_uint(v.w)), "r"(bar)
                 : "memory");
}

// L2 policy: lines kept in preference to others (read again soon).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// global loads and stores
// read-only data read once: skip L1
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_stream_f1(const float *p) {
    float v;
    asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// exp(d) for d <= 0 by the change of base exp(d) = 2^(d * log2(e)), with the
// hardware base-2 exponential ex2.approx.ftz.f32 (relative error below 2^-22;
// results below 2^-126 flush to 0, i.e. an absolute error below 1.2e-38).
// Rounding the product d * log2(e) adds a relative error of about
// |d| * 2^-24 to the result -- at most 2.2e-8 absolute, since |d| * exp(d)
// <= 1/e for d <= 0.
__device__ __forceinline__ float ex2_ftz(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}
__device__ __forceinline__ float exp_le0(float d) { return ex2_ftz(d * 1.4426950408889634f); }

// ---------------------------------------------------------------------------
// Online row state.
//
// Over the columns pushed so far: m is their max (NaN is skipped: it never
// compares greater), idx the first column holding m (kNoIndex if none), and
// t = sum of exp(x_j - m) over every pushed column but one that holds m --
// so the row's exp-sum is 1 + t. Keeping the "1" out of t lets the loss be
// formed as (m - x[label]) + log1p(t) without cancellation.
//
// Push x (column j):
//   x >  m:  t <- (1 + t) * exp(m - x),  m <- x,  idx <- j
//   x == m:  t <- t + 1                  (a tie; idx keeps the first)
//   else:    t <- t + exp(x - m)         (NaN x makes t NaN, and it stays NaN)
// x == m also covers -inf == -inf and +inf == +inf, where x - m is NaN.
// In the first two cases exp takes -|x - m|, so one exp serves both; it is
// exp_le0 (above), as in the common path. (CUDA's expf on this path -- the
// one a warp takes whenever one of its lanes meets a new max -- cost 9% of
// ce_rows on 4096 x 32000 and 18% on 256 x 151936.)
//
// Merge two states: the winner has the larger m (ties: smaller idx); then
//   t <- t_w + (1 + t_l) * exp(m_l - m_w).
// The merge is symmetric, so a butterfly gives every lane the same bits.

struct RowState {
    float m;
    float t;
    int idx;
};

__device__ __forceinline__ RowState empty_state() { return RowState{-INFINITY, 0.0f, kNoIndex}; }

template <bool kStats>
__device__ __forceinline__ void push(RowState &s, float x, int j) {
    const bool gt = x > s.m;
    const bool eq = x == s.m;
    if (kStats) {
        const float e = eq ? 1.0f : exp_le0(-fabsf(x - s.m));
        s.t = gt ? fmaf(s.t, e, e) : s.t + e;
    }
    s.idx = gt ? j : (eq ? min(s.idx, j) : s.idx);
    s.m = gt ? x : s.m;
}

template <bool kStats>
__device__ __forceinline__ void push4(RowState &s, float4 v, int j) {
    push<kStats>(s, v.x, j);
    push<kStats>(s, v.y, j + 1);
    push<kStats>(s, v.z, j + 2);
    push<kStats>(s, v.w, j + 3);
}

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

// exp(v - m) lane by lane (every lane <= m), the subtraction and the scaling
// by log2(e) done two lanes per instruction (Blackwell paired f32 ops).
__device__ __forceinline__ float4 exp4_sub(float4 v, float m) {
    const float2 nm = make_float2(-m, -m), l2e = make_float2(1.4426950408889634f, 1.4426950408889634f);
    const float2 a = __fmul2_rn(__fadd2_rn(make_float2(v.x, v.y), nm), l2e);
    const float2 b = __fmul2_rn(__fadd2_rn(make_float2(v.z, v.w), nm), l2e);
    return make_float4(ex2_ftz(a.x), ex2_ftz(a.y), ex2_ftz(b.x), ex2_ftz(b.y));
}

__device__ __forceinline__ float4 mul4(float4 v, float c) {
    const float2 cc = make_float2(c, c);
    const float2 a = __fmul2_rn(make_float2(v.x, v.y), cc);
    const float2 b = __fmul2_rn(make_float2(v.z, v.w), cc);
    return make_float4(a.x, a.y, b.x, b.y);
}

// (v - m) - l lane by lane, two lanes per instruction: a log-softmax row
// from its max m and l = log(sum).
__device__ __forceinline__ float4 sub2_4(float4 v, float m, float l) {
    const float2 nm = make_float2(-m, -m), nl = make_float2(-l, -l);
    const float2 a = __fadd2_rn(__fadd2_rn(make_float2(v.x, v.y), nm), nl);
    const float2 b = __fadd2_rn(__fadd2_rn(make_float2(v.z, v.w), nm), nl);
    return make_float4(a.x, a.y, b.x, b.y);
}

// Push four consecutive columns j..j+3. Common case: none of them exceeds the
// running max m (and m is above -inf), so each adds exp(x - m) -- a tie adds
// exactly 1 and keeps the first index, a NaN makes t NaN. Otherwise (a new
// max, or no finite value yet, or all four NaN) the exact scalar update runs.
// Both take exp_le0 (ex2.approx of d * log2(e), above: below about 2.5e-7
// relative and 2.2e-8 absolute for the rounding of the product).
template <bool kStats>
__device__ __forceinline__ void push_vec(RowState &s, float4 v, int j) {
    const float mv = max4(v);
    if (mv <= s.m && s.m != -INFINITY) {
        if (kStats) {
            // the same bits as exp_le0 lane by lane, two lanes per f32 instruction
            // (256 x 151936 row losses, L2 flushed: 35.3 -> 34.7 us)
            const float4 e = exp4_sub(v, s.m);
            s.t += (e.x + e.y) + (e.z + e.w);
        }
    } else {
        push4<kStats>(s, v, j);
    }
}

template <bool kStats>
__device__ __forceinline__ RowState merge(const RowState a, const RowState b) {
    const bool b_wins = (b.m > a.m) || (b.m == a.m && b.idx < a.idx);
    RowState r;
    r.m = b_wins ? b.m : a.m;
    r.idx = b_wins ? b.idx : a.idx;
    r.t = 0.0f;
    if (kStats) {
        const float wt = b_wins ? b.t : a.t;
        const float lt = b_wins ? a.t : b.t;
        const float lm = b_wins ? a.m : b.m;
        const float e = (lm == r.m) ? 1.0f : exp_le0(lm - r.m);
        r.t = fmaf(1.0f + lt, e, wt);
    }
    return r;
}

template <bool kStats>
__device__ __forceinline__ RowState shfl_xor_state(const RowState &s, int o) {
    RowState q;
    q.m = __shfl_xor_sync(kFullMask, s.m, o);
    q.t = kStats ? __shfl_xor_sync(kFullMask, s.t, o) : 0.0f;
    q.idx = __shfl_xor_sync(kFullMask, s.idx, o);
    return q;
}

template <bool kStats>
__device__ __forceinline__ RowState warp_reduce(RowState s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = merge<kStats>(s, shfl_xor_state<kStats>(s, o));
    return s;
}


// Reduce over the CTA into warp 0: every lane of warp 0 returns the CTA's
// state (other warps return garbage). `red` holds >= 32 states in shared
// memory. Contains one __syncthreads.
template <bool kStats>
__device__ __forceinline__ RowState block_reduce_w0(RowState s, RowState *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    s = warp_reduce<kStats>(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    RowState r = empty_state();
    if (warp == 0) {
        if (lane < nwarps) r = red[lane];
        r = warp_reduce<kStats>(r);
    }
    return r;
}

// What a CTA publishes to its cluster peers for one row.
struct __align__(16) Xchg {
    float m;
    float t;
    int idx;
    float xl;  // x[label], if the label column lies in this CTA's slice
};

__device__ __forceinline__ Xchg ld_peer_xchg(const Xchg *x, uint32_t rank) {
    const float4 v = ld_dsmem_f4(peer_smem(x, rank));
    return Xchg{v.x, v.y, __float_as_int(v.z), v.w};
}

// In warp 0: merge the C published states of the cluster (lane r reads CTA
// r's), a fixed tree, so every CTA of the cluster gets the same bits. Lane 0
// returns the row state; *xl gets the x[label] published by CTA `owner`.
template <bool kStats>
__device__ __forceinline__ RowState cluster_merge_w0(const Xchg *x, uint32_t C, uint32_t owner, float *xl) {
    const int lane = threadIdx.x & 31;
    RowState s = empty_state();
    float v = 0.0f;
    if (lane < static_cast<int>(C)) {
        const Xchg q = ld_peer_xchg(x, static_cast<uint32_t>(lane));
        s = RowState{q.m, q.t, q.idx};
        v = q.xl;
    }
    *xl = __shfl_sync(kFullMask, v, static_cast<int>(owner));
    return warp_reduce<kStats>(s);
}

// Row-state exchange among the C CTAs of a cluster by pushes: for row k of
// the cluster, thread 0 of every CTA stores its state into slot k % 2 of
// every CTA (st.async, completing 16 bytes on that CTA's slot barrier), and
// warp 0 of every CTA waits for the C states of its own slot and merges them
// in rank order -- the same bits in every CTA, and no cluster barrier per
// row. Two slots suffice: a CTA pushes row k + 2 only after it has merged
// row k + 1, which needs this CTA's push of row k + 1, which this CTA makes
// only after it has read slot k % 2 for row k. The cluster must pass one
// cluster barrier between push_xchg_init and the first push (so that every
// slot barrier exists), and one before any CTA exits.
struct PushXchg {
    Xchg slot[2][16];
    uint64_t bar[2];
};

// thread 0; K = rows this cluster will exchange
__device__ __forceinline__ void push_xchg_init(PushXchg &x, int64_t K, uint32_t C) {
    for (int i = 0; i < 2; ++i) mbar_init(&x.bar[i], 1);
    fence_mbar_init();
    for (int i = 0; i < 2; ++i)
        if (i < K) mbar_arrive_expect_tx(&x.bar[i], 16u * C);
}

// thread 0
__device__ __forceinline__ void push_xchg_publish(PushXchg &x, int64_t k, uint32_t rank, uint32_t C,
                                                  const RowState &st, float xl) {
    const int xs = static_cast<int>(k & 1);
    const float4 v = make_float4(st.m, st.t, __int_as_float(st.idx), xl);
    for (uint32_t r = 0; r < C; ++r) st_async_peer(peer_smem(&x.slot[xs][rank], r), v, peer_smem(&x.bar[xs], r));
}

// all of warp 0: the merged row state (every lane); *xl = the x[label]
// published by CTA `owner`. Re-arms the slot for row k + 2.
template <bool kStats>
__device__ __forceinline__ RowState push_xchg_merge(PushXchg &x, int64_t k, int64_t K, uint32_t C, uint32_t owner,
                                                    float *xl, bool *failed) {
    const int lane = threadIdx.x & 31;
    const int xs = static_cast<int>(k & 1);
    if (!*failed) *failed = !mbar_wait_bounded(&x.bar[xs], static_cast<uint32_t>(k >> 1) & 1u);
    RowState q = empty_state();
    float v = 0.0f;
    if (lane < static_cast<int>(C)) {
        const Xchg e = x.slot[xs][lane];
        q = RowState{e.m, e.t, e.idx};
        v = e.xl;
    }
    *xl = __shfl_sync(kFullMask, v, static_cast<int>(owner));
    const RowState g = warp_reduce<kStats>(q);
    if (lane == 0 && k + 2 < K) mbar_arrive_expect_tx(&x.bar[xs], 16u * C);
    return g;
}

}  // namespace cerows
