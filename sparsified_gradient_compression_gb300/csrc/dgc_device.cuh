// dgc_device.cuh -- device-side building blocks shared by the libdgc kernels (sm_103a).
//
// Keys, the SplitMix64 output function, status reporting, block-wide scans, and the
// decoupled look-back that turns per-tile counts into global offsets in one pass with a
// bounded wait.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dgc.h"

namespace dgc {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;  // SplitMix64 increment
constexpr uint32_t kNoKey = 0x80000000u;             // above every 31-bit |v| key
constexpr uint32_t kRunEscape = 0xFFFFu;
constexpr uint32_t kMagic = 0x31434744u;             // "DGC1" little-endian
constexpr uint64_t kBillion = 1000000000ull;
constexpr uint32_t kDefaultSpinLimit = 1u << 21;     // polls of a look-back flag (~0.1-1 s)
constexpr unsigned kFull = 0xFFFFFFFFu;

// |x| as an integer with the order of |x| for finite x (+0 and -0 tie; NaN above inf).
__device__ __forceinline__ uint32_t key_of(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// SplitMix64 output function (Steele, Lea and Flood, OOPSLA 2014).
__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// ceil(n * ppb / 1e9) for n < 2^32, ppb <= 1e9 (the product fits in 64 bits).
__host__ __device__ __forceinline__ uint64_t count_ppb(uint64_t n, uint64_t ppb) {
    return (n * ppb + (kBillion - 1)) / kBillion;
}

// First error wins; the library never clears a status word.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// Exclusive scan across a block of kThreads threads (kThreads a multiple of 32, <= 1024).
// `smem` holds at least 33 T. Returns the exclusive prefix; *total gets the block sum.
template <int kThreads, typename T>
__device__ __forceinline__ T block_excl_scan(T x, T* smem, T* total) {
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T inc = warp_incl_scan(x);
    if (lane == 31) smem[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        T w = lane < kWarps ? smem[lane] : T(0);
        T wi = warp_incl_scan(w);
        if (lane < kWarps) smem[lane] = wi - w;
        if (lane == kWarps - 1) smem[32] = wi;
    }
    __syncthreads();
    T res = smem[warp] + inc - x;
    *total = smem[32];
    __syncthreads();
    return res;
}

// ---------------------------------------------------------------- decoupled look-back
// One 64-bit status word per tile: bits 63..62 flag (0 none yet, 1 aggregate, 2 inclusive
// prefix), bits 61..0 value. A tile publishes its own aggregate first, then walks back over
// its predecessors 32 at a time (one lane each), adding aggregates until it meets an inclusive
// prefix. Tiles take their ids from an atomic ticket in launch order, so every predecessor is
// already running and will publish without waiting on anything: the wait ends. It is still
// bounded: after `spin_limit` polls the tile reports DGC_ETIMEOUT, raises *abort and counts the
// missing predecessors as zero (the call's results are then invalid, but every write stays
// inside its buffer because writers check capacities).
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValMask = (1ull << 62) - 1;

// Called by all 32 lanes of one warp; returns the exclusive prefix of `tile`.
__device__ __forceinline__ uint64_t lookback_exclusive(uint64_t* st, uint32_t tile, uint64_t agg,
                                                       uint32_t spin_limit, int32_t* status,
                                                       int32_t* abort_flag) {
    const int lane = threadIdx.x & 31;
    if (tile == 0) {
        if (lane == 0) st_relaxed(&st[0], kFlagInc | (agg & kValMask));
        return 0;
    }
    if (lane == 0) st_relaxed(&st[tile], kFlagAgg | (agg & kValMask));
    uint64_t excl = 0;
    int64_t pred = (int64_t)tile - 1;
    while (true) {
        const int64_t i = pred - lane;
        uint64_t w = (i >= 0) ? ld_relaxed(&st[i]) : kFlagInc;  // before tile 0: prefix 0
        uint32_t spins = 0;
        while (__any_sync(kFull, (w >> 62) == 0)) {
            if (++spins > spin_limit) {
                if (lane == 0) {
                    report(status, DGC_ETIMEOUT);
                    if (abort_flag) atomicExch(abort_flag, 1);
                }
                if ((w >> 62) == 0) w = kFlagInc;
                break;
            }
            __nanosleep(64);
            if ((w >> 62) == 0) w = ld_relaxed(&st[i]);
        }
        const unsigned inc = __ballot_sync(kFull, (w >> 62) == 2);
        uint64_t val = w & kValMask;
        if (inc) {
            const int first = __ffs(inc) - 1;
            if (lane > first) val = 0;
            excl += warp_sum(val);
            break;
        }
        excl += warp_sum(val);
        pred -= 32;
    }
    if (lane == 0) st_relaxed(&st[tile], kFlagInc | ((excl + agg) & kValMask));
    return excl;
}

// Decoupled look-back walked by a whole block (kThreads predecessors per round trip), for
// kernels whose other warps would otherwise idle during the walk. Same status words, limits
// and timeout behaviour as lookback_exclusive. Every thread of the block must call it; `sm`
// is shared scratch of at least 2 uint32 + 33 uint64.
// With publish_agg false the caller has already published the tile's aggregate (or, for tile
// 0, its inclusive prefix).
template <int kThreads>
__device__ __forceinline__ uint64_t block_lookback(uint64_t* st, uint32_t tile, uint64_t agg,
                                                   uint32_t spin_limit, int32_t* status,
                                                   int32_t* abort_flag, uint32_t* sm_u32,
                                                   uint64_t* sm_u64, bool publish_agg = true) {
    const int tid = threadIdx.x;
    if (tid == 0 && publish_agg)
        st_relaxed(&st[tile], (tile == 0 ? kFlagInc : kFlagAgg) | (agg & kValMask));
    if (tile == 0) return 0;
    uint64_t excl = 0;
    int64_t pred = (int64_t)tile - 1;
    while (true) {
        const int64_t i = pred - tid;
        uint64_t w = (i >= 0) ? ld_relaxed(&st[i]) : kFlagInc;  // before tile 0: prefix 0
        uint32_t spins = 0;
        uint32_t nearest;  // 0xFFFFFFFF: no inclusive prefix among these predecessors
        while (true) {
            if (tid == 0) sm_u32[0] = 0xFFFFFFFFu;
            __syncthreads();
            if ((w >> 62) == 2) atomicMin(&sm_u32[0], (uint32_t)tid);
            __syncthreads();
            nearest = sm_u32[0];  // nearest predecessor with an inclusive prefix
            const bool need = ((w >> 62) == 0) && (uint32_t)tid < nearest;
            if (!__syncthreads_or(need)) break;
            if (++spins > spin_limit) {
                if (tid == 0) {
                    report(status, DGC_ETIMEOUT);
                    if (abort_flag) atomicExch(abort_flag, 1);
                }
                if ((w >> 62) == 0) w = kFlagInc;
                continue;
            }
            if (need) {
                __nanosleep(64);
                w = ld_relaxed(&st[i]);
            }
        }
        uint64_t val = ((uint32_t)tid <= nearest) ? (w & kValMask) : 0;
        uint64_t sum;
        block_excl_scan<kThreads>(val, sm_u64, &sum);
        excl += sum;
        if (nearest != 0xFFFFFFFFu) break;
        pred -= kThreads;
    }
    if (tid == 0) st_relaxed(&st[tile], kFlagInc | ((excl + agg) & kValMask));
    return excl;
}

// ------------------------------------------------- bulk copies (TMA) and mbarriers, sm_90+
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
// Non-blocking probe of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Order this thread's earlier generic-proxy accesses to shared memory before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to this
// block's shared memory; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from this block's
// shared memory to global memory, as part of the thread's current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every bulk group this thread committed has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Largest s in [0, n) with a[s] <= x, for a non-decreasing a with a[0] <= x (n >= 1).
template <typename T>
__device__ __forceinline__ int upper_bound_minus1(const T* a, int n, T x) {
    int lo = 0, hi = n;  // invariant: a[lo] <= x, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace dgc

// Internal (not exported): count kernel launches for dgc_launch_count().
void dgc_internal_count_launches(uint64_t k);
int dgc_internal_sm_count();
