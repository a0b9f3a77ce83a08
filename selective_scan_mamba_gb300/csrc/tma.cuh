// tma.cuh -- tensor-memory-accelerator copies and mbarriers (sm_90+ PTX, used on sm_103a).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// make initialised barriers visible to the async (TMA) proxy
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------------------------------
// Bounded waits.  A kernel that waits on mbarriers calls wait_setup() from thread 0 before
// its first __syncthreads.  A wait polls its barrier up to the CTA's limit (default 2^24
// polls, far longer than any copy or MMA takes).  If the limit runs out, the wait counts
// the event in a device counter that the host reads and clears (ssm_device_status and
// ssm_wait_timeouts), marks the CTA as aborted and returns false.  From then on every wait
// in the CTA returns false within 1024 polls.  The kernel keeps to its normal control flow and meets
// every block barrier, but its threads issue no further copies or MMAs.  Before the CTA
// frees its tensor memory and exits, the threads that issued asynchronous work wait
// (mbar_drain, with the default limit and ignoring the abort) for what they issued.  The
// outputs of an aborted call are not valid; the host learns of it through the counter.
// ---------------------------------------------------------------------------------------

// One counter per translation unit; ssm_device_status reads and clears each of them.
static __device__ unsigned int g_ssm_wait_timeouts = 0;

// Host side: reads this translation unit's counter into *count and clears it.  Waits for
// the device first, so that the kernels launched before it have finished.
static inline cudaError_t take_wait_timeouts(unsigned int* count) {
    *count = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    unsigned int v = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_ssm_wait_timeouts, sizeof(v))) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_ssm_wait_timeouts, &zero, sizeof(zero))) != cudaSuccess) return e;
    *count = v;
    return cudaSuccess;
}

constexpr uint32_t kWaitPolls = 1u << 24;

static __shared__ uint32_t s_wait_abort;  // nonzero once a wait in this CTA gave up
static __shared__ uint32_t s_wait_limit;  // polls before a wait gives up

// Thread 0, before the kernel's first __syncthreads.  limit 0 = kWaitPolls; the limit is
// counted in whole blocks of 1024 polls (at least one block).
__device__ __forceinline__ void wait_setup(uint32_t limit) {
    s_wait_abort = 0;
    s_wait_limit = limit ? limit : kWaitPolls;
}

__device__ __forceinline__ bool wait_aborted() {
    return *reinterpret_cast<volatile uint32_t*>(&s_wait_abort) != 0;
}

// The same, one answer for the whole warp (all 32 lanes must call it): for decisions that
// guard warp-collective instructions such as an elected-lane MMA issue.
__device__ __forceinline__ bool wait_aborted_warp() {
    return __any_sync(0xffffffffu, wait_aborted());
}

// Slow path of the waits, taken after 1024 unsuccessful polls: polls on, reading the abort
// flag and the limit once per 1024 polls.
__device__ __forceinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 1024;; i += 1024) {
        if (wait_aborted()) return false;
        if (i >= *reinterpret_cast<volatile uint32_t*>(&s_wait_limit)) break;
        for (uint32_t j = 0; j < 1024; ++j)
            if (mbar_try_wait(bar, parity)) return true;
    }
    *reinterpret_cast<volatile uint32_t*>(&s_wait_abort) = 1u;
    atomicAdd(&g_ssm_wait_timeouts, 1u);
    return false;
}
static __device__ __noinline__ bool mbar_wait_slow_call(uint64_t* bar, uint32_t parity) {
    return mbar_wait_slow(bar, parity);
}

// Waits for phase `parity` of the barrier.  Returns false if the CTA has aborted or the
// limit ran out (which aborts it); the caller then skips issuing further work.  The first
// 1024 polls are a bare loop of constant length, with the abort flag and the limit read
// only on the slow path: loops that read them on every pass made the waiting threads take
// issue slots from the working ones (the SSD walk measured 1.7x slower).  The exact form
// was chosen by measurement: for waits by every thread (the Mamba-1 kernels) the slow path
// is inlined; for waits by one lane of a warp (mbar_wait_lane, the SSD walk's hand-offs)
// it is a call.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < 1024u; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity);
}
__device__ __forceinline__ bool mbar_wait_lane(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < 1024u; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow_call(bar, parity);
}

// Waits for work this thread issued before the CTA exits: polls up to kWaitPolls whether
// or not the CTA has aborted (a copy or MMA still in flight must land before the shared
// and tensor memory it writes is released).  Counts a failure like mbar_wait.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
#pragma unroll 1
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicAdd(&g_ssm_wait_timeouts, 1u);
    return false;
}

// After an abort, by the thread that issued the copies of a ring of `stages` barriers:
// copy number j (0, 1, 2, ... in issue order) completed on bars[j % stages] in phase
// (j / stages) & 1, and `last` is the number of the last copy issued (-1: none).  Phases
// of one barrier complete in order, so the last `stages` copies are the ones to wait for.
__device__ __forceinline__ void drain_ring(uint64_t* bars, int stages, long long last) {
    for (long long j = last - stages + 1; j <= last; ++j)
        if (j >= 0) mbar_drain(&bars[j % stages], static_cast<uint32_t>((j / stages) & 1));
}

// mbar_wait polled by lane 0 alone; the other lanes wait at __syncwarp, which also makes
// what lane 0 observed visible to them.  Keeps a large CTA's waiting warps off the issue
// slots.  All 32 lanes must call it.  (A try_wait with a suspend-time hint measured
// slower here: the sleeping thread wakes late.)
__device__ __forceinline__ void mbar_wait_warp(uint64_t* bar, uint32_t parity) {
    if ((threadIdx.x & 31) == 0) mbar_wait_lane(bar, parity);
    __syncwarp();
}

// mbar_wait_warp that also tells the whole warp whether the wait succeeded (false: the CTA
// has aborted).  For the warps that issue copies or MMAs: they issue only after a wait
// that succeeded, so they need no separate read of the abort flag on their critical path.
__device__ __forceinline__ bool mbar_wait_warp_ok(uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_lane(bar, parity) ? 1 : 0;
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2-D tiled bulk tensor load: box at (x = inner element index, y = row) into smem,
// completion signalled on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of element (row, byte b within the row) in a tile written by TMA with
// CU_TENSOR_MAP_SWIZZLE_128B and 128-byte rows (tile base 1024-byte aligned): the
// 16-byte chunk index is XORed with row % 8.
__device__ __forceinline__ int sw128(int row, int byte_in_row) {
    return row * 128 + ((((byte_in_row >> 4) ^ (row & 7)) << 4) | (byte_in_row & 15));
}

}  // namespace ssm
