// common.cuh -- small device helpers shared by the scan kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssmscan.h"

#define SSM_LOG2E 1.4426950408889634f
#define SSM_LN2 0.6931471805599453f

namespace ssm {

// ---------------------------------------------------------------------------------------
// storage types
// ---------------------------------------------------------------------------------------
struct bf16_t {
    uint16_t bits;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// round to nearest, ties to even (inputs are finite)
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}
// two floats -> packed bf16x2 (low half = a), round to nearest even, via the hardware cvt
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
struct io;
template <>
struct io<float> {
    static __device__ __forceinline__ float load(const float* p, size_t i) { return __ldg(p + i); }
    static __device__ __forceinline__ void store(float* p, size_t i, float v) { p[i] = v; }
    static constexpr int bytes = 4;
};
template <>
struct io<bf16_t> {
    static __device__ __forceinline__ float load(const bf16_t* p, size_t i) {
        return bf16_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
    }
    static __device__ __forceinline__ void store(bf16_t* p, size_t i, float v) {
        reinterpret_cast<uint16_t*>(p)[i] = f32_to_bf16(v);
    }
    static constexpr int bytes = 2;
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16_t v) { return bf16_to_f32(v.bits); }

// CNT consecutive elements from 16-byte aligned shared (or global) memory, widened to fp32
template <int CNT>
__device__ __forceinline__ void load_f32(const float* p, float* out) {
    static_assert(CNT % 4 == 0, "");
#pragma unroll
    for (int i = 0; i < CNT / 4; ++i) {
        const float4 v = reinterpret_cast<const float4*>(p)[i];
        out[4 * i] = v.x;
        out[4 * i + 1] = v.y;
        out[4 * i + 2] = v.z;
        out[4 * i + 3] = v.w;
    }
}
template <int CNT>
__device__ __forceinline__ void load_f32(const bf16_t* p, float* out) {
    static_assert(CNT % 8 == 0, "");
#pragma unroll
    for (int i = 0; i < CNT / 8; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            out[8 * i + 2 * j] = lo_bf16(w[j]);
            out[8 * i + 2 * j + 1] = hi_bf16(w[j]);
        }
    }
}

// 4 consecutive elements (8-byte aligned for bf16, 16-byte for fp32), widened to fp32
__device__ __forceinline__ void load4_f32(const float* p, float* out) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x;
    out[1] = v.y;
    out[2] = v.z;
    out[3] = v.w;
}
__device__ __forceinline__ void load4_f32(const bf16_t* p, float* out) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    out[0] = lo_bf16(v.x);
    out[1] = hi_bf16(v.x);
    out[2] = lo_bf16(v.y);
    out[3] = hi_bf16(v.y);
}

// Store CNT consecutive outputs; `room` = how many of them lie inside the row.  Whole
// rows go out as 16-byte vectors (the destination is 16-byte aligned then), ragged
// ends element by element.
template <typename Tout, int CNT>
__device__ __forceinline__ void store_row(Tout* dst, const float* v, int room);
template <int CNT>
__device__ __forceinline__ void store_row(float* dst, const float* v, int room) {
    if (room >= CNT) {
#pragma unroll
        for (int i = 0; i < CNT / 4; ++i)
            reinterpret_cast<float4*>(dst)[i] =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < CNT; ++i)
            if (i < room) dst[i] = v[i];
    }
}
template <int CNT>
__device__ __forceinline__ void store_row(bf16_t* dst, const float* v, int room) {
    if (room >= CNT) {
#pragma unroll
        for (int i = 0; i < CNT / 8; ++i)
            reinterpret_cast<uint4*>(dst)[i] =
                make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                           pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                           pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    } else {
#pragma unroll
        for (int i = 0; i < CNT; ++i)
            if (i < room) reinterpret_cast<uint16_t*>(dst)[i] = f32_to_bf16(v[i]);
    }
}

// ---------------------------------------------------------------------------------------
// math: fast hardware approximations (MUFU) and the accurate library routines
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v).  Accurate variant: library log1pf/expf.  For v > 20
// the result equals v to within 2.1e-9 absolute.
__device__ __forceinline__ float softplus_accurate(float v) {
    return v > 20.f ? v : log1pf(expf(v));
}
// Fast variant for bfloat16 inputs, by the identity softplus(v) = max(v, 0) +
// log(1 + e^-|v|): MUFU.EX2 of -|v|, MUFU.LG2 of 1 + that, one FMA; no branches, so
// independent evaluations interleave.  The absolute error is ~1e-7 (lg2.approx near 1
// and the rounding of 1 + e^-|v|); where softplus(v) < 1e-6 (v < -14) the result may be
// 0, which changes Delta, e^(Delta A) and Delta B x by less than 1e-6 absolute.
__device__ __forceinline__ float softplus_fast(float v) {
    const float t = ex2_approx(-fabsf(v) * SSM_LOG2E);
    return fmaf(lg2_approx(1.f + t), SSM_LN2, fmaxf(v, 0.f));
}
__device__ __forceinline__ float silu_accurate(float v) { return v / (1.f + expf(-v)); }
__device__ __forceinline__ float silu_fast(float v) {
    return v * rcp_approx(1.f + ex2_approx(-v * SSM_LOG2E));
}

// (e^z - 1)/z for the ZOH input weight, with expm1f for accuracy near z = 0
__device__ __forceinline__ float phi1f(float zz) {
    return fabsf(zz) < 1e-7f ? 1.f + 0.5f * zz : expm1f(zz) / zz;
}

// ---------------------------------------------------------------------------------------
// packed float32x2 arithmetic (sm_100+): one instruction, two lanes of work
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched by launch_dependent() may start while
// the kernel before it in the stream is still running: it calls grid_dep_wait() before it
// reads what that kernel writes or writes what it reads (the wait returns once the earlier
// grid has completed and its writes are visible).  grid_dep_launch() lets the next such
// kernel be scheduled before this one ends.  Both do nothing in an ordinary launch.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------------------
// asynchronous global->shared copies (16 bytes, zero-filled past src_bytes)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace ssm
