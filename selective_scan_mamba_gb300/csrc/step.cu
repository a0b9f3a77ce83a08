// step.cu -- single-step decode update (sm_103a), in place on the fp32 state.
//
// ("From S4 to Mamba-3", 03/System: the incremental step() used for decoding.)
// For every row (b, h, p) of the state [Bt, H, P, N]:
//   Delta    = softplus(dt[b,h] + bias[h])
//   h[n]    <- exp(Delta A) h[n] + w Delta-weighted x[p] B[n]    (A = A[h] or A[h, n])
//   y[p]     = (sum_n C[n] h[n] + D[h] x[p]) * SiLU(z[p])
// The step is bound by HBM traffic on the state (read once, written once).  A row of N
// floats is served by LPR = N / (4 NV) lanes, each holding NV float4 groups; a warp
// covers 32 / LPR rows at once, loads and stores are 16-byte and coalesced, and the
// row sum is a shuffle tree over the LPR lanes.  Every warp keeps UNROLL rows of loads
// in flight.  Other dstates take a scalar path (one thread per row).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

template <typename Tin>
__device__ __forceinline__ float step_delta(const StepArgs& a, int b, int hd) {
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const float v = to_f32(DT[static_cast<size_t>(b) * a.nheads + hd]) +
                    (a.dt_bias ? a.dt_bias[hd] : 0.f);
    return a.dt_softplus ? softplus_accurate(v) : v;
}

// Vector path.  A CTA owns kRowsPerCta consecutive state rows; its prologue computes, once
// per (batch, head) in that range, the step Delta, the decay exp(Delta A) and the input
// weight, plus the B/C offset, into shared memory (softplus and exp run once per head,
// not once per lane).  Each warp then streams rows: LPR lanes per row, NV float4 groups
// per lane, UNROLL rows of loads in flight, f32x2 arithmetic, a shuffle tree for y.
constexpr int kStepThreads = 256;

template <typename Tin, typename Tout, int NV, int LPR, int UNROLL, bool PER_STATE>
__global__ void __launch_bounds__(kStepThreads) step_vec(StepArgs a, int rows_per_cta,
                                                         int log2p) {
    constexpr int RPW = 32 / LPR;  // rows per warp per pass
    const int N = a.dstate;
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    const long long r0 = static_cast<long long>(blockIdx.x) * rows_per_cta;
    const long long r1 = min(rows, r0 + rows_per_cta);
    const int P = a.headdim;
    // (batch, head) range of this CTA
    const long long bh0 = log2p >= 0 ? (r0 >> log2p) : r0 / P;
    const long long bh1 = log2p >= 0 ? ((r1 - 1) >> log2p) : (r1 - 1) / P;
    const int nbh = static_cast<int>(bh1 - bh0 + 1);
    extern __shared__ float s_step[];
    float* s_dt = s_step;            // Delta
    float* s_da = s_dt + nbh;        // exp(Delta A_h)            (scalar-A form)
    float* s_w = s_da + nbh;         // input weight / Delta       (1 for exp-Euler)
    float* s_d = s_w + nbh;          // D_h
    int* s_bc = reinterpret_cast<int*>(s_d + nbh);  // B/C row offset (b * G + g) * N
    int* s_h = s_bc + nbh;                          // head index
    const int per_group = a.nheads / a.ngroups;
    const Tin* DT = static_cast<const Tin*>(a.dt);
    for (int i = threadIdx.x; i < nbh; i += blockDim.x) {
        const long long bh = bh0 + i;
        const int hd = static_cast<int>(bh % a.nheads);
        const int b = static_cast<int>(bh / a.nheads);
        const float v = to_f32(DT[bh]) + (a.dt_bias ? a.dt_bias[hd] : 0.f);
        const float dt = a.dt_softplus ? softplus_accurate(v) : v;
        s_dt[i] = dt;
        if (!PER_STATE) {
            const float za = dt * a.A[hd];
            s_da[i] = expf(za);
            s_w[i] = a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f;
        }
        s_d[i] = a.D ? a.D[hd] : 0.f;
        s_bc[i] = (b * a.ngroups + hd / per_group) * N;
        s_h[i] = hd;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, li = lane % LPR;
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);

    for (long long base = r0 + static_cast<long long>(warp) * RPW * UNROLL; base < r1;
         base += static_cast<long long>(nwarps) * RPW * UNROLL) {
        float4 hv[UNROLL][NV];
        long long rr[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            rr[u] = base + u * RPW + sub;
            if (rr[u] < r1) {
                const float4* sp = reinterpret_cast<const float4*>(a.state + rr[u] * N);
#pragma unroll
                for (int v = 0; v < NV; ++v) hv[u][v] = __ldcs(sp + li + v * LPR);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long r = rr[u] < r1 ? rr[u] : r1 - 1;
            const int i = static_cast<int>((log2p >= 0 ? (r >> log2p) : r / P) - bh0);
            const float dt = s_dt[i];
            const float xp = to_f32(X[r]);
            const float dx = dt * xp;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int n0 = 4 * (li + v * LPR);
                float bv[4], cv[4];
                load4_f32(Bp + s_bc[i] + n0, bv);
                load4_f32(Cp + s_bc[i] + n0, cv);
                float2 da01, da23;
                float wdx01, wdx23, wdx2, wdx3;
                if (PER_STATE) {
                    const float* Ah = a.A + static_cast<size_t>(s_h[i]) * N + n0;
                    float ww[4], dd[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float za = dt * Ah[j];
                        dd[j] = expf(za);
                        ww[j] = a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f;
                    }
                    da01 = make_float2(dd[0], dd[1]);
                    da23 = make_float2(dd[2], dd[3]);
                    wdx01 = ww[0] * dx;
                    wdx23 = ww[1] * dx;
                    wdx2 = ww[2] * dx;
                    wdx3 = ww[3] * dx;
                } else {
                    const float d = s_da[i];
                    da01 = da23 = make_float2(d, d);
                    wdx01 = wdx23 = wdx2 = wdx3 = s_w[i] * dx;
                }
                float2 h01 = make_float2(hv[u][v].x, hv[u][v].y);
                float2 h23 = make_float2(hv[u][v].z, hv[u][v].w);
                h01 = fma2(da01, h01, make_float2(wdx01 * bv[0], wdx23 * bv[1]));
                h23 = fma2(da23, h23, make_float2(wdx2 * bv[2], wdx3 * bv[3]));
                hv[u][v] = make_float4(h01.x, h01.y, h23.x, h23.y);
                acc = fma2(make_float2(cv[0], cv[1]), h01, acc);
                acc = fma2(make_float2(cv[2], cv[3]), h23, acc);
            }
            float sum = acc.x + acc.y;
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, off);  // xor < LPR stays in the row's lanes
            if (rr[u] < r1) {
                float4* sp = reinterpret_cast<float4*>(a.state + rr[u] * N);
#pragma unroll
                for (int v = 0; v < NV; ++v) __stcs(sp + li + v * LPR, hv[u][v]);
                if (li == 0) {
                    float yv = sum + s_d[i] * xp;
                    if (Z) yv *= silu_accurate(to_f32(Z[r]));
                    io<Tout>::store(static_cast<Tout*>(a.y), r, yv);
                }
            }
        }
    }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(128) step_scalar(StepArgs a) {
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int N = a.dstate;
    const int p = static_cast<int>(r % a.headdim);
    (void)p;
    const long long bh = r / a.headdim;
    const int hd = static_cast<int>(bh % a.nheads);
    const int b = static_cast<int>(bh / a.nheads);
    const int g = hd / (a.nheads / a.ngroups);
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const float dt = step_delta<Tin>(a, b, hd);
    const float xp = to_f32(X[r]);
    float acc = 0.f;
    float* hrow = a.state + r * N;
    for (int n = 0; n < N; ++n) {
        const size_t bc = (static_cast<size_t>(b) * a.ngroups + g) * N + n;
        const float av = a.a_per_state ? a.A[static_cast<size_t>(hd) * N + n] : a.A[hd];
        const float za = dt * av;
        const float w = a.disc == SSM_DISC_ZOH ? dt * phi1f(za) : dt;
        const float hn = expf(za) * hrow[n] + w * xp * to_f32(Bp[bc]);
        hrow[n] = hn;
        acc += to_f32(Cp[bc]) * hn;
    }
    float yv = acc + (a.D ? a.D[hd] : 0.f) * xp;
    if (Z) yv *= silu_accurate(to_f32(Z[r]));
    io<Tout>::store(static_cast<Tout*>(a.y), r, yv);
}

template <typename Tin, typename Tout, int NV, int LPR, int UNROLL>
static cudaError_t launch_vec(const StepArgs& a, long long rows, cudaStream_t s) {
    // rows per CTA: enough for every warp to run two passes of UNROLL rows
    const int rows_per_cta = (kStepThreads / 32) * (32 / LPR) * UNROLL * 2;
    const long long grid = (rows + rows_per_cta - 1) / rows_per_cta;
    int log2p = -1;
    if ((a.headdim & (a.headdim - 1)) == 0) {
        log2p = 0;
        while ((1 << log2p) < a.headdim) ++log2p;
    }
    // per-CTA (batch, head) table: at most rows_per_cta / headdim + 2 entries
    const int nbh_max = rows_per_cta / a.headdim + 2;
    const size_t smem = static_cast<size_t>(nbh_max) * 6 * sizeof(float);
    if (a.a_per_state)
        step_vec<Tin, Tout, NV, LPR, UNROLL, true>
            <<<static_cast<unsigned>(grid), kStepThreads, smem, s>>>(a, rows_per_cta, log2p);
    else
        step_vec<Tin, Tout, NV, LPR, UNROLL, false>
            <<<static_cast<unsigned>(grid), kStepThreads, smem, s>>>(a, rows_per_cta, log2p);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t launch_step_t(const StepArgs& a, cudaStream_t s) {
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    if (rows == 0) return cudaSuccess;
    switch (a.dstate) {
        case 16: return launch_vec<Tin, Tout, 1, 4, 4>(a, rows, s);
        case 32: return launch_vec<Tin, Tout, 1, 8, 4>(a, rows, s);
        case 64: return launch_vec<Tin, Tout, 1, 16, 4>(a, rows, s);
        case 128: return launch_vec<Tin, Tout, 1, 32, 4>(a, rows, s);
        case 256: return launch_vec<Tin, Tout, 2, 32, 4>(a, rows, s);
        default: {
            const unsigned blocks = static_cast<unsigned>((rows + 127) / 128);
            step_scalar<Tin, Tout><<<blocks, 128, 0, s>>>(a);
            return cudaGetLastError();
        }
    }
}

cudaError_t step_launch(const StepArgs& a, cudaStream_t s) {
    if (a.in_dtype == SSM_BF16)
        return a.out_dtype == SSM_BF16 ? launch_step_t<bf16_t, bf16_t>(a, s)
                                       : launch_step_t<bf16_t, float>(a, s);
    return a.out_dtype == SSM_BF16 ? launch_step_t<float, bf16_t>(a, s)
                                   : launch_step_t<float, float>(a, s);
}

}  // namespace ssm
