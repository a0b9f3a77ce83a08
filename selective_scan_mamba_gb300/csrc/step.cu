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

template <typename Tin, typename Tout, int NV, int LPR, int UNROLL>
__global__ void __launch_bounds__(256) step_vec(StepArgs a) {
    constexpr int RPW = 32 / LPR;  // rows per warp per pass
    const int N = a.dstate;
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, li = lane % LPR;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int per_group = a.nheads / a.ngroups;
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);

    for (long long base = warp * RPW * UNROLL; base < rows; base += nwarps * RPW * UNROLL) {
        float4 hv[UNROLL][NV];
        long long rr[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            rr[u] = base + u * RPW + sub;
            if (rr[u] < rows) {
                const float4* sp = reinterpret_cast<const float4*>(a.state + rr[u] * N);
#pragma unroll
                for (int v = 0; v < NV; ++v) hv[u][v] = sp[li + v * LPR];
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const long long r = rr[u] < rows ? rr[u] : rows - 1;
            const int p = static_cast<int>(r % a.headdim);
            const long long bh = r / a.headdim;
            const int hd = static_cast<int>(bh % a.nheads);
            const int b = static_cast<int>(bh / a.nheads);
            const int g = hd / per_group;
            const float dt = step_delta<Tin>(a, b, hd);
            const float xp = to_f32(X[r]);
            const float dx = dt * xp;
            // scalar-A form: one decay and one input weight for the whole row
            const float za_h = a.a_per_state ? 0.f : dt * a.A[hd];
            const float dA_h = a.a_per_state ? 0.f : expf(za_h);
            const float w_h = (a.a_per_state || a.disc != SSM_DISC_ZOH) ? 1.f : phi1f(za_h);
            float acc = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int n0 = 4 * (li + v * LPR);
                float bv[4], cv[4], av[4];
                const size_t bc = (static_cast<size_t>(b) * a.ngroups + g) * N + n0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    bv[j] = to_f32(Bp[bc + j]);
                    cv[j] = to_f32(Cp[bc + j]);
                }
                float* hp = &hv[u][v].x;
                if (a.a_per_state) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) av[j] = a.A[static_cast<size_t>(hd) * N + n0 + j];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float za = dt * av[j];
                        const float w = a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f;
                        hp[j] = expf(za) * hp[j] + (w * dx) * bv[j];
                        acc += cv[j] * hp[j];
                    }
                } else {
                    const float wdx = w_h * dx;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        hp[j] = dA_h * hp[j] + wdx * bv[j];
                        acc += cv[j] * hp[j];
                    }
                }
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);  // xor < LPR stays in the row's lanes
            if (rr[u] < rows) {
                float4* sp = reinterpret_cast<float4*>(a.state + rr[u] * N);
#pragma unroll
                for (int v = 0; v < NV; ++v) sp[li + v * LPR] = hv[u][v];
                if (li == 0) {
                    float yv = acc + (a.D ? a.D[hd] : 0.f) * xp;
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

template <typename Tin, typename Tout>
static cudaError_t launch_step_t(const StepArgs& a, cudaStream_t s) {
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    if (rows == 0) return cudaSuccess;
    const int N = a.dstate;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    auto grid_for = [&](int rows_per_warp_pass) {
        const long long warps_needed = (rows + rows_per_warp_pass - 1) / rows_per_warp_pass;
        long long blocks = (warps_needed + 7) / 8;
        const long long cap = static_cast<long long>(sms) * 16;
        return static_cast<unsigned>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
    };
    constexpr int U = 4;
    switch (N) {
        case 16:
            step_vec<Tin, Tout, 1, 4, U><<<grid_for(8 * U), 256, 0, s>>>(a);
            return cudaGetLastError();
        case 32:
            step_vec<Tin, Tout, 1, 8, U><<<grid_for(4 * U), 256, 0, s>>>(a);
            return cudaGetLastError();
        case 64:
            step_vec<Tin, Tout, 1, 16, U><<<grid_for(2 * U), 256, 0, s>>>(a);
            return cudaGetLastError();
        case 128:
            step_vec<Tin, Tout, 1, 32, U><<<grid_for(1 * U), 256, 0, s>>>(a);
            return cudaGetLastError();
        case 256:
            step_vec<Tin, Tout, 2, 32, U><<<grid_for(1 * U), 256, 0, s>>>(a);
            return cudaGetLastError();
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
