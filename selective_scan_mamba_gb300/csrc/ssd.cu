// ssd.cu -- Mamba-2 chunked SSD scan (sm_103a), CUDA-core version.
//
// ("From S4 to Mamba-3", 03/System, mamba2_minimal.py: with a scalar A per head the
// recurrence becomes chunked decayed-attention matmuls with a carried (N, P) state;
// 04/Approach: the result must equal the sequential scan for any chunk size.)
//
// With Q-step chunks and, inside chunk c, s_t = sum of Delta*A_h over the chunk up to
// and including step t:
//   K2a  chunk state    S_c[p,n] = sum_s exp(s_end - s_s) w_s x_s[p] B_s[n]
//   K2b  state passing  h_in(c)  = exp(s_end(c-1)) h_in(c-1) + S_{c-1},  h_in(0) = h0
//   K2c  chunk output   y_t[p]   = sum_{s<=t} (C_t.B_s) exp(s_t - s_s) w_s x_s[p]
//                                  + exp(s_t) C_t . h_in(c)[p, :] + D_h x_t[p], gated
// w_s = Delta_s (exp-Euler) or Delta_s (e^z - 1)/z with z = Delta_s A_h (ZOH).
// The chunk states live in the caller's workspace; K2b overwrites each S_c with the
// state entering chunk c.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

constexpr int kSsdThreads = 256;
constexpr int kSub = 32;  // sub-tile of steps staged in shared memory

// Delta, running sum of Delta*A and input weight of one chunk, into shared memory.
// Every thread of the block must call it.
template <typename Tin>
__device__ void ssd_chunk_prep(const SsdArgs& a, int b, int hd, int t0, int q, float* cum,
                               float* wts, float* scratch) {
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const float Ah = a.A[hd];
    const float bias = a.dt_bias ? a.dt_bias[hd] : 0.f;
    for (int i = threadIdx.x; i < a.chunk; i += blockDim.x) {
        float dt = 0.f;
        if (i < q) {
            const float v =
                to_f32(DT[(static_cast<size_t>(b) * a.seqlen + t0 + i) * a.nheads + hd]) + bias;
            dt = a.dt_softplus ? softplus_accurate(v) : v;
        }
        scratch[i] = dt * Ah;
        wts[i] = a.disc == SSM_DISC_ZOH ? dt * phi1f(dt * Ah) : dt;
    }
    __syncthreads();
    // inclusive prefix sum (Hillis-Steele, ping-pong between scratch and cum)
    float* src = scratch;
    float* dst = cum;
    for (int off = 1; off < a.chunk; off <<= 1) {
        for (int i = threadIdx.x; i < a.chunk; i += blockDim.x)
            dst[i] = src[i] + (i >= off ? src[i - off] : 0.f);
        __syncthreads();
        float* tmp = src;
        src = dst;
        dst = tmp;
    }
    if (src != cum) {
        for (int i = threadIdx.x; i < a.chunk; i += blockDim.x) cum[i] = src[i];
        __syncthreads();
    }
}

// ---- K2a: chunk states --------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_state(SsdArgs a) {
    const int c = blockIdx.x, hd = blockIdx.y, b = blockIdx.z;
    const int P = a.headdim, N = a.dstate, Q = a.chunk;
    const int nch = (a.seqlen + Q - 1) / Q;
    const int t0 = c * Q;
    const int q = min(Q, a.seqlen - t0);
    const int g = hd / (a.nheads / a.ngroups);
    extern __shared__ float sm[];
    float* cum = sm;
    float* wts = cum + Q;
    float* scr = wts + Q;
    float* xs = scr + Q;           // [kSub][P]
    float* bs = xs + kSub * P;     // [kSub][N]
    ssd_chunk_prep<Tin>(a, b, hd, t0, q, cum, wts, scr);
    const float cend = cum[q - 1];
    constexpr int MAXJ = 32;       // P*N / threads <= 32 (P*N <= 8192)
    const int per = (P * N) / kSsdThreads;
    float acc[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) acc[j] = 0.f;
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    for (int s0 = 0; s0 < q; s0 += kSub) {
        for (int i = threadIdx.x; i < kSub * P; i += blockDim.x) {
            const int si = i / P, p = i % P, s = s0 + si;
            float v = 0.f;
            if (s < q)
                v = to_f32(X[((static_cast<size_t>(b) * a.seqlen + t0 + s) * a.nheads + hd) * P + p]) *
                    wts[s] * expf(cend - cum[s]);
            xs[i] = v;
        }
        for (int i = threadIdx.x; i < kSub * N; i += blockDim.x) {
            const int si = i / N, n = i % N, s = s0 + si;
            bs[i] = s < q ? to_f32(Bp[((static_cast<size_t>(b) * a.seqlen + t0 + s) * a.ngroups + g) * N + n])
                          : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
            if (j < per) {
                const int idx = threadIdx.x + j * kSsdThreads;
                const int p = idx / N, n = idx % N;
                float s_ = acc[j];
                for (int si = 0; si < kSub; ++si) s_ += xs[si * P + p] * bs[si * N + n];
                acc[j] = s_;
            }
        }
        __syncthreads();
    }
    float* S = a.ws_states + ((static_cast<size_t>(b) * a.nheads + hd) * nch + c) * P * N;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j)
        if (j < per) S[threadIdx.x + j * kSsdThreads] = acc[j];
    if (threadIdx.x == 0)
        a.ws_decay[(static_cast<size_t>(b) * a.nheads + hd) * nch + c] = expf(cend);
}

// ---- K2b: state passing (sequential over chunks, parallel over (b, h, p, n)) ------------
__global__ void __launch_bounds__(kSsdThreads) ssd_state_pass(SsdArgs a) {
    const int hd = blockIdx.y, b = blockIdx.z;
    const int PN = a.headdim * a.dstate;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= PN) return;
    const int nch = (a.seqlen + a.chunk - 1) / a.chunk;
    const size_t bh = static_cast<size_t>(b) * a.nheads + hd;
    float h = a.h0 ? a.h0[bh * PN + e] : 0.f;
    float* S = a.ws_states + bh * nch * PN + e;
    const float* dec = a.ws_decay + bh * nch;
    for (int c = 0; c < nch; ++c) {
        const float sc = S[static_cast<size_t>(c) * PN];
        S[static_cast<size_t>(c) * PN] = h;  // state entering chunk c
        h = dec[c] * h + sc;
    }
    if (a.h_final) a.h_final[bh * PN + e] = h;
}

// ---- K2c: chunk outputs -------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_out(SsdArgs a) {
    const int c = blockIdx.x, hd = blockIdx.y, b = blockIdx.z;
    const int P = a.headdim, N = a.dstate, Q = a.chunk;
    const int nch = (a.seqlen + Q - 1) / Q;
    const int t0 = c * Q;
    const int q = min(Q, a.seqlen - t0);
    const int g = hd / (a.nheads / a.ngroups);
    extern __shared__ float sm[];
    float* cum = sm;
    float* wts = cum + Q;
    float* scr = wts + Q;
    float* hin = scr + Q;                  // [P][N+1]
    float* cs = hin + P * (N + 1);         // [kSub][N]
    float* bs = cs + kSub * N;             // [kSub][N+1]
    float* xs = bs + kSub * (N + 1);       // [kSub][P]
    float* M = xs + kSub * P;              // [kSub][kSub]
    ssd_chunk_prep<Tin>(a, b, hd, t0, q, cum, wts, scr);
    const float* Hin = a.ws_states + ((static_cast<size_t>(b) * a.nheads + hd) * nch + c) * P * N;
    for (int i = threadIdx.x; i < P * N; i += blockDim.x) hin[(i / N) * (N + 1) + i % N] = Hin[i];
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const float Dh = a.D ? a.D[hd] : 0.f;
    constexpr int MAXJ = 16;               // kSub * P / threads <= 16 (P <= 128)
    const int per = (kSub * P) / kSsdThreads;
    __syncthreads();
    for (int ts = 0; ts < q; ts += kSub) {
        for (int i = threadIdx.x; i < kSub * N; i += blockDim.x) {
            const int ti = i / N, n = i % N, t = ts + ti;
            cs[i] = t < q ? to_f32(Cp[((static_cast<size_t>(b) * a.seqlen + t0 + t) * a.ngroups + g) * N + n])
                          : 0.f;
        }
        float acc[MAXJ];
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) acc[j] = 0.f;
        for (int s0 = 0; s0 <= ts; s0 += kSub) {
            __syncthreads();
            for (int i = threadIdx.x; i < kSub * N; i += blockDim.x) {
                const int si = i / N, n = i % N, s = s0 + si;
                bs[si * (N + 1) + n] =
                    s < q ? to_f32(Bp[((static_cast<size_t>(b) * a.seqlen + t0 + s) * a.ngroups + g) * N + n])
                          : 0.f;
            }
            for (int i = threadIdx.x; i < kSub * P; i += blockDim.x) {
                const int si = i / P, p = i % P, s = s0 + si;
                xs[i] = s < q ? to_f32(X[((static_cast<size_t>(b) * a.seqlen + t0 + s) * a.nheads + hd) * P + p])
                              : 0.f;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kSub * kSub; e += blockDim.x) {
                const int ti = e / kSub, si = e % kSub;
                const int t = ts + ti, s = s0 + si;
                float m = 0.f;
                if (s <= t && t < q) {
                    float dot = 0.f;
                    for (int n = 0; n < N; ++n) dot += cs[ti * N + n] * bs[si * (N + 1) + n];
                    m = dot * expf(cum[t] - cum[s]) * wts[s];
                }
                M[e] = m;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < MAXJ; ++j) {
                if (j < per) {
                    const int idx = threadIdx.x + j * kSsdThreads;
                    const int ti = idx / P, p = idx % P;
                    float s_ = acc[j];
                    for (int si = 0; si < kSub; ++si) s_ += M[ti * kSub + si] * xs[si * P + p];
                    acc[j] = s_;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
            if (j < per) {
                const int idx = threadIdx.x + j * kSsdThreads;
                const int ti = idx / P, p = idx % P, t = ts + ti;
                if (t < q) {
                    float dot = 0.f;
                    for (int n = 0; n < N; ++n) dot += cs[ti * N + n] * hin[p * (N + 1) + n];
                    const size_t yi = ((static_cast<size_t>(b) * a.seqlen + t0 + t) * a.nheads + hd) * P + p;
                    float v = acc[j] + expf(cum[t]) * dot + Dh * to_f32(X[yi]);
                    if (Z) v *= silu_accurate(to_f32(Z[yi]));
                    io<Tout>::store(static_cast<Tout*>(a.y), yi, v);
                }
            }
        }
        __syncthreads();
    }
}

static size_t ssd_cuda_core_workspace_bytes(const SsdArgs& a) {
    const size_t nch = (static_cast<size_t>(a.seqlen) + a.chunk - 1) / a.chunk;
    const size_t states =
        static_cast<size_t>(a.batch) * a.nheads * nch * a.headdim * a.dstate * sizeof(float);
    const size_t decay = static_cast<size_t>(a.batch) * a.nheads * nch * sizeof(float);
    return ((states + 255) / 256) * 256 + ((decay + 255) / 256) * 256;
}

size_t ssd_workspace_bytes(const SsdArgs& a) {
    return ssd_tc_supported(a) ? ssd_tc_workspace_bytes(a) : ssd_cuda_core_workspace_bytes(a);
}

template <typename Tin, typename Tout>
static cudaError_t ssd_launch_t(const SsdArgs& a, cudaStream_t s) {
    const int Q = a.chunk, P = a.headdim, N = a.dstate;
    const int nch = (a.seqlen + Q - 1) / Q;
    if (nch > 0) {
        const dim3 grid(nch, a.nheads, a.batch);
        const size_t sm_a = (3 * Q + kSub * P + kSub * N) * sizeof(float);
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(ssd_chunk_state<Tin>), static_cast<int>(sm_a));
        if (e != cudaSuccess) return e;
        ssd_chunk_state<Tin><<<grid, kSsdThreads, sm_a, s>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const dim3 gpass((P * N + kSsdThreads - 1) / kSsdThreads, a.nheads, a.batch);
    ssd_state_pass<<<gpass, kSsdThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nch == 0) return e;
    const size_t sm_c = (3 * Q + P * (N + 1) + kSub * N + kSub * (N + 1) + kSub * P + kSub * kSub) *
                        sizeof(float);
    e = set_smem_attr(reinterpret_cast<const void*>(ssd_chunk_out<Tin, Tout>), static_cast<int>(sm_c));
    if (e != cudaSuccess) return e;
    ssd_chunk_out<Tin, Tout><<<dim3(nch, a.nheads, a.batch), kSsdThreads, sm_c, s>>>(a);
    return cudaGetLastError();
}

cudaError_t ssd_launch(const SsdArgs& a, cudaStream_t s) {
    if (ssd_tc_supported(a)) return ssd_tc_launch(a, a.ws_states, s);
    if (a.in_dtype == SSM_BF16)
        return a.out_dtype == SSM_BF16 ? ssd_launch_t<bf16_t, bf16_t>(a, s)
                                       : ssd_launch_t<bf16_t, float>(a, s);
    return a.out_dtype == SSM_BF16 ? ssd_launch_t<float, bf16_t>(a, s)
                                   : ssd_launch_t<float, float>(a, s);
}

}  // namespace ssm
