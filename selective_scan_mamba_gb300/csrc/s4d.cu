// s4d.cu -- S4D: linear time-invariant SSM with a complex diagonal A, exact ZOH.
//
// ("From S4 to Mamba-3", 03/System, s4_minimal.py; Likely questions Q01.)  Per channel d
// and state n, Delta = exp(log_dt[d]), z = Delta A[n]:
//   Abar = e^z,  Bbar = Delta B (e^z - 1)/z   (1 + z/2 + z^2/6 for |z| < 1e-4)
//   recurrent:   h_t = Abar h_{t-1} + Bbar u_t,  y_t = Re sum_n C h_t + D u_t
//   convolution: K_l = Re sum_n C Bbar Abar^l,  y = K * u + D u.
//
// Two kernels:
//   - s4d_scan runs the recurrent form (the O(1)-state form, equal to the convolution from
//     a zero state): a CTA of 128 threads owns 128 / TPC channels of one batch row, two
//     complex states per thread; Abar, Bbar and C sit in registers (Abar and Bbar computed
//     once per state in double precision, then rounded), u and y pass through shared
//     memory in 32-step chunks so that global accesses are coalesced rows; when that
//     leaves few CTAs the sequence is cut into segments (a states-only pass over all but
//     the last, then every segment from the state carried through the ones before it);
//   - s4d_kernel_gen writes the convolution kernel K [dim, L]: per channel the states'
//     C Bbar and z once, then per step l the sum of Re(C Bbar exp(l z)) with the phase
//     l Im z reduced modulo 2 pi in double precision (it reaches 1e5 rad at long L).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kST = 32;
constexpr int kSThreads = 128;
constexpr int kSS = 2;           // complex states per thread (more threads: L is sequential)
constexpr int kSRow = kST + 1;

// Abar = e^z and Bbar = Delta B phi1(z) for one state, in double precision
__device__ void s4d_disc(double dt, double ar, double ai, double br, double bi, double* abr,
                         double* abi, double* bbr, double* bbi) {
    const double zr = dt * ar, zi = dt * ai;
    const double ex = exp(zr);
    double sn, cs;
    sincos(zi, &sn, &cs);
    *abr = ex * cs;
    *abi = ex * sn;
    double pr, pi;
    if (sqrt(zr * zr + zi * zi) < 1e-4) {
        pr = 1.0 + zr / 2.0 + (zr * zr - zi * zi) / 6.0;
        pi = zi / 2.0 + (2.0 * zr * zi) / 6.0;
    } else {
        const double s2 = sin(zi / 2.0);
        const double nr = expm1(zr) * cs - 2.0 * s2 * s2;
        const double ni = ex * sn;
        const double den = zr * zr + zi * zi;
        pr = (nr * zr + ni * zi) / den;
        pi = (ni * zr - nr * zi) / den;
    }
    *bbr = dt * (br * pr - bi * pi);
    *bbi = dt * (br * pi + bi * pr);
}

// STATES: the segment pass of a time-split scan.  Segment `seg` covers steps
// [seg * seg_len, (seg + 1) * seg_len); this pass runs segments 0 .. nseg-2 from a zero
// state and writes their end states (no outputs).  The main pass starts segment seg from
// h0 carried through those: h <- Abar^seg_len h + h_end(j) for j < seg (Abar^seg_len in
// double precision).
template <typename Tin, typename Tout, int TPC, bool STATES>
__global__ void __launch_bounds__(kSThreads) s4d_scan(ssm_s4d_params a, int cps, int nseg, int seg_len,
                                                      float* seg_state) {
    constexpr int N = TPC * kSS;
    constexpr int CPB = kSThreads / TPC;
    const int Dm = a.dim;
    const int segs_here = STATES ? nseg - 1 : nseg;
    const int seg = blockIdx.x % segs_here;
    const int rest = blockIdx.x / segs_here;
    const int b = rest / cps, part_i = rest % cps;
    const int tbeg = seg * seg_len, tend = min(a.seqlen, tbeg + seg_len);
    const int L = a.seqlen;
    const int l0 = static_cast<int>((static_cast<long long>(part_i) * Dm) / cps);
    const int l1 = static_cast<int>((static_cast<long long>(part_i + 1) * Dm) / cps);
    const int nchan = l1 - l0;

    __shared__ float s_u[CPB * kSRow];
    __shared__ float s_y[CPB * kSRow];
    const int tid = threadIdx.x;
    const int c = tid / TPC, gi = tid % TPC;
    const bool active = c < nchan;
    const int d = l0 + (active ? c : 0);
    const size_t row = static_cast<size_t>(b) * Dm + d;

    float abr[kSS], abi[kSS], bbr[kSS], bbi[kSS], cr[kSS], ci[kSS], hr[kSS], hi[kSS];
    const double dt = exp(static_cast<double>(a.log_dt[d]));
    const size_t rows = static_cast<size_t>(a.batch) * Dm;
#pragma unroll
    for (int i = 0; i < kSS; ++i) {
        const size_t k = (static_cast<size_t>(d) * N + kSS * gi + i) * 2;
        double r0, r1, r2, r3;
        s4d_disc(dt, a.A[k], a.A[k + 1], a.B[k], a.B[k + 1], &r0, &r1, &r2, &r3);
        abr[i] = static_cast<float>(r0);
        abi[i] = static_cast<float>(r1);
        bbr[i] = static_cast<float>(r2);
        bbi[i] = static_cast<float>(r3);
        cr[i] = a.C[k];
        ci[i] = a.C[k + 1];
        const size_t hk = (row * N + kSS * gi + i) * 2;
        double h_r = (!STATES && active && a.h0) ? a.h0[hk] : 0.0;
        double h_i = (!STATES && active && a.h0) ? a.h0[hk + 1] : 0.0;
        if (!STATES && seg > 0) {
            // carry through the earlier segments: h <- Abar^seg_len h + h_end(j)
            const double zr = dt * a.A[k] * seg_len, zi = dt * a.A[k + 1] * seg_len;
            const double mag = exp(zr);
            double sn, cs;
            sincos(fmod(zi, 6.283185307179586), &sn, &cs);
            const double pr = mag * cs, pi = mag * sn;
            for (int j = 0; j < seg; ++j) {
                const float* hs = seg_state + ((j * rows + row) * N + kSS * gi + i) * 2;
                const double nr = pr * h_r - pi * h_i + hs[0];
                h_i = pr * h_i + pi * h_r + hs[1];
                h_r = nr;
            }
        }
        hr[i] = static_cast<float>(h_r);
        hi[i] = static_cast<float>(h_i);
    }
    const float Dd = a.D_skip ? a.D_skip[d] : 0.f;
    const Tin* U = static_cast<const Tin*>(a.u);

    // the next chunk's u is loaded into registers before the current chunk's recurrence
    // and stored to shared memory after it, so its latency hides behind the recurrence
    constexpr int KU = (CPB * kST + kSThreads - 1) / kSThreads;
    float r_u[KU];
    auto fetch = [&](int t0) {
        const int tl = min(kST, tend - t0);
#pragma unroll
        for (int k = 0; k < KU; ++k) {
            const int j = tid + k * kSThreads;
            const int cc = j / kST, t = j % kST;
            r_u[k] = (j < CPB * kST && cc < nchan && t < tl)
                         ? io<Tin>::load(U, (static_cast<size_t>(b) * Dm + l0 + cc) * L + t0 + t)
                         : 0.f;
        }
    };
    if (tbeg < tend) fetch(tbeg);
    for (int t0 = tbeg; t0 < tend; t0 += kST) {
        const int tl = min(kST, tend - t0);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KU; ++k) {
            const int j = tid + k * kSThreads;
            if (j < CPB * kST) s_u[(j / kST) * kSRow + j % kST] = r_u[k];
        }
        __syncthreads();
        if (t0 + kST < tend) fetch(t0 + kST);
        for (int t = 0; t < tl; ++t) {
            const float u = s_u[c * kSRow + t];
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kSS; ++i) {
                const float nr = fmaf(abr[i], hr[i], fmaf(-abi[i], hi[i], bbr[i] * u));
                hi[i] = fmaf(abr[i], hi[i], fmaf(abi[i], hr[i], bbi[i] * u));
                hr[i] = nr;
                if (!STATES) acc = fmaf(cr[i], hr[i], fmaf(-ci[i], hi[i], acc));
            }
            if (!STATES) {
#pragma unroll
                for (int off = 1; off < TPC; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (gi == 0) s_y[c * kSRow + t] = acc + Dd * u;
            }
        }
        if (STATES) continue;
        __syncthreads();
        for (int j = tid; j < CPB * kST; j += kSThreads) {
            const int cc = j / kST, t = j % kST;
            if (cc >= nchan || t >= tl) continue;
            io<Tout>::store(static_cast<Tout*>(a.y), (static_cast<size_t>(b) * Dm + l0 + cc) * L + t0 + t,
                            s_y[cc * kSRow + t]);
        }
    }
    if (STATES) {
        if (active) {
#pragma unroll
            for (int i = 0; i < kSS; ++i) {
                float* hs = seg_state + ((seg * rows + row) * N + kSS * gi + i) * 2;
                hs[0] = hr[i];
                hs[1] = hi[i];
            }
        }
    } else if (active && a.h_final && seg == nseg - 1) {
#pragma unroll
        for (int i = 0; i < kSS; ++i) {
            const size_t hk = (row * N + kSS * gi + i) * 2;
            a.h_final[hk] = hr[i];
            a.h_final[hk + 1] = hi[i];
        }
    }
}

// K[d, l] = Re sum_n C Bbar exp(l z).  One CTA per (channel, 1024 steps): the states'
// w = C Bbar and z are computed once (double precision) into shared memory; each thread
// then sums over the states for its steps, with |Abar^l| = exp(l Re z) and the phase
// l Im z reduced modulo 2 pi in double precision before the float sine and cosine.
constexpr int kKThreads = 256;
constexpr int kKSteps = 1024;

__global__ void __launch_bounds__(kKThreads) s4d_kernel_gen(ssm_s4d_params a, float* K, int L) {
    __shared__ float s_wr[64], s_wi[64], s_zr[64];
    __shared__ double s_zi[64];
    const int d = blockIdx.y;
    const int N = a.dstate;
    const double dt = exp(static_cast<double>(a.log_dt[d]));
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        const size_t k = (static_cast<size_t>(d) * N + n) * 2;
        double abr, abi, bbr, bbi;
        s4d_disc(dt, a.A[k], a.A[k + 1], a.B[k], a.B[k + 1], &abr, &abi, &bbr, &bbi);
        s_wr[n] = static_cast<float>(a.C[k] * bbr - a.C[k + 1] * bbi);
        s_wi[n] = static_cast<float>(a.C[k] * bbi + a.C[k + 1] * bbr);
        s_zr[n] = static_cast<float>(dt * a.A[k]);
        s_zi[n] = dt * a.A[k + 1];
    }
    __syncthreads();
    const double inv_two_pi = 0.15915494309189535, two_pi = 6.283185307179586;
    const int l_end = min(L, (blockIdx.x + 1) * kKSteps);
    for (int l = blockIdx.x * kKSteps + threadIdx.x; l < l_end; l += blockDim.x) {
        float acc = 0.f;
        for (int n = 0; n < N; ++n) {
            const double x = static_cast<double>(l) * s_zi[n];
            const float ph = static_cast<float>(x - two_pi * floor(x * inv_two_pi));
            float sn, cs;
            sincosf(ph, &sn, &cs);
            const float mag = expf(static_cast<float>(l) * s_zr[n]);
            acc += mag * (s_wr[n] * cs - s_wi[n] * sn);
        }
        K[static_cast<size_t>(d) * L + l] = acc;
    }
}

// Time split: with few channel blocks the sequence is cut into segments so that about
// four CTAs per SM run (measured: three segments 0.415 ms, eight 0.490 ms on the
// 8 x 256 x 32-state shape: the states-only pass grows with the count); each segment at least 256 steps and a whole number of chunks.
struct S4dPlan {
    int cps, nseg, seg_len;
    size_t ws_bytes;
};
S4dPlan s4d_plan(const ssm_s4d_params& a) {
    const int tpc = a.dstate / kSS;
    const int cpb = kSThreads / tpc;
    S4dPlan p;
    p.cps = (a.dim + cpb - 1) / cpb;
    const long long base = static_cast<long long>(a.batch) * p.cps;
    int sms = 148, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long want = (4LL * sms + base - 1) / base;
    const long long by_len = a.seqlen / 256;
    if (want > by_len) want = by_len;
    if (want > 64) want = 64;
    p.nseg = want < 1 ? 1 : static_cast<int>(want);
    const int chunks = (a.seqlen + kST - 1) / kST;
    p.seg_len = ((chunks + p.nseg - 1) / p.nseg) * kST;
    if (p.seg_len == 0) p.seg_len = kST;
    p.nseg = (a.seqlen + p.seg_len - 1) / p.seg_len;
    if (p.nseg < 1) p.nseg = 1;
    p.ws_bytes = static_cast<size_t>(p.nseg - 1) * a.batch * a.dim * a.dstate * 2 * sizeof(float);
    return p;
}

template <typename Tin, typename Tout, int TPC>
cudaError_t launch_s4d(const ssm_s4d_params& a, void* ws, cudaStream_t s) {
    const S4dPlan p = s4d_plan(a);
    float* seg_state = static_cast<float*>(ws);
    const int base = a.batch * p.cps;
    if (p.nseg > 1) {
        s4d_scan<Tin, Tout, TPC, true><<<base * (p.nseg - 1), kSThreads, 0, s>>>(a, p.cps, p.nseg, p.seg_len,
                                                                                 seg_state);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    s4d_scan<Tin, Tout, TPC, false><<<base * p.nseg, kSThreads, 0, s>>>(a, p.cps, p.nseg, p.seg_len, seg_state);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t dispatch_s4d(const ssm_s4d_params& a, void* ws, cudaStream_t s) {
    switch (a.dstate) {
        case 4: return launch_s4d<Tin, Tout, 4 / kSS>(a, ws, s);
        case 8: return launch_s4d<Tin, Tout, 8 / kSS>(a, ws, s);
        case 16: return launch_s4d<Tin, Tout, 16 / kSS>(a, ws, s);
        case 32: return launch_s4d<Tin, Tout, 32 / kSS>(a, ws, s);
        case 64: return launch_s4d<Tin, Tout, 64 / kSS>(a, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool s4d_supported(int dstate) {
    return dstate == 4 || dstate == 8 || dstate == 16 || dstate == 32 || dstate == 64;
}

size_t s4d_workspace_size(const ssm_s4d_params& a) {
    if (a.seqlen <= 0) return 0;
    return s4d_plan(a).ws_bytes;
}

cudaError_t s4d_launch(const ssm_s4d_params& a, void* workspace, cudaStream_t s) {
    const bool ib = a.in_dtype == SSM_BF16, ob = a.out_dtype == SSM_BF16;
    if (ib && ob) return dispatch_s4d<bf16_t, bf16_t>(a, workspace, s);
    if (ib) return dispatch_s4d<bf16_t, float>(a, workspace, s);
    if (ob) return dispatch_s4d<float, bf16_t>(a, workspace, s);
    return dispatch_s4d<float, float>(a, workspace, s);
}

cudaError_t s4d_kernel_launch(const ssm_s4d_params& a, float* K, int L, cudaStream_t s) {
    if (L == 0) return cudaSuccess;
    const dim3 grid((L + kKSteps - 1) / kKSteps, a.dim);
    s4d_kernel_gen<<<grid, kKThreads, 0, s>>>(a, K, L);
    return cudaGetLastError();
}

}  // namespace ssm
