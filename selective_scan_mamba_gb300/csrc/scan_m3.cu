// scan_m3.cu -- Mamba-3 scan: complex diagonal transition, exponential-trapezoidal rule.
//
// ("From S4 to Mamba-3", 03/System, mamba3_minimal.py; 04/Approach, "Complex transitions
// for state tracking".)  Per channel d and state n, A = A_re + i A_im (A_re < 0):
//   Abar_t = exp(Delta_t A)
//   h_t    = Abar_t (h_{t-1} + (1 - lambda_t) Delta_t B_{t-1} x_{t-1}) + lambda_t Delta_t B_t x_t
//   y_t    = (Re sum_n C_t h_t + D x_t) SiLU(z_t)
// which is the exponential-Euler Mamba-1 scan at lambda = 1, A_im = 0.
//
// A CTA of 128 threads owns 128 / TPC channels of one (batch, group) (TPC threads per
// channel, four complex states per thread, in registers for the whole sequence).  Per
// 32-step chunk the CTA stages in shared memory, per (channel, step), Delta, the two input
// weights p_t = (1 - lambda_t) Delta_t x_{t-1} and q_t = lambda_t Delta_t x_t, x and the
// gate, and the B rows t0-1 .. t0+31 and C rows of the group; the recurrence then reads
// shared memory only, sums Re(C h) over the channel's threads with shuffles, and the
// chunk's outputs leave in coalesced rows.  When that leaves few CTAs, the sequence is
// cut into time segments (a states-only pass over all but the last, then every segment
// from the state carried through the ones before it).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kMT = 32;          // steps per chunk
constexpr int kMThreads = 128;
constexpr int kMS = 4;           // complex states per thread
constexpr int kMRow = kMT + 1;

struct M3Layout {  // float offsets
    int dl, p, q, x, gate, y, bs, cs, total;
    __host__ __device__ M3Layout(int cpb, int n) {
        dl = 0;                      // [cpb][kMRow] Delta
        p = dl + cpb * kMRow;        // (1 - lambda) Delta x_{t-1}
        q = p + cpb * kMRow;         // lambda Delta x_t
        x = q + cpb * kMRow;         // x
        gate = x + cpb * kMRow;      // SiLU(z) or 1
        y = gate + cpb * kMRow;      // outputs
        bs = y + cpb * kMRow;        // [kMT + 1][n] B rows t0-1 .. t0+kMT-1
        cs = bs + (kMT + 1) * n;     // [kMT][n] C rows
        total = cs + kMT * n;
    }
};

// sin and cos of x: Cody-Waite reduction to r = x - k 2pi with 2pi split into a float
// head and its tail (2pi - head, -1.748455531e-7), then the MUFU forms on |r| <= pi
// (absolute error ~4e-7 there).  Exact for |x| well below 2^10.
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
    const float k = rintf(x * 0.15915494309189535f);
    float r = fmaf(-k, 6.2831854820251465f, x);
    r = fmaf(-k, -1.7484555314695172e-7f, r);
    __sincosf(r, s, c);
}

// STATES: the segment pass of a time-split scan.  Segment `seg` covers steps
// [seg * seg_len, (seg + 1) * seg_len); this pass runs segments 0 .. nseg-2 from a zero
// state and writes their end states and sums of Delta (no outputs).  The main pass starts
// segment seg from h0 carried through those: h <- exp(A sum Delta_j) h + h_end(j).  The
// trapezoid's left-end term at a segment's first step reads x and B of the step before,
// so each segment (in both passes) adds it as an input from a zero-state start.
template <typename Tin, typename Tout, int TPC, bool STATES>
__global__ void __launch_bounds__(kMThreads) m3_scan(ssm_mamba3_params a, int cps, int nseg, int seg_len,
                                                     float* seg_state, float* seg_dsum) {
    constexpr int N = TPC * kMS;
    constexpr int CPB = kMThreads / TPC;
    const int L = a.seqlen, Dm = a.dim, G = a.ngroups;
    const int per_group = Dm / G;
    const int segs_here = STATES ? nseg - 1 : nseg;
    const int seg = blockIdx.x % segs_here;
    const int rest = blockIdx.x / segs_here;
    const int tbeg = seg * seg_len, tend = min(L, tbeg + seg_len);
    const int pair = rest / cps, part_i = rest % cps;
    const int b = pair / G, g = pair % G;
    const int l0 = static_cast<int>((static_cast<long long>(part_i) * per_group) / cps);
    const int l1 = static_cast<int>((static_cast<long long>(part_i + 1) * per_group) / cps);
    const int nchan = l1 - l0;
    const int d0 = g * per_group + l0;

    extern __shared__ __align__(16) float sm[];
    const M3Layout lay(CPB, N);
    const int tid = threadIdx.x;
    const int c = tid / TPC, gi = tid % TPC;
    const bool active = c < nchan;
    const int d = d0 + (active ? c : 0);
    const size_t row = static_cast<size_t>(b) * Dm + d;
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* DL = static_cast<const Tin*>(a.delta);
    const Tin* LM = static_cast<const Tin*>(a.lam);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const size_t bc_base = (static_cast<size_t>(b) * G + g) * N * static_cast<size_t>(L);

    const size_t rows = static_cast<size_t>(a.batch) * Dm;
    float are2[kMS], aim[kMS], hr[kMS], hi[kMS];
#pragma unroll
    for (int i = 0; i < kMS; ++i) {
        const size_t k = static_cast<size_t>(d) * N + kMS * gi + i;
        are2[i] = a.A_re[k] * SSM_LOG2E;
        aim[i] = a.A_im[k];
        const size_t hk = (row * N + kMS * gi + i) * 2;
        hr[i] = (!STATES && active && a.h0) ? a.h0[hk] : 0.f;
        hi[i] = (!STATES && active && a.h0) ? a.h0[hk + 1] : 0.f;
        if (!STATES && active) {
            // carry through the earlier segments: h <- exp(A sum Delta_j) h + h_end(j)
            for (int j = 0; j < seg; ++j) {
                const float ds = seg_dsum[j * rows + row];
                const float mag = expf(a.A_re[k] * ds);
                float sn, cs;
                sincosf(aim[i] * ds, &sn, &cs);
                const float ar = mag * cs, ai = mag * sn;
                const float* hs = seg_state + ((j * rows + row) * N + kMS * gi + i) * 2;
                const float nr = ar * hr[i] - ai * hi[i] + hs[0];
                hi[i] = ar * hi[i] + ai * hr[i] + hs[1];
                hr[i] = nr;
            }
        }
    }
    const float Dd = a.D_skip ? a.D_skip[d] : 0.f;
    float dsum = 0.f;  // sum of Delta over the segment (segment pass)

    // Prefetch: the next chunk's inputs are loaded into registers before the current
    // chunk's recurrence runs and written to shared memory after it, so the loads' latency
    // hides behind the recurrence (for TPC >= 4, where a thread stages at most 8
    // (channel, step) cells and a few B, C values).
    constexpr int KS = (CPB * kMT + kMThreads - 1) / kMThreads;
    constexpr int KB = (N * (kMT + 1) + kMThreads - 1) / kMThreads;
    constexpr bool PREF = KS <= 8;
    constexpr int RS = PREF ? KS : 1, RB = PREF ? KB : 1;
    float r_dl[RS], r_lm[RS], r_x[RS], r_xp[RS], r_z[RS], r_b[RB], r_c[RB];
    auto fetch = [&](int t0) {
        const int tl = min(kMT, tend - t0);
#pragma unroll
        for (int k = 0; k < RS; ++k) {
            const int j = tid + k * kMThreads;
            const int cc = j / kMT, t = j % kMT;
            r_dl[k] = r_lm[k] = r_x[k] = r_xp[k] = r_z[k] = 0.f;
            if (j < CPB * kMT && cc < nchan && t < tl) {
                const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
                r_dl[k] = io<Tin>::load(DL, i) + (a.delta_bias ? a.delta_bias[d0 + cc] : 0.f);
                r_lm[k] = io<Tin>::load(LM, i);
                r_x[k] = io<Tin>::load(X, i);
                r_xp[k] = (t0 + t > 0) ? io<Tin>::load(X, i - 1) : 0.f;
                if (Z) r_z[k] = io<Tin>::load(Z, i);
            }
        }
#pragma unroll
        for (int k = 0; k < RB; ++k) {
            const int j = tid + k * kMThreads;
            const int n = j / (kMT + 1), tt = j % (kMT + 1);  // B row t0 - 1 + tt
            const int t = t0 - 1 + tt;
            r_b[k] = r_c[k] = 0.f;
            if (j < N * (kMT + 1)) {
                if (t >= 0 && tt <= tl) r_b[k] = io<Tin>::load(Bp, bc_base + static_cast<size_t>(n) * L + t);
                if (tt < tl) r_c[k] = io<Tin>::load(Cp, bc_base + static_cast<size_t>(n) * L + t0 + tt);
            }
        }
    };
    auto put = [&](int t0) {
        const int tl = min(kMT, tend - t0);
#pragma unroll
        for (int k = 0; k < RS; ++k) {
            const int j = tid + k * kMThreads;
            if (j >= CPB * kMT) continue;
            const int cc = j / kMT, t = j % kMT;
            float dl = 0.f, p = 0.f, q = 0.f, xv = 0.f, gv = 1.f;
            if (cc < nchan && t < tl) {
                dl = a.delta_softplus ? softplus_accurate(r_dl[k]) : r_dl[k];
                xv = r_x[k];
                p = (1.f - r_lm[k]) * dl * r_xp[k];
                q = r_lm[k] * dl * xv;
                if (Z) gv = silu_accurate(r_z[k]);
            }
            sm[lay.dl + cc * kMRow + t] = dl;
            sm[lay.p + cc * kMRow + t] = p;
            sm[lay.q + cc * kMRow + t] = q;
            sm[lay.x + cc * kMRow + t] = xv;
            sm[lay.gate + cc * kMRow + t] = gv;
        }
#pragma unroll
        for (int k = 0; k < RB; ++k) {
            const int j = tid + k * kMThreads;
            if (j >= N * (kMT + 1)) continue;
            const int n = j / (kMT + 1), tt = j % (kMT + 1);
            sm[lay.bs + tt * N + n] = r_b[k];
            if (tt < kMT) sm[lay.cs + tt * N + n] = r_c[k];
        }
    };
    if (PREF && tbeg < tend) fetch(tbeg);

    for (int t0 = tbeg; t0 < tend; t0 += kMT) {
        const int tl = min(kMT, tend - t0);
        __syncthreads();  // the previous chunk's tiles and outputs are done with
        if constexpr (PREF) {
            put(t0);
        } else {
        for (int j = tid; j < CPB * kMT; j += kMThreads) {
            const int cc = j / kMT, t = j % kMT;
            float dl = 0.f, p = 0.f, q = 0.f, xv = 0.f, gv = 1.f;
            if (cc < nchan && t < tl) {
                const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
                const float v = io<Tin>::load(DL, i) + (a.delta_bias ? a.delta_bias[d0 + cc] : 0.f);
                dl = a.delta_softplus ? softplus_accurate(v) : v;
                const float lm = io<Tin>::load(LM, i);
                xv = io<Tin>::load(X, i);
                const float xp = (t0 + t > 0) ? io<Tin>::load(X, i - 1) : 0.f;
                p = (1.f - lm) * dl * xp;
                q = lm * dl * xv;
                if (Z) gv = silu_accurate(io<Tin>::load(Z, i));
            }
            sm[lay.dl + cc * kMRow + t] = dl;
            sm[lay.p + cc * kMRow + t] = p;
            sm[lay.q + cc * kMRow + t] = q;
            sm[lay.x + cc * kMRow + t] = xv;
            sm[lay.gate + cc * kMRow + t] = gv;
        }
        for (int j = tid; j < N * (kMT + 1); j += kMThreads) {
            const int n = j / (kMT + 1), tt = j % (kMT + 1);  // B row t0 - 1 + tt
            const int t = t0 - 1 + tt;
            sm[lay.bs + tt * N + n] = (t >= 0 && tt <= tl) ? io<Tin>::load(Bp, bc_base + static_cast<size_t>(n) * L + t) : 0.f;
            if (tt < kMT)
                sm[lay.cs + tt * N + n] = tt < tl ? io<Tin>::load(Cp, bc_base + static_cast<size_t>(n) * L + t0 + tt) : 0.f;
        }
        }  // not prefetched
        __syncthreads();
        if (PREF && t0 + kMT < tend) fetch(t0 + kMT);
        for (int t = 0; t < tl; ++t) {
            const float dl = sm[lay.dl + c * kMRow + t];
            const float p = sm[lay.p + c * kMRow + t], q = sm[lay.q + c * kMRow + t];
            const float4 bp = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kMS * gi);
            const float4 bc = *reinterpret_cast<const float4*>(sm + lay.bs + (t + 1) * N + kMS * gi);
            const float4 cv = *reinterpret_cast<const float4*>(sm + lay.cs + t * N + kMS * gi);
            const float bpa[kMS] = {bp.x, bp.y, bp.z, bp.w}, bca[kMS] = {bc.x, bc.y, bc.z, bc.w};
            const float cva[kMS] = {cv.x, cv.y, cv.z, cv.w};
            float acc = 0.f;
            if (STATES) dsum += dl;
#pragma unroll
            for (int i = 0; i < kMS; ++i) {
                const float mag = ex2_approx(dl * are2[i]);
                float sn, cs;
                sincos_reduced(dl * aim[i], &sn, &cs);
                const float ar = mag * cs, ai = mag * sn;
                const float pr = hr[i] + p * bpa[i], pi = hi[i];
                hr[i] = ar * pr - ai * pi + q * bca[i];
                hi[i] = ar * pi + ai * pr;
                if (!STATES) acc += cva[i] * hr[i];
            }
            if (!STATES) {
#pragma unroll
                for (int off = 1; off < TPC; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (gi == 0)
                    sm[lay.y + c * kMRow + t] = (acc + Dd * sm[lay.x + c * kMRow + t]) * sm[lay.gate + c * kMRow + t];
            }
        }
        if (STATES) continue;
        __syncthreads();
        for (int j = tid; j < CPB * kMT; j += kMThreads) {
            const int cc = j / kMT, t = j % kMT;
            if (cc >= nchan || t >= tl) continue;
            const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
            io<Tout>::store(static_cast<Tout*>(a.y), i, sm[lay.y + cc * kMRow + t]);
        }
    }
    if (STATES) {
        if (active) {
#pragma unroll
            for (int i = 0; i < kMS; ++i) {
                float* hs = seg_state + ((seg * rows + row) * N + kMS * gi + i) * 2;
                hs[0] = hr[i];
                hs[1] = hi[i];
            }
            if (gi == 0) seg_dsum[seg * rows + row] = dsum;
        }
    } else if (active && a.h_final && seg == nseg - 1) {
#pragma unroll
        for (int i = 0; i < kMS; ++i) {
            const size_t hk = (row * N + kMS * gi + i) * 2;
            a.h_final[hk] = hr[i];
            a.h_final[hk + 1] = hi[i];
        }
    }
}

// Time split: when the channel blocks fill fewer than two CTAs per SM, the sequence is
// cut into segments so that about two run; each segment at least 256 steps and a whole
// number of chunks.  (The states-only pass costs about as much as the extra occupancy
// gains at 2.5 CTAs per SM: 1.08 ms unsplit against ~1.12 ms in two segments on the
// 8 x 1536-channel layer.)
struct M3Plan {
    int cps, nseg, seg_len;
    size_t off_dsum, ws_bytes;
};
M3Plan m3_plan(const ssm_mamba3_params& a) {
    const int tpc = a.dstate / kMS;
    const int cpb = kMThreads / tpc;
    const int per_group = a.dim / a.ngroups;
    M3Plan p;
    p.cps = (per_group + cpb - 1) / cpb;
    const long long base = static_cast<long long>(a.batch) * a.ngroups * p.cps;
    int sms = 148, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long want = (2LL * sms + base - 1) / base;
    const long long by_len = a.seqlen / 256;
    if (want > by_len) want = by_len;
    if (want > 64) want = 64;
    p.nseg = want < 1 ? 1 : static_cast<int>(want);
    const int chunks = (a.seqlen + kMT - 1) / kMT;
    p.seg_len = ((chunks + p.nseg - 1) / p.nseg) * kMT;
    if (p.seg_len == 0) p.seg_len = kMT;
    p.nseg = (a.seqlen + p.seg_len - 1) / p.seg_len;
    if (p.nseg < 1) p.nseg = 1;
    const size_t rows = static_cast<size_t>(a.batch) * a.dim;
    const size_t st = static_cast<size_t>(p.nseg - 1) * rows * a.dstate * 2 * sizeof(float);
    p.off_dsum = (st + 255) / 256 * 256;
    p.ws_bytes = p.nseg > 1 ? p.off_dsum + static_cast<size_t>(p.nseg - 1) * rows * sizeof(float) : 0;
    return p;
}

template <typename Tin, typename Tout, int TPC, bool STATES>
cudaError_t launch_m3_pass(const ssm_mamba3_params& a, const M3Plan& p, int grid, float* st, float* ds,
                           cudaStream_t s) {
    constexpr int CPB = kMThreads / TPC;
    const M3Layout lay(CPB, TPC * kMS);
    const size_t smem = static_cast<size_t>(lay.total) * sizeof(float);
    auto k = m3_scan<Tin, Tout, TPC, STATES>;
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(k), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k<<<grid, kMThreads, smem, s>>>(a, p.cps, p.nseg, p.seg_len, st, ds);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int TPC>
cudaError_t launch_m3(const ssm_mamba3_params& a, void* ws, cudaStream_t s) {
    const M3Plan p = m3_plan(a);
    unsigned char* base = static_cast<unsigned char*>(ws);
    float* st = reinterpret_cast<float*>(base);
    float* ds = base ? reinterpret_cast<float*>(base + p.off_dsum) : nullptr;
    const int grid1 = a.batch * a.ngroups * p.cps;
    if (p.nseg > 1) {
        cudaError_t e = launch_m3_pass<Tin, Tout, TPC, true>(a, p, grid1 * (p.nseg - 1), st, ds, s);
        if (e != cudaSuccess) return e;
    }
    return launch_m3_pass<Tin, Tout, TPC, false>(a, p, grid1 * p.nseg, st, ds, s);
}

template <typename Tin, typename Tout>
cudaError_t dispatch_m3(const ssm_mamba3_params& a, void* ws, cudaStream_t s) {
    switch (a.dstate) {
        case 4: return launch_m3<Tin, Tout, 1>(a, ws, s);
        case 8: return launch_m3<Tin, Tout, 2>(a, ws, s);
        case 16: return launch_m3<Tin, Tout, 4>(a, ws, s);
        case 32: return launch_m3<Tin, Tout, 8>(a, ws, s);
        case 64: return launch_m3<Tin, Tout, 16>(a, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool m3_supported(int dstate) {
    return dstate == 4 || dstate == 8 || dstate == 16 || dstate == 32 || dstate == 64;
}

size_t m3_workspace_size(const ssm_mamba3_params& a) {
    if (a.seqlen <= 0) return 0;
    return m3_plan(a).ws_bytes;
}

cudaError_t m3_launch(const ssm_mamba3_params& a, void* workspace, cudaStream_t s) {
    const bool ib = a.in_dtype == SSM_BF16, ob = a.out_dtype == SSM_BF16;
    if (ib && ob) return dispatch_m3<bf16_t, bf16_t>(a, workspace, s);
    if (ib) return dispatch_m3<bf16_t, float>(a, workspace, s);
    if (ob) return dispatch_m3<float, bf16_t>(a, workspace, s);
    return dispatch_m3<float, float>(a, workspace, s);
}

}  // namespace ssm
