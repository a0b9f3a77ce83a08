// scan_m1_bwd.cu -- backward of the Mamba-1 selective scan (exponential-Euler).
//
// The pages train every model through this scan ("From S4 to Mamba-3", 03/System: one
// shared trainer; 05/Evaluation: per-model training-step latency), so the reverse-mode
// derivative of the recurrence belongs to the path.  Forward, per channel d and state n:
//   Delta_t = softplus(delta_t + bias_d),  E_t[n] = exp(Delta_t A[d,n]),
//   h_t[n] = E_t[n] h_{t-1}[n] + Delta_t B_t[n] x_t,
//   o_t = sum_n C_t[n] h_t[n] + D_d x_t,   y_t = o_t SiLU(z_t).
// Backward, walking t downwards with g = dL/dh_t carried from later steps:
//   G_t = g + do_t C_t,   do_t = dy_t SiLU(z_t),   dz_t = dy_t o_t SiLU'(z_t)
//   dC_t[n] = sum_d do_t h_t[n],   dB_t[n] = sum_d G_t[n] Delta_t x_t
//   dx_t = sum_n G_t Delta_t B_t + do_t D,   dDelta_t = sum_n G_t (B_t x_t + h_{t-1} E_t A)
//   dA[n] += G_t h_{t-1} E_t Delta_t,   g <- G_t E_t,   d(delta)_t = dDelta_t sigmoid(v_t).
//
// One launch computes everything per CTA, then a small launch sums the partials:
//   - a CTA owns 128 / TPC channels of one (batch, group) (TPC threads per channel, four
//     consecutive states per thread);
//   - pass 1 runs the recurrence forwards and keeps h at the start of every 16-step chunk
//     (the checkpoints, in the workspace);
//   - pass 2 walks the chunks last to first: it stages the chunk's inputs in shared
//     memory, recomputes h_t over the chunk from its checkpoint into a shared buffer
//     (with the pre-gate output o_t), sums dC over the CTA's channels from that buffer,
//     walks the chunk backwards overwriting h_t by G_t (h_t is dead once step t+1 has
//     used it), then sums dB over the channels from the same buffer;
//   - dB, dC partial sums per CTA and dA, dD, dbias partial sums per batch row go to the
//     workspace; the second launch adds them up, so the result does not depend on the
//     order in which CTAs run.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kBT = 16;          // steps per chunk
constexpr int kBThreads = 128;   // threads per CTA (four CTAs per SM)
constexpr int kBS = 4;           // states per thread
constexpr int kRow = kBT + 1;    // padded row of the per-(channel, step) tiles

struct BwdLayout {  // float offsets into dynamic shared memory (16-byte aligned blocks)
    int h, bs, cs, red, dl, dlx, xs, dout, o, sg, zz, gx, gd, total;
    __host__ __device__ BwdLayout(int cpb, int n) {
        h = 0;                                  // [kBT][kBThreads][kBS]: h_t, then G_t
        bs = h + kBT * kBThreads * kBS;         // [kBT][n] B
        cs = bs + kBT * n;                      // [kBT][n] C
        red = cs + kBT * n;                     // [kBThreads][4] partial sums over channels
        dl = red + kBThreads * 4;               // [cpb][kRow] Delta
        dlx = dl + cpb * kRow;                  // Delta x
        xs = dlx + cpb * kRow;                  // x
        dout = xs + cpb * kRow;                 // dL/do
        o = dout + cpb * kRow;                  // pre-gate output
        sg = o + cpb * kRow;                    // softplus' (sigmoid) or 1
        zz = sg + cpb * kRow;                   // z
        gx = zz + cpb * kRow;                   // dx
        gd = gx + cpb * kRow;                   // d(delta)
        total = gd + cpb * kRow;
    }
};

struct BwdWs {  // byte offsets into the workspace
    size_t ckpt, part_bc, part_a, part_d, part_bias, bytes;
};

__host__ __device__ inline int bwd_cpb(int tpc) { return kBThreads / tpc; }

template <typename T>
__device__ __forceinline__ float ldf(const T* p, size_t i) {
    return io<T>::load(p, i);
}

__device__ __forceinline__ float sigmoid_fast(float v) { return rcp_approx(1.f + ex2_approx(-v * SSM_LOG2E)); }

template <typename Tin, typename Tdy, int TPC>
__global__ void __launch_bounds__(kBThreads, 4)
    m1_scan_bwd(M1BwdArgs a, int cps, float* ckpt, float* part_bc, float* part_a, float* part_d,
                float* part_bias) {
    constexpr int N = TPC * kBS;
    constexpr int CPB = kBThreads / TPC;
    constexpr int NQ = kBT * N / 4;         // (step, 4 states) cells of a chunk
    // channel slices summed in parallel per cell (1: each thread sums whole cells)
    constexpr int SPLIT = NQ < kBThreads ? kBThreads / NQ : 1;
    const int L = a.fwd.seqlen, Dm = a.fwd.dim, G = a.fwd.ngroups;
    const int per_group = Dm / G;
    const int pair = blockIdx.x / cps, part_i = blockIdx.x % cps;
    const int b = pair / G, g = pair % G;
    const int l0 = static_cast<int>((static_cast<long long>(part_i) * per_group) / cps);
    const int l1 = static_cast<int>((static_cast<long long>(part_i + 1) * per_group) / cps);
    const int nchan = l1 - l0;
    const int d0 = g * per_group + l0;
    const int nch = (L + kBT - 1) / kBT;

    extern __shared__ __align__(16) float sm[];
    const BwdLayout lay(CPB, N);
    float* hbuf = sm + lay.h;
    const int tid = threadIdx.x;
    const int c = tid / TPC, gi = tid % TPC;
    const bool active = c < nchan;
    const int d = d0 + (active ? c : 0);
    const size_t row = static_cast<size_t>(b) * Dm + d;  // (b, d)
    const Tin* X = static_cast<const Tin*>(a.fwd.x);
    const Tin* DL = static_cast<const Tin*>(a.fwd.delta);
    const Tin* Z = static_cast<const Tin*>(a.fwd.z);
    const Tin* Bp = static_cast<const Tin*>(a.fwd.B);
    const Tin* Cp = static_cast<const Tin*>(a.fwd.C);
    const Tdy* DY = static_cast<const Tdy*>(a.dy);
    const size_t bc_base = (static_cast<size_t>(b) * G + g) * N * static_cast<size_t>(L);

    float Av[kBS], A2[kBS];  // A, and A log2(e) for the exponentials
#pragma unroll
    for (int i = 0; i < kBS; ++i) {
        Av[i] = a.fwd.A[static_cast<size_t>(d) * N + kBS * gi + i];
        A2[i] = Av[i] * SSM_LOG2E;
    }
    const float Dd = a.fwd.D_skip ? a.fwd.D_skip[d] : 0.f;

    // stage Delta (and Delta x, x, sigmoid, dL/do, z) of the CTA's channels and B (C)
    // for a chunk
    auto stage = [&](int t0, int tl, bool full) {
        for (int j = tid; j < CPB * kBT; j += kBThreads) {
            const int cc = j / kBT, t = j % kBT;
            float dl = 0.f, xv = 0.f, sgv = 1.f, dov = 0.f, zv = 0.f;
            if (cc < nchan && t < tl) {
                const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
                const float v = ldf(DL, i) + (a.fwd.delta_bias ? a.fwd.delta_bias[d0 + cc] : 0.f);
                dl = a.fwd.delta_softplus ? softplus_fast(v) : v;
                xv = ldf(X, i);
                if (full) {
                    sgv = a.fwd.delta_softplus ? sigmoid_fast(v) : 1.f;
                    dov = ldf(DY, i);
                    if (Z) {
                        zv = ldf(Z, i);
                        dov *= silu_fast(zv);
                    }
                }
            }
            sm[lay.dl + cc * kRow + t] = dl;
            sm[lay.dlx + cc * kRow + t] = dl * xv;
            if (full) {
                sm[lay.xs + cc * kRow + t] = xv;
                sm[lay.sg + cc * kRow + t] = sgv;
                sm[lay.dout + cc * kRow + t] = dov;
                sm[lay.zz + cc * kRow + t] = zv;
            }
        }
        for (int j = tid; j < N * kBT; j += kBThreads) {
            const int n = j / kBT, t = j % kBT;
            const size_t i = bc_base + static_cast<size_t>(n) * L + t0 + t;
            sm[lay.bs + t * N + n] = t < tl ? ldf(Bp, i) : 0.f;
            if (full) sm[lay.cs + t * N + n] = t < tl ? ldf(Cp, i) : 0.f;
        }
    };
    // sum over the CTA's channels of w[channel][t] * buf[t][channel][n] for every (t, n) of
    // the chunk, into the partial row `dst` ([N][L] at column t0): cell q = (t, 4 states)
    // per thread slice, SPLIT slices of the channels, then the slices added
    auto channel_sum = [&](int wofs, float* dst, int t0, int tl) {
      for (int q0 = 0; q0 < (NQ > kBThreads ? NQ : 1); q0 += kBThreads) {
        const int q = NQ > kBThreads ? q0 + tid : tid % NQ, sl = NQ > kBThreads ? 0 : tid / NQ;
        const int t = q / (N / 4), n4 = q % (N / 4);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < tl) {
            for (int cc = sl; cc < nchan; cc += SPLIT) {
                const float w = sm[wofs + cc * kRow + t];
                const float4 v = *reinterpret_cast<const float4*>(hbuf + (t * kBThreads + cc * TPC + n4) * kBS);
                s.x += w * v.x;
                s.y += w * v.y;
                s.z += w * v.z;
                s.w += w * v.w;
            }
        }
        if (SPLIT > 1) {
            *reinterpret_cast<float4*>(sm + lay.red + tid * 4) = s;
            __syncthreads();
            if (sl == 0) {
#pragma unroll
                for (int k = 1; k < SPLIT; ++k) {
                    const float4 o = *reinterpret_cast<const float4*>(sm + lay.red + (tid + k * NQ) * 4);
                    s.x += o.x;
                    s.y += o.y;
                    s.z += o.z;
                    s.w += o.w;
                }
            }
        }
        if (sl == 0 && t < tl) {
            dst[static_cast<size_t>(4 * n4 + 0) * L + t0 + t] = s.x;
            dst[static_cast<size_t>(4 * n4 + 1) * L + t0 + t] = s.y;
            dst[static_cast<size_t>(4 * n4 + 2) * L + t0 + t] = s.z;
            dst[static_cast<size_t>(4 * n4 + 3) * L + t0 + t] = s.w;
        }
      }
    };

    // pass 1: checkpoints h_{t0 - 1} of every chunk
    float h[kBS];
#pragma unroll
    for (int i = 0; i < kBS; ++i) h[i] = (active && a.fwd.h0) ? a.fwd.h0[row * N + kBS * gi + i] : 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        const int t0 = ch * kBT, tl = min(kBT, L - t0);
        if (active)
            *reinterpret_cast<float4*>(ckpt + (row * nch + ch) * N + kBS * gi) = make_float4(h[0], h[1], h[2], h[3]);
        __syncthreads();
        stage(t0, tl, false);
        __syncthreads();
        for (int t = 0; t < tl; ++t) {
            const float dl = sm[lay.dl + c * kRow + t], dlx = sm[lay.dlx + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float bb[kBS] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < kBS; ++i) h[i] = ex2_approx(dl * A2[i]) * h[i] + dlx * bb[i];
        }
    }

    // pass 2: chunks last to first
    float gcar[kBS], dAacc[kBS];
#pragma unroll
    for (int i = 0; i < kBS; ++i) {
        gcar[i] = (active && a.dh_final) ? a.dh_final[row * N + kBS * gi + i] : 0.f;
        dAacc[i] = 0.f;
    }
    float dDacc = 0.f, dbacc = 0.f;
    float* pbc = part_bc + (static_cast<size_t>(pair) * cps + part_i) * 2 * N * static_cast<size_t>(L);
    for (int ch = nch - 1; ch >= 0; --ch) {
        const int t0 = ch * kBT, tl = min(kBT, L - t0);
        __syncthreads();  // the previous chunk's tiles are no longer read
        stage(t0, tl, true);
        float hs[kBS];
        {
            const float4 v = active ? *reinterpret_cast<const float4*>(ckpt + (row * nch + ch) * N + kBS * gi)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            hs[0] = v.x; hs[1] = v.y; hs[2] = v.z; hs[3] = v.w;
        }
        __syncthreads();
        // recompute h_t over the chunk, and the pre-gate output
#pragma unroll
        for (int i = 0; i < kBS; ++i) h[i] = hs[i];
        for (int t = 0; t < tl; ++t) {
            const float dl = sm[lay.dl + c * kRow + t], dlx = sm[lay.dlx + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float4 cv = *reinterpret_cast<const float4*>(sm + lay.cs + t * N + kBS * gi);
            const float bb[kBS] = {bv.x, bv.y, bv.z, bv.w}, cb[kBS] = {cv.x, cv.y, cv.z, cv.w};
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kBS; ++i) {
                h[i] = ex2_approx(dl * A2[i]) * h[i] + dlx * bb[i];
                acc += cb[i] * h[i];
            }
            *reinterpret_cast<float4*>(hbuf + (t * kBThreads + tid) * kBS) = make_float4(h[0], h[1], h[2], h[3]);
#pragma unroll
            for (int off = 1; off < TPC; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (gi == 0) sm[lay.o + c * kRow + t] = acc + Dd * sm[lay.xs + c * kRow + t];
        }
        __syncthreads();
        // dC_t[n] = sum over the CTA's channels of do_t h_t[n]; dz from the pre-gate output
        channel_sum(lay.dout, pbc + static_cast<size_t>(N) * L, t0, tl);
        if (a.dz) {
            for (int j = tid; j < CPB * kBT; j += kBThreads) {
                const int cc = j / kBT, t = j % kBT;
                if (cc >= nchan || t >= tl) continue;
                const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
                const float zv = sm[lay.zz + cc * kRow + t];
                const float sgz = sigmoid_fast(zv);
                a.dz[i] = ldf(DY, i) * sm[lay.o + cc * kRow + t] * sgz * (1.f + zv * (1.f - sgz));
            }
        }
        __syncthreads();
        // backwards over the chunk: G_t replaces h_t in the buffer
        for (int t = tl - 1; t >= 0; --t) {
            float hp[kBS];
            if (t > 0) {
                const float4 v = *reinterpret_cast<const float4*>(hbuf + ((t - 1) * kBThreads + tid) * kBS);
                hp[0] = v.x; hp[1] = v.y; hp[2] = v.z; hp[3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < kBS; ++i) hp[i] = hs[i];
            }
            const float dl = sm[lay.dl + c * kRow + t], xv = sm[lay.xs + c * kRow + t];
            const float dov = sm[lay.dout + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float4 cv = *reinterpret_cast<const float4*>(sm + lay.cs + t * N + kBS * gi);
            const float bb[kBS] = {bv.x, bv.y, bv.z, bv.w}, cb[kBS] = {cv.x, cv.y, cv.z, cv.w};
            float gx = 0.f, gd = 0.f, Gt[kBS];
#pragma unroll
            for (int i = 0; i < kBS; ++i) {
                const float E = ex2_approx(dl * A2[i]);
                Gt[i] = gcar[i] + dov * cb[i];
                gx += Gt[i] * bb[i];
                const float hE = hp[i] * E;
                gd += Gt[i] * (bb[i] * xv + hE * Av[i]);
                dAacc[i] += Gt[i] * hE * dl;
                gcar[i] = Gt[i] * E;
            }
            gx *= dl;
            *reinterpret_cast<float4*>(hbuf + (t * kBThreads + tid) * kBS) = make_float4(Gt[0], Gt[1], Gt[2], Gt[3]);
#pragma unroll
            for (int off = 1; off < TPC; off <<= 1) {
                gx += __shfl_xor_sync(0xffffffffu, gx, off);
                gd += __shfl_xor_sync(0xffffffffu, gd, off);
            }
            if (gi == 0) {
                const float dv = gd * sm[lay.sg + c * kRow + t];
                sm[lay.gx + c * kRow + t] = gx + dov * Dd;
                sm[lay.gd + c * kRow + t] = dv;
                dDacc += dov * xv;
                dbacc += dv;
            }
        }
        __syncthreads();
        // dB_t[n] = sum over the CTA's channels of G_t[n] Delta_t x_t
        channel_sum(lay.dlx, pbc, t0, tl);
        for (int j = tid; j < CPB * kBT; j += kBThreads) {
            const int cc = j / kBT, t = j % kBT;
            if (cc >= nchan || t >= tl) continue;
            const size_t i = (static_cast<size_t>(b) * Dm + d0 + cc) * L + t0 + t;
            a.dx[i] = sm[lay.gx + cc * kRow + t];
            a.ddelta[i] = sm[lay.gd + cc * kRow + t];
        }
    }
    if (active) {
        if (a.dh0)
            *reinterpret_cast<float4*>(a.dh0 + row * N + kBS * gi) = make_float4(gcar[0], gcar[1], gcar[2], gcar[3]);
        *reinterpret_cast<float4*>(part_a + row * N + kBS * gi) = make_float4(dAacc[0], dAacc[1], dAacc[2], dAacc[3]);
        if (gi == 0) {
            part_d[row] = dDacc;
            part_bias[row] = dbacc;
        }
    }
}

// dB, dC: sum of the per-CTA partials of each (batch, group); dA, dD, dbias: sum over the
// batch.  One thread per output element.
__global__ void m1_scan_bwd_reduce(M1BwdArgs a, int cps, const float* part_bc, const float* part_a,
                                   const float* part_d, const float* part_bias) {
    const int L = a.fwd.seqlen, Dm = a.fwd.dim, G = a.fwd.ngroups, N = a.fwd.dstate, Bt = a.fwd.batch;
    const size_t nbc = static_cast<size_t>(Bt) * G * N * L;
    const size_t na = static_cast<size_t>(Dm) * N;
    const size_t total = 2 * nbc + na + 2 * static_cast<size_t>(Dm);
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (i < 2 * nbc) {
            const int which = i < nbc ? 0 : 1;  // 0: dB, 1: dC
            const size_t e = i % nbc;           // (pair, n, t)
            const size_t pair = e / (static_cast<size_t>(N) * L), nt = e % (static_cast<size_t>(N) * L);
            float s = 0.f;
            for (int p = 0; p < cps; ++p)
                s += part_bc[((pair * cps + p) * 2 + which) * N * static_cast<size_t>(L) + nt];
            (which ? a.dC : a.dB)[e] = s;
        } else if (i < 2 * nbc + na) {
            const size_t e = i - 2 * nbc;  // (d, n)
            float s = 0.f;
            for (int bb = 0; bb < Bt; ++bb) s += part_a[static_cast<size_t>(bb) * na + e];
            a.dA[e] = s;
        } else {
            const size_t e = i - 2 * nbc - na;
            const int dd = static_cast<int>(e % Dm);
            const float* src = e < static_cast<size_t>(Dm) ? part_d : part_bias;
            float* dst = e < static_cast<size_t>(Dm) ? a.dD_skip : a.ddelta_bias;
            if (!dst) continue;
            float s = 0.f;
            for (int bb = 0; bb < Bt; ++bb) s += src[static_cast<size_t>(bb) * Dm + dd];
            dst[dd] = s;
        }
    }
}

// threads per channel for each supported dstate (four states per thread); smaller
// dstates would need more channels per CTA than the shared-memory tiles hold
int bwd_tpc(int n) {
    switch (n) {
        case 16: return 4;
        case 32: return 8;
        case 64: return 16;
        default: return 0;
    }
}

BwdWs bwd_ws(const M1BwdArgs& a, int cps) {
    const ssm_scan_params& f = a.fwd;
    const size_t rows = static_cast<size_t>(f.batch) * f.dim;
    const size_t nch = (static_cast<size_t>(f.seqlen) + kBT - 1) / kBT;
    const size_t pairs = static_cast<size_t>(f.batch) * f.ngroups;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    BwdWs w;
    w.ckpt = 0;
    w.part_bc = r256(rows * nch * f.dstate * 4);
    w.part_a = w.part_bc + r256(pairs * cps * 2 * f.dstate * static_cast<size_t>(f.seqlen) * 4);
    w.part_d = w.part_a + r256(rows * f.dstate * 4);
    w.part_bias = w.part_d + r256(rows * 4);
    w.bytes = w.part_bias + r256(rows * 4);
    return w;
}

int bwd_cps(const M1BwdArgs& a) {
    const int tpc = bwd_tpc(a.fwd.dstate);
    const int cpb = bwd_cpb(tpc);
    const int per_group = a.fwd.dim / a.fwd.ngroups;
    return (per_group + cpb - 1) / cpb;
}

template <typename Tin, typename Tdy, int TPC>
cudaError_t launch_bwd(const M1BwdArgs& a, void* ws, cudaStream_t s) {
    const int cps = bwd_cps(a);
    const BwdWs w = bwd_ws(a, cps);
    unsigned char* base = static_cast<unsigned char*>(ws);
    const BwdLayout lay(bwd_cpb(TPC), TPC * kBS);
    const size_t smem = static_cast<size_t>(lay.total) * sizeof(float);
    auto k = m1_scan_bwd<Tin, Tdy, TPC>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = a.fwd.batch * a.fwd.ngroups * cps;
    float* part_bc = reinterpret_cast<float*>(base + w.part_bc);
    float* part_a = reinterpret_cast<float*>(base + w.part_a);
    float* part_d = reinterpret_cast<float*>(base + w.part_d);
    float* part_bias = reinterpret_cast<float*>(base + w.part_bias);
    if (grid > 0)
        k<<<grid, kBThreads, smem, s>>>(a, cps, reinterpret_cast<float*>(base + w.ckpt), part_bc, part_a,
                                        part_d, part_bias);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    m1_scan_bwd_reduce<<<2 * 152, 256, 0, s>>>(a, cps, part_bc, part_a, part_d, part_bias);
    return cudaGetLastError();
}

template <typename Tin, typename Tdy>
cudaError_t dispatch_tpc(const M1BwdArgs& a, void* ws, cudaStream_t s) {
    switch (bwd_tpc(a.fwd.dstate)) {
        case 4: return launch_bwd<Tin, Tdy, 4>(a, ws, s);
        case 8: return launch_bwd<Tin, Tdy, 8>(a, ws, s);
        case 16: return launch_bwd<Tin, Tdy, 16>(a, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool m1_bwd_supported(const M1BwdArgs& a) {
    return a.fwd.disc == SSM_DISC_EXP_EULER && bwd_tpc(a.fwd.dstate) > 0;
}

size_t m1_bwd_workspace_size(const M1BwdArgs& a) {
    if (!m1_bwd_supported(a)) return 0;
    return bwd_ws(a, bwd_cps(a)).bytes;
}

cudaError_t m1_bwd_launch(const M1BwdArgs& a, void* workspace, cudaStream_t s) {
    const bool in_bf = a.fwd.in_dtype == SSM_BF16, dy_bf = a.fwd.out_dtype == SSM_BF16;
    if (in_bf && dy_bf) return dispatch_tpc<bf16_t, bf16_t>(a, workspace, s);
    if (in_bf) return dispatch_tpc<bf16_t, float>(a, workspace, s);
    if (dy_bf) return dispatch_tpc<float, bf16_t>(a, workspace, s);
    return dispatch_tpc<float, float>(a, workspace, s);
}

}  // namespace ssm
