// step.cu -- decode update (sm_103a), in place on the fp32 state: one step, or T
// consecutive tokens with the state held in registers between them.
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
__device__ __forceinline__ float step_delta(const StepArgs& a, long long tok_off, int b, int hd) {
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const float v = to_f32(DT[tok_off + static_cast<size_t>(b) * a.nheads + hd]) +
                    (a.dt_bias ? a.dt_bias[hd] : 0.f);
    return a.dt_softplus ? softplus_accurate(v) : v;
}

// Vector path.  A CTA owns kRowsPerCta consecutive state rows; its prologue computes, once
// per (batch, head) in that range, the step Delta, the decay exp(Delta A) and the input
// weight, plus the B/C offset, into shared memory (softplus and exp run once per head,
// not once per lane).  Each warp then streams rows: LPR lanes per row, NV float4 groups
// per lane, UNROLL rows of loads in flight, f32x2 arithmetic, a shuffle tree for y.
constexpr int kStepThreads = 256;

// One token (the common decode step): the state row is loaded, updated and stored per row.
template <typename Tin, typename Tout, int NV, int LPR, int UNROLL, bool PER_STATE>
__global__ void __launch_bounds__(kStepThreads) step_vec1(StepArgs a, int rows_per_cta,
                                                         int log2p) {
    // dependent launch: let the next launch be scheduled, then wait for the one before
    // (its writes, for instance this layer's input) before touching global memory
    grid_dep_launch();
    grid_dep_wait();
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

template <typename Tin, typename Tout, int NV, int LPR, int UNROLL, bool PER_STATE>
__global__ void __launch_bounds__(kStepThreads) step_vec(StepArgs a, int rows_per_cta,
                                                         int log2p, int tab) {
    // dependent launch: let the next launch be scheduled, then wait for the one before
    // (its writes, for instance this layer's input) before touching global memory
    grid_dep_launch();
    grid_dep_wait();
    constexpr int RPW = 32 / LPR;  // rows per warp per pass
    const int N = a.dstate;
    const int T = a.ntok;
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    const long long r0 = static_cast<long long>(blockIdx.x) * rows_per_cta;
    const long long r1 = min(rows, r0 + rows_per_cta);
    const int P = a.headdim;
    // token strides of the token-major inputs
    const long long sx = rows;                                                  // x, z, y
    const long long sdt = static_cast<long long>(a.batch) * a.nheads;           // dt
    const long long sbc = static_cast<long long>(a.batch) * a.ngroups * N;      // B, C
    // (batch, head) range of this CTA
    const long long bh0 = log2p >= 0 ? (r0 >> log2p) : r0 / P;
    const long long bh1 = log2p >= 0 ? ((r1 - 1) >> log2p) : (r1 - 1) / P;
    const int nbh = static_cast<int>(bh1 - bh0 + 1);
    extern __shared__ float s_step[];
    float* s_d = s_step;                             // D_h
    int* s_bc = reinterpret_cast<int*>(s_d + nbh);   // B/C row offset (b * G + g) * N
    int* s_h = s_bc + nbh;                           // head index
    float* s_dt = reinterpret_cast<float*>(s_h + nbh);  // [T][nbh] Delta      (when tab)
    float* s_da = s_dt + T * nbh;                        // [T][nbh] exp(Delta A_h) (scalar-A form)
    float* s_w = s_da + T * nbh;                         // [T][nbh] input weight / Delta
    const int per_group = a.nheads / a.ngroups;
    const Tin* DT = static_cast<const Tin*>(a.dt);
    for (int i = threadIdx.x; i < nbh; i += blockDim.x) {
        const long long bh = bh0 + i;
        const int hd = static_cast<int>(bh % a.nheads);
        const int b = static_cast<int>(bh / a.nheads);
        s_d[i] = a.D ? a.D[hd] : 0.f;
        s_bc[i] = (b * a.ngroups + hd / per_group) * N;
        s_h[i] = hd;
    }
    // per-token step quantities: in shared memory once per (token, batch, head) when the
    // table fits, otherwise recomputed where used
    auto step_q = [&](int tok, long long bh, int hd, float& dt, float& da, float& w) {
        const float v = to_f32(DT[tok * sdt + bh]) + (a.dt_bias ? a.dt_bias[hd] : 0.f);
        dt = a.dt_softplus ? softplus_accurate(v) : v;
        if (!PER_STATE) {
            const float za = dt * a.A[hd];
            da = expf(za);
            w = a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f;
        }
    };
    if (tab) {
        for (int j = threadIdx.x; j < T * nbh; j += blockDim.x) {
            const int tok = j / nbh, i = j % nbh;
            float dt, da = 0.f, w = 0.f;
            step_q(tok, bh0 + i, static_cast<int>((bh0 + i) % a.nheads), dt, da, w);
            s_dt[j] = dt;
            s_da[j] = da;
            s_w[j] = w;
        }
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
        for (int tok = 0; tok < T; ++tok) {  // the state stays in registers across tokens
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const long long r = rr[u] < r1 ? rr[u] : r1 - 1;
                const long long bhr = log2p >= 0 ? (r >> log2p) : r / P;
                const int i = static_cast<int>(bhr - bh0);
                float dt, dsa = 0.f, wsa = 0.f;
                if (tab) {
                    dt = s_dt[tok * nbh + i];
                    dsa = s_da[tok * nbh + i];
                    wsa = s_w[tok * nbh + i];
                } else {
                    step_q(tok, bhr, s_h[i], dt, dsa, wsa);
                }
                const float xp = to_f32(X[tok * sx + r]);
                const float dx = dt * xp;
                const Tin* Bt = Bp + tok * sbc + s_bc[i];
                const Tin* Ct = Cp + tok * sbc + s_bc[i];
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int n0 = 4 * (li + v * LPR);
                    float bv[4], cv[4];
                    load4_f32(Bt + n0, bv);
                    load4_f32(Ct + n0, cv);
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
                        da01 = da23 = make_float2(dsa, dsa);
                        wdx01 = wdx23 = wdx2 = wdx3 = wsa * dx;
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
                if (rr[u] < r1 && li == 0) {
                    float yv = sum + s_d[i] * xp;
                    if (Z) yv *= silu_accurate(to_f32(Z[tok * sx + r]));
                    io<Tout>::store(static_cast<Tout*>(a.y), tok * sx + r, yv);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (rr[u] < r1) {
                float4* sp = reinterpret_cast<float4*>(a.state + rr[u] * N);
#pragma unroll
                for (int v = 0; v < NV; ++v) __stcs(sp + li + v * LPR, hv[u][v]);
            }
        }
    }
}

// Several tokens, Mamba-2 form (A per head), N = 32 NV.  A CTA of 8 warps owns ROWS = 32 UNR
// consecutive state rows (each warp 4 row slots x UNR; 8 lanes per row, NV float4 per
// lane) and keeps them in registers for all T tokens.  Tokens go in blocks of up to
// `tb_max`; per block the CTA stages in shared memory x and the output gate silu(z) of its
// rows, (exp(Delta A), w Delta) for each (batch, head) it touches and the B and C rows of
// each (batch, group).  The row work reads only shared memory.  y partial sums of
// TG = 8 / UNR consecutive tokens x UNR rows are reduced together over the row's 8 lanes
// by a butterfly reduce-scatter (7 shuffles for 8 sums), after which lane li holds sum li
// and writes that y.  SHARED: every CTA's rows lie in one (batch, group), so the UNR row
// slots read the same B and C values.
constexpr int kTokThreads = 256;

struct TokSmem {  // float offsets of the staged arrays, all 16-byte aligned
    int q, x, g, bc, total;
};
__host__ __device__ inline int tok_align4(int v) { return (v + 3) & ~3; }
__host__ __device__ inline TokSmem tok_smem(int nbh_max, int nbg_max, int tb, int n, int rows) {
    TokSmem o;
    o.q = tok_align4(nbh_max);                  // [nbh_max] D, then [tb][nbh_max] float2
    o.x = o.q + tok_align4(tb * nbh_max * 2);   // [tb][rows] x
    o.g = o.x + tb * rows;                      // [tb][rows] silu(z) (or 1)
    o.bc = o.g + tb * rows;                     // [tb][nbg_max][2n] B then C
    o.total = o.bc + tb * nbg_max * 2 * n;
    return o;
}

template <int NV>
struct TokShape {
    static constexpr int UNR = NV == 4 ? 4 : 2;  // row slots per thread (the fastest measured)
    static constexpr int TG = 8 / UNR;            // tokens per reduction group
    static constexpr int ROWS = 32 * UNR;         // rows per CTA
};

template <typename Tin, typename Tout, int NV, bool SHARED>
__global__ void __launch_bounds__(kTokThreads) step_tok(StepArgs a, int log2p, int nbh_max,
                                                        int nbg_max, int tb_max) {
    // dependent launch: let the next launch be scheduled, then wait for the one before
    // (its writes, for instance this layer's input) before touching global memory
    grid_dep_launch();
    grid_dep_wait();
    constexpr int LPR = 8, RPW = 4;
    constexpr int UNR = TokShape<NV>::UNR, TG = TokShape<NV>::TG, ROWS = TokShape<NV>::ROWS;
    constexpr int N = 32 * NV;
    const int T = a.ntok;
    const int P = a.headdim, H = a.nheads, G = a.ngroups;
    const long long rows = static_cast<long long>(a.batch) * H * P;
    const long long r0 = static_cast<long long>(blockIdx.x) * ROWS;
    const long long r1 = min(rows, r0 + ROWS);
    const int nr = static_cast<int>(r1 - r0);
    const long long sdt = static_cast<long long>(a.batch) * H;
    const long long sbc = static_cast<long long>(a.batch) * G * N;
    const int per_group = H / G;
    auto bh_of = [&](long long r) { return log2p >= 0 ? (r >> log2p) : r / P; };
    auto bg_of = [&](long long bh) { return (bh / H) * G + (bh % H) / per_group; };
    const long long bh0 = bh_of(r0), bh1 = bh_of(r1 - 1);
    const long long bg0 = bg_of(bh0);
    const int nbh = static_cast<int>(bh1 - bh0 + 1);
    const int nbg = static_cast<int>(bg_of(bh1) - bg0 + 1);

    extern __shared__ __align__(16) float s_tok[];
    const TokSmem L = tok_smem(nbh_max, nbg_max, tb_max, N, ROWS);
    float* s_D = s_tok;
    float2* s_q = reinterpret_cast<float2*>(s_tok + L.q);
    float* s_x = s_tok + L.x;
    float* s_g = s_tok + L.g;
    float* s_bc = s_tok + L.bc;
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    for (int i = threadIdx.x; i < nbh; i += blockDim.x) {
        const int hd = static_cast<int>((bh0 + i) % H);
        s_D[i] = a.D ? a.D[hd] : 0.f;
    }

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPR, li = lane % LPR;
    int rl[UNR], bi[UNR], gi[UNR];
    float4 hv[UNR][NV];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
        rl[u] = warp * (RPW * UNR) + u * RPW + sub;
        const long long r = r0 + min(rl[u], nr - 1);
        const long long bh = bh_of(r);
        bi[u] = static_cast<int>(bh - bh0);
        gi[u] = SHARED ? 0 : static_cast<int>(bg_of(bh) - bg0);
        if (rl[u] < nr) {
            const float4* sp = reinterpret_cast<const float4*>(a.state + (r0 + rl[u]) * N);
#pragma unroll
            for (int v = 0; v < NV; ++v) hv[u][v] = __ldcs(sp + li + v * LPR);
        } else {
#pragma unroll
            for (int v = 0; v < NV; ++v) hv[u][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // the (row slot, token) whose y this lane writes after each reduction
    const int my_u = li / TG, my_t = li % TG;
    int my_rl = rl[0], my_bi = bi[0];
#pragma unroll
    for (int u = 1; u < UNR; ++u)
        if (my_u == u) { my_rl = rl[u]; my_bi = bi[u]; }

    for (int t0 = 0; t0 < T; t0 += tb_max) {
        const int tb = min(tb_max, T - t0);
        __syncthreads();  // the previous block's staged values are no longer read
        for (int j = threadIdx.x; j < tb * nbh; j += blockDim.x) {
            const int tk = j / nbh, i = j % nbh;
            const long long bh = bh0 + i;
            const int hd = static_cast<int>(bh % H);
            const float v = to_f32(DT[(t0 + tk) * sdt + bh]) + (a.dt_bias ? a.dt_bias[hd] : 0.f);
            const float dt = a.dt_softplus ? softplus_accurate(v) : v;
            const float za = dt * a.A[hd];
            s_q[tk * nbh_max + i] = make_float2(expf(za), (a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f) * dt);
        }
        for (int j = threadIdx.x; j < tb * ROWS; j += blockDim.x) {
            const int tk = j / ROWS, r = j % ROWS;
            float xv = 0.f, gv = 1.f;
            if (r < nr) {
                const long long off = (t0 + tk) * rows + r0 + r;
                xv = to_f32(X[off]);
                if (Z) gv = silu_accurate(to_f32(Z[off]));
            }
            s_x[j] = xv;
            s_g[j] = gv;
        }
        for (int j = threadIdx.x; j < tb * nbg * (2 * N / 4); j += blockDim.x) {
            const int n4 = j % (2 * N / 4), gb = (j / (2 * N / 4)) % nbg, tk = j / (2 * N / 4) / nbg;
            const int n = 4 * n4;
            const Tin* src = (n < N ? Bp : Cp) + (t0 + tk) * sbc + (bg0 + gb) * N + (n % N);
            float vv[4];
            load4_f32(src, vv);
            *reinterpret_cast<float4*>(s_bc + (tk * nbg_max + gb) * 2 * N + n) =
                make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
        __syncthreads();
        for (int tg = 0; tg < tb; tg += TG) {
            float ps[UNR * TG];  // partial y sums, index u * TG + token
#pragma unroll
            for (int k = 0; k < TG; ++k) {
                if (tg + k < tb) {
                    const int tk = tg + k;
                    const float* bc0 = s_bc + (tk * nbg_max) * 2 * N;
#pragma unroll
                    for (int u = 0; u < UNR; ++u) {
                        const float2 q = s_q[tk * nbh_max + bi[u]];
                        const float wdx = q.y * s_x[tk * ROWS + rl[u]];
                        const float2 da = make_float2(q.x, q.x);
                        const float2 wd2 = make_float2(wdx, wdx);
                        const float* bc = bc0 + (SHARED ? 0 : gi[u] * 2 * N);
                        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            const int n0 = 4 * (li + v * LPR);
                            const float4 b4 = *reinterpret_cast<const float4*>(bc + n0);
                            const float4 c4 = *reinterpret_cast<const float4*>(bc + N + n0);
                            float2 h01 = make_float2(hv[u][v].x, hv[u][v].y);
                            float2 h23 = make_float2(hv[u][v].z, hv[u][v].w);
                            h01 = fma2(da, h01, mul2(wd2, make_float2(b4.x, b4.y)));
                            h23 = fma2(da, h23, mul2(wd2, make_float2(b4.z, b4.w)));
                            hv[u][v] = make_float4(h01.x, h01.y, h23.x, h23.y);
                            acc0 = fma2(make_float2(c4.x, c4.y), h01, acc0);
                            acc1 = fma2(make_float2(c4.z, c4.w), h23, acc1);
                        }
                        ps[u * TG + k] = (acc0.x + acc1.x) + (acc0.y + acc1.y);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < UNR; ++u) ps[u * TG + k] = 0.f;
                }
            }
            // reduce-scatter over the 8 lanes of the row: lane li ends with sum li
            float r4[4], r2[2];
            const bool b4 = li & 4, b2 = li & 2, b1 = li & 1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float send = b4 ? ps[k] : ps[k + 4];
                const float keep = b4 ? ps[k + 4] : ps[k];
                r4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float send = b2 ? r4[k] : r4[k + 2];
                const float keep = b2 ? r4[k + 2] : r4[k];
                r2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
            }
            const float sum = (b1 ? r2[1] : r2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? r2[0] : r2[1], 1);
            const int tk = tg + my_t;
            if (tk < tb && my_rl < nr) {
                const float xp = s_x[tk * ROWS + my_rl];
                const float yv = (sum + s_D[my_bi] * xp) * s_g[tk * ROWS + my_rl];
                io<Tout>::store(static_cast<Tout*>(a.y), static_cast<long long>(t0 + tk) * rows + r0 + my_rl, yv);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
        if (rl[u] < nr) {
            float4* sp = reinterpret_cast<float4*>(a.state + (r0 + rl[u]) * N);
#pragma unroll
            for (int v = 0; v < NV; ++v) __stcs(sp + li + v * LPR, hv[u][v]);
        }
    }
}

template <typename Tin, typename Tout, int NV, bool SHARED>
static cudaError_t launch_tok_k(const StepArgs& a, long long rows, int log2p, cudaStream_t s) {
    constexpr int N = 32 * NV, ROWS = TokShape<NV>::ROWS;
    const int P = a.headdim;
    // (batch, head) pairs one ROWS-row span can touch: exact when P divides ROWS or ROWS
    // divides P
    const int nbh_max = (ROWS % P == 0) ? ROWS / P : (P % ROWS == 0) ? 1 : ROWS / P + 2;
    const int nbg_max = SHARED ? 1 : nbh_max;
    const int budget = 40 * 1024 / 4;  // floats of shared memory per CTA
    int tb = 32;
    if (tb > a.ntok) tb = a.ntok;
    while (tb > 1 && tok_smem(nbh_max, nbg_max, tb, N, ROWS).total > budget) --tb;
    const size_t smem = static_cast<size_t>(tok_smem(nbh_max, nbg_max, tb, N, ROWS).total) * sizeof(float);
    auto k = step_tok<Tin, Tout, NV, SHARED>;
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(k), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long grid = (rows + ROWS - 1) / ROWS;
    return launch_dependent(k, static_cast<unsigned>(grid), kTokThreads, smem, s, a, log2p, nbh_max, nbg_max, tb);
}

template <typename Tin, typename Tout, int NV>
static cudaError_t launch_tok(const StepArgs& a, long long rows, cudaStream_t s) {
    constexpr int ROWS = TokShape<NV>::ROWS;
    const int P = a.headdim;
    int log2p = -1;
    if ((P & (P - 1)) == 0) {
        log2p = 0;
        while ((1 << log2p) < P) ++log2p;
    }
    // a group spans P * H / G consecutive rows (batches start on group boundaries): when
    // that is a multiple of ROWS no CTA crosses a group
    const long long group_rows = static_cast<long long>(P) * (a.nheads / a.ngroups);
    if (group_rows % ROWS == 0) return launch_tok_k<Tin, Tout, NV, true>(a, rows, log2p, s);
    return launch_tok_k<Tin, Tout, NV, false>(a, rows, log2p, s);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(128) step_scalar(StepArgs a) {
    // dependent launch: let the next launch be scheduled, then wait for the one before
    // (its writes, for instance this layer's input) before touching global memory
    grid_dep_launch();
    grid_dep_wait();
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
    const long long sdt = static_cast<long long>(a.batch) * a.nheads;
    const long long sbc = static_cast<long long>(a.batch) * a.ngroups * N;
    float* hrow = a.state + r * N;
    for (int tok = 0; tok < a.ntok; ++tok) {
        const float dt = step_delta<Tin>(a, tok * sdt, b, hd);
        const float xp = to_f32(X[tok * rows + r]);
        float acc = 0.f;
        for (int n = 0; n < N; ++n) {
            const size_t bc = tok * sbc + (static_cast<size_t>(b) * a.ngroups + g) * N + n;
            const float av = a.a_per_state ? a.A[static_cast<size_t>(hd) * N + n] : a.A[hd];
            const float za = dt * av;
            const float w = a.disc == SSM_DISC_ZOH ? dt * phi1f(za) : dt;
            const float hn = expf(za) * hrow[n] + w * xp * to_f32(Bp[bc]);
            hrow[n] = hn;
            acc += to_f32(Cp[bc]) * hn;
        }
        float yv = acc + (a.D ? a.D[hd] : 0.f) * xp;
        if (Z) yv *= silu_accurate(to_f32(Z[tok * rows + r]));
        io<Tout>::store(static_cast<Tout*>(a.y), tok * rows + r, yv);
    }
}

// Mamba-1 form, one token (A per state, P = 1, N = 16): every row is one (batch, channel)
// with its own Delta, so there is no per-head work to share through a prologue.  LPR
// lanes per row (16 / LPR states each, in float4 groups), 32 / LPR rows per warp per pass,
// UNROLL passes per warp; every load of a pass (state, A, B, C, Delta, x, z, bias, D) is
// issued before any of them is used, so a warp waits for one memory round trip per pass.
template <typename Tin, typename Tout, int LPR, int UNROLL>
__global__ void __launch_bounds__(kStepThreads, 2) step_m1row(StepArgs a, unsigned rows) {
    // dependent launch: let the next launch be scheduled, then wait for the one before
    // (its writes, for instance this layer's input) before touching global memory
    grid_dep_launch();
    grid_dep_wait();
    constexpr int N = 16, NV = N / LPR / 4, RPW = 32 / LPR;
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const unsigned H = static_cast<unsigned>(a.nheads);
    const unsigned per_group = H / static_cast<unsigned>(a.ngroups);
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const unsigned nwarps = (gridDim.x * blockDim.x) >> 5;
    const unsigned per_pass = RPW * UNROLL;
    for (unsigned base = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * per_pass; base < rows;
         base += nwarps * per_pass) {
        float4 hv[UNROLL][NV], av[UNROLL][NV];
        float bv[UNROLL][NV][4], cv[UNROLL][NV][4];
        float dtr[UNROLL], xr[UNROLL], zr[UNROLL], bias[UNROLL], dsk[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const unsigned r0 = base + u * RPW + sub;
            const unsigned r = r0 < rows ? r0 : rows - 1;  // past the end: reread the last row
            const unsigned b = r / H, hd = r - b * H;
            const size_t bc = (static_cast<size_t>(b) * a.ngroups + hd / per_group) * N;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int q = li + v * LPR;  // float4 group of the row: states 4q .. 4q + 3
                hv[u][v] = __ldcs(reinterpret_cast<const float4*>(a.state + static_cast<size_t>(r) * N) + q);
                av[u][v] = __ldg(reinterpret_cast<const float4*>(a.A + static_cast<size_t>(hd) * N) + q);
                load4_f32(Bp + bc + 4 * q, bv[u][v]);
                load4_f32(Cp + bc + 4 * q, cv[u][v]);
            }
            dtr[u] = to_f32(DT[r]);
            xr[u] = to_f32(X[r]);
            zr[u] = Z ? to_f32(Z[r]) : 0.f;
            bias[u] = a.dt_bias ? a.dt_bias[hd] : 0.f;
            dsk[u] = a.D ? a.D[hd] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const unsigned r = base + u * RPW + sub;
            const float v = dtr[u] + bias[u];
            const float dt = a.dt_softplus ? softplus_accurate(v) : v;
            const float dx = dt * xr[u];
            float acc = 0.f;
#pragma unroll
            for (int g = 0; g < NV; ++g) {
                const float A4[4] = {av[u][g].x, av[u][g].y, av[u][g].z, av[u][g].w};
                float h4[4] = {hv[u][g].x, hv[u][g].y, hv[u][g].z, hv[u][g].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float za = dt * A4[j];
                    const float w = a.disc == SSM_DISC_ZOH ? phi1f(za) : 1.f;
                    h4[j] = expf(za) * h4[j] + (w * dx) * bv[u][g][j];
                    acc = fmaf(cv[u][g][j], h4[j], acc);
                }
                hv[u][g] = make_float4(h4[0], h4[1], h4[2], h4[3]);
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (r < rows) {
#pragma unroll
                for (int g = 0; g < NV; ++g)
                    __stcs(reinterpret_cast<float4*>(a.state + static_cast<size_t>(r) * N) + li + g * LPR, hv[u][g]);
                if (li == 0) {
                    float yv = acc + dsk[u] * xr[u];
                    if (Z) yv *= silu_accurate(zr[u]);
                    io<Tout>::store(static_cast<Tout*>(a.y), r, yv);
                }
            }
        }
    }
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
    const int nbh_max = rows_per_cta / a.headdim + 2;
    if (a.ntok == 1) {
        const size_t smem1 = static_cast<size_t>(nbh_max) * 6 * sizeof(float);
        if (a.a_per_state)
            return launch_dependent(step_vec1<Tin, Tout, NV, LPR, UNROLL, true>, static_cast<unsigned>(grid),
                                    kStepThreads, smem1, s, a, rows_per_cta, log2p);
        return launch_dependent(step_vec1<Tin, Tout, NV, LPR, UNROLL, false>, static_cast<unsigned>(grid),
                                kStepThreads, smem1, s, a, rows_per_cta, log2p);
    }
    // several tokens: per-CTA (batch, head) table, plus the per-token step quantities when
    // they fit in 48 KB
    const size_t base = static_cast<size_t>(nbh_max) * 3 * sizeof(float);
    const size_t tabb = static_cast<size_t>(nbh_max) * 3 * a.ntok * sizeof(float);
    const int tab = base + tabb <= 48 * 1024 ? 1 : 0;
    const size_t smem = base + (tab ? tabb : 0);
    if (a.a_per_state)
        return launch_dependent(step_vec<Tin, Tout, NV, LPR, UNROLL, true>, static_cast<unsigned>(grid),
                                kStepThreads, smem, s, a, rows_per_cta, log2p, tab);
    return launch_dependent(step_vec<Tin, Tout, NV, LPR, UNROLL, false>, static_cast<unsigned>(grid),
                            kStepThreads, smem, s, a, rows_per_cta, log2p, tab);
}

template <typename Tin, typename Tout>
static cudaError_t launch_step_t(const StepArgs& a, cudaStream_t s) {
    const long long rows = static_cast<long long>(a.batch) * a.nheads * a.headdim;
    if (rows == 0) return cudaSuccess;
    if (a.ntok > 1 && !a.a_per_state) {  // several tokens: state held in registers throughout
        switch (a.dstate) {
            case 64: return launch_tok<Tin, Tout, 2>(a, rows, s);
            case 128: return launch_tok<Tin, Tout, 4>(a, rows, s);
            case 256: return launch_tok<Tin, Tout, 8>(a, rows, s);
            default: break;
        }
    }
    if (a.ntok == 1 && a.a_per_state && a.headdim == 1 && a.dstate == 16 && rows < (1LL << 31)) {
        constexpr int kL = 2, kU = 3, kRows = 32 / kL * kU;  // lanes per row, passes, rows per warp
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const long long warps = (rows + kRows - 1) / kRows;
        const long long want = (warps + kStepThreads / 32 - 1) / (kStepThreads / 32);
        const long long grid = want < 2LL * sms ? want : 2LL * sms;  // 2 CTAs per SM resident
        return launch_dependent(step_m1row<Tin, Tout, kL, kU>, static_cast<unsigned>(grid), kStepThreads, 0, s,
                                a, static_cast<unsigned>(rows));
    }
    switch (a.dstate) {
        case 16: return launch_vec<Tin, Tout, 1, 4, 4>(a, rows, s);
        case 32: return launch_vec<Tin, Tout, 2, 4, 4>(a, rows, s);
        case 64: return launch_vec<Tin, Tout, 2, 8, 4>(a, rows, s);
        case 128: return launch_vec<Tin, Tout, 4, 8, 4>(a, rows, s);
        case 256: return launch_vec<Tin, Tout, 2, 32, 4>(a, rows, s);
        default: {
            const unsigned blocks = static_cast<unsigned>((rows + 127) / 128);
            return launch_dependent(step_scalar<Tin, Tout>, blocks, 128, 0, s, a);
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
