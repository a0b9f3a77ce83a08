// scan_m1.cu -- Mamba-1 selective scan kernels (sm_103a).
//
// Computes, per channel (b, d) and state n ("From S4 to Mamba-3", 03/System,
// mamba_minimal.py: input-dependent Delta, B, C run as a time-loop scan):
//   Delta_t = softplus(delta_t + bias_d)
//   h_t[n]  = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B_t[n] x_t
//   y_t     = (sum_n C_t[n] h_t[n] + D_d x_t) * SiLU(z_t)
//
// Two kernels:
//  * m1_scan_tiled -- the fast path.  One wave of CTAs (a fixed number per SM), each
//    owning a contiguous, balanced range of channels for the whole sequence.  Time is
//    walked in tiles of T steps; every tile of x, delta, z, B and C is read from HBM
//    exactly once with 16-byte cp.async copies into a double-buffered shared-memory
//    stage.  TPC threads share a channel, each holding NS = N / TPC states in fp32
//    registers.  Per tile: (1) the channel's threads compute Delta and Delta*x for
//    their slice of the tile (softplus once per (b, d, t)) and B, C are widened to
//    fp32 once per CTA; (2) each thread runs the recurrence over the T steps with
//    packed f32x2 arithmetic and one MUFU.EX2 per state update, keeping its partial
//    C.h per step in registers; (3) the partials are reduce-scattered across the
//    channel's threads so each owns T / TPC finished outputs, to which it adds the
//    skip term, applies the gate and stores bf16/fp32 y.
//  * m1_scan_generic -- any dstate <= 256, any sequence length or alignment, ZOH:
//    one warp per channel, lanes over states, direct global loads.  Slow and simple.
#include <cuda_runtime.h>
#include <stdlib.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

// --------------------------------------------------------------------------------------
// generic path
// --------------------------------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(128) m1_scan_generic(M1Args a) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nch = a.batch * a.dim;
    if (warp >= nch) return;
    const int b = warp / a.dim, d = warp % a.dim;
    const int g = d / (a.dim / a.ngroups);
    const int N = a.dstate;
    constexpr int MAXS = 8;  // states per lane: N <= 256
    float h[MAXS], Av[MAXS];
    const size_t row = (static_cast<size_t>(b) * a.dim + d) * a.seqlen;
    const size_t bcrow = (static_cast<size_t>(b) * a.ngroups + g) * N;
#pragma unroll
    for (int j = 0; j < MAXS; ++j) {
        int n = lane + 32 * j;
        h[j] = (n < N && a.h0) ? a.h0[(static_cast<size_t>(b) * a.dim + d) * N + n] : 0.f;
        Av[j] = n < N ? a.A[static_cast<size_t>(d) * N + n] : 0.f;
    }
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* DL = static_cast<const Tin*>(a.delta);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    for (int t = 0; t < a.seqlen; ++t) {
        float v = io<Tin>::load(DL, row + t) + bias;
        float dt = a.delta_softplus ? softplus_accurate(v) : v;
        float xt = io<Tin>::load(X, row + t);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < MAXS; ++j) {
            int n = lane + 32 * j;
            if (n < N) {
                size_t bc = (bcrow + n) * a.seqlen + t;
                float za = dt * Av[j];
                float w = a.disc == SSM_DISC_ZOH ? dt * phi1f(za) : dt;
                h[j] = expf(za) * h[j] + w * io<Tin>::load(Bp, bc) * xt;
                acc += io<Tin>::load(Cp, bc) * h[j];
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            float yv = acc + Dd * xt;
            if (Z) yv *= silu_accurate(io<Tin>::load(Z, row + t));
            io<Tout>::store(static_cast<Tout*>(a.y), row + t, yv);
        }
    }
    if (a.h_final) {
#pragma unroll
        for (int j = 0; j < MAXS; ++j) {
            int n = lane + 32 * j;
            if (n < N) a.h_final[(static_cast<size_t>(b) * a.dim + d) * N + n] = h[j];
        }
    }
}

// --------------------------------------------------------------------------------------
// fast tiled path
// --------------------------------------------------------------------------------------
// B and C are kept widened to fp32 as [pair][t][N]; the 16-byte groups of four states in
// row t are XOR-swizzled by (t / 8) % 4 so that the transposing writes of step (1b) do
// not pile onto a few banks, while every thread still reads its states as float4.
template <int N>
__device__ __forceinline__ int bc_col(int t, int n) {
    return ((((n >> 2) ^ ((t >> 3) & 3)) & ((N >> 2) - 1)) << 2) | (n & 3);
}

template <typename Tin, typename Tout, int TPC, int NS, int T, bool FAST>
__global__ void __launch_bounds__(kM1MaxThreads) m1_scan_tiled(M1Args a) {
    constexpr int N = TPC * NS;
    constexpr int ES = static_cast<int>(sizeof(Tin));
    constexpr int VEC = 16 / ES;              // elements per 16-byte vector
    constexpr int ROWB = T * ES;              // bytes of one tile row
    constexpr int CHUNKS = ROWB / 16;         // 16-byte copies per tile row
    constexpr int TO = T / TPC;               // outputs owned per thread per tile
    constexpr int DTXS = T + 1;               // float2 row stride of (Delta, Delta*x)
    constexpr int LOG2TPC = TPC == 1 ? 0 : (TPC == 2 ? 1 : (TPC == 4 ? 2 : 3));
    static_assert(N == 16, "the tiled path is built for dstate = 16");
    static_assert(ROWB % 16 == 0 && TO % VEC == 0 && TO % 8 == 0, "tile shape");
    static_assert(NS % 4 == 0, "states per thread must be a multiple of 4");

    const int nch_total = a.batch * a.dim;
    const int c0 = static_cast<int>((static_cast<long long>(blockIdx.x) * nch_total) / gridDim.x);
    const int c1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * nch_total) / gridDim.x);
    const int nch = c1 - c0;            // channels owned by this CTA (<= a.cpb_max)
    const int cpb = a.cpb_max;
    const int per_group = a.dim / a.ngroups;
    const int pair0 = (c0 / a.dim) * a.ngroups + (c0 % a.dim) / per_group;
    const int pair_last = nch > 0 ? ((c1 - 1) / a.dim) * a.ngroups + ((c1 - 1) % a.dim) / per_group
                                  : pair0;
    const int npairs = pair_last - pair0 + 1;  // <= kM1MaxPairs (checked on the host)
    const bool has_z = a.z != nullptr;

    extern __shared__ __align__(16) unsigned char smem[];
    // stage layout: X[cpb][T], DL[cpb][T], Z[cpb][T], B[np][N][T], C[np][N][T] (Tin)
    const int stage_bytes = (3 * cpb + 2 * kM1MaxPairs * N) * ROWB;
    unsigned char* stage0 = smem;
    unsigned char* stage1 = smem + stage_bytes;
    float2* dtx = reinterpret_cast<float2*>(smem + 2 * stage_bytes);
    // B/C rows are read as float4: start them on a 16-byte boundary whatever cpb is
    const int dtx_bytes = (cpb * DTXS * static_cast<int>(sizeof(float2)) + 15) & ~15;
    float* Bf = reinterpret_cast<float*>(smem + 2 * stage_bytes + dtx_bytes);  // [np][T][N], swizzled
    float* Cf = Bf + kM1MaxPairs * T * N;

    const int tid = threadIdx.x;
    const int gi = tid % TPC;        // state slice
    const bool active = tid / TPC < nch;
    const int c = active ? tid / TPC : 0;  // local channel (idle threads shadow channel 0)
    const int ch = c0 + (active ? c : 0);
    const int b = ch / a.dim, d = ch % a.dim;
    const int pr = (b * a.ngroups + d / per_group) - pair0;
    const int L = a.seqlen;
    const int ntiles = (L + T - 1) / T;

    // ---- issue the copies of one tile into a stage --------------------------------------
    auto issue_tile = [&](int k, unsigned char* st) {
        const int t0 = k * T;
        const int rows_xdz = (has_z ? 3 : 2) * nch;
        const int rows = rows_xdz + 2 * npairs * N;
        const int left = (L - t0) * ES;  // bytes left in each row from t0
        for (int i = tid; i < rows * CHUNKS; i += blockDim.x) {
            const int r = i / CHUNKS, q = i % CHUNKS;
            const unsigned char* src;
            unsigned char* dst;
            if (r < rows_xdz) {
                const int which = r / nch, rc = r % nch;
                const void* base = which == 0 ? a.x : (which == 1 ? a.delta : a.z);
                src = static_cast<const unsigned char*>(base) +
                      (static_cast<size_t>(c0 + rc) * L) * ES;
                dst = st + (which * cpb + rc) * ROWB;
            } else {
                const int rr = r - rows_xdz;
                const int which = rr / (npairs * N), pn = rr % (npairs * N);
                const void* base = which == 0 ? a.B : a.C;
                src = static_cast<const unsigned char*>(base) +
                      (static_cast<size_t>(pair0) * N + pn) * L * ES;
                dst = st + (3 * cpb + which * kM1MaxPairs * N + pn) * ROWB;
            }
            const int off = q * 16;
            int nb = left - off;
            nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
            const unsigned char* sp = src + (nb > 0 ? static_cast<size_t>(t0) * ES + off : 0);
            cp_async16(dst + off, sp, nb);
        }
    };

    // ---- per-thread constants -----------------------------------------------------------
    float h[NS], A2[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const int n = gi * NS + j;
        h[j] = (active && a.h0) ? a.h0[static_cast<size_t>(ch) * N + n] : 0.f;
        const float av = a.A[static_cast<size_t>(d) * N + n];
        A2[j] = FAST ? av * SSM_LOG2E : av;   // exp(dt*A) = exp2(dt*A*log2 e)
    }
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;
    // byte offsets of this thread's float4 groups inside a swizzled B/C row, per swizzle key
    int colb[4][NS / 4];
#pragma unroll
    for (int key = 0; key < 4; ++key)
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) colb[key][q] = bc_col<N>(key * 8, gi * NS + 4 * q);

    if (ntiles > 0) issue_tile(0, stage0);
    cp_async_commit();

    for (int k = 0; k < ntiles; ++k) {
        unsigned char* st = (k & 1) ? stage1 : stage0;
        if (k + 1 < ntiles) issue_tile(k + 1, (k & 1) ? stage0 : stage1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();  // tile k resident for every thread

        const int t0 = k * T;
        const Tin* Xs = reinterpret_cast<const Tin*>(st);
        const Tin* Ds = reinterpret_cast<const Tin*>(st + cpb * ROWB);
        const Tin* Zs = reinterpret_cast<const Tin*>(st + 2 * cpb * ROWB);
        const Tin* Bs = reinterpret_cast<const Tin*>(st + 3 * cpb * ROWB);
        const Tin* Cs = Bs + kM1MaxPairs * N * T;
        const int tb = gi * TO;  // first step of this thread's slice

        // (1a) Delta and Delta*x for this thread's slice of its channel's tile
        if (active) {
#pragma unroll
            for (int i0 = 0; i0 < TO; i0 += VEC) {
                float dv[VEC], xv[VEC];
                load_f32<VEC>(Ds + c * T + tb + i0, dv);
                load_f32<VEC>(Xs + c * T + tb + i0, xv);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const float v = dv[i] + bias;
                    float dt = a.delta_softplus ? (FAST ? softplus_fast(v) : softplus_accurate(v)) : v;
                    dt = (t0 + tb + i0 + i < L) ? dt : 0.f;   // padded steps leave h unchanged
                    dtx[c * DTXS + tb + i0 + i] = make_float2(dt, dt * xv[i]);
                }
            }
        }
        // (1b) B, C widened to fp32, transposed to [pair][t][n]: one 16-byte chunk (VEC
        // consecutive steps of one state row) per work item
        for (int i = tid; i < npairs * N * CHUNKS; i += blockDim.x) {
            const int row = i / CHUNKS, q = i % CHUNKS;  // row = p * N + n
            const int p = row / N, n = row % N;
            float bv[VEC], cv[VEC];
            load_f32<VEC>(Bs + row * T + q * VEC, bv);
            load_f32<VEC>(Cs + row * T + q * VEC, cv);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int t = q * VEC + j;
                Bf[(p * T + t) * N + bc_col<N>(t, n)] = bv[j];
                Cf[(p * T + t) * N + bc_col<N>(t, n)] = cv[j];
            }
        }
        __syncthreads();

        // (2) the recurrence over the tile
        float part[T];
        {
            const float2* drow = dtx + c * DTXS;
            const unsigned char* Bb = reinterpret_cast<const unsigned char*>(Bf + pr * T * N);
            const unsigned char* Cb = reinterpret_cast<const unsigned char*>(Cf + pr * T * N);
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const float2 dd = drow[t];
                const int key = (t >> 3) & 3;
                float2 acc = make_float2(0.f, 0.f);
                const float2 dt2 = make_float2(dd.x, dd.x);
                const float2 dx2 = make_float2(dd.y, dd.y);
#pragma unroll
                for (int q = 0; q < NS / 4; ++q) {
                    const float4 bv = *reinterpret_cast<const float4*>(Bb + t * N * 4 + colb[key][q] * 4);
                    const float4 cv = *reinterpret_cast<const float4*>(Cb + t * N * 4 + colb[key][q] * 4);
                    float2 z0, z1;
                    if (FAST) {
                        z0 = mul2(dt2, make_float2(A2[4 * q], A2[4 * q + 1]));
                        z1 = mul2(dt2, make_float2(A2[4 * q + 2], A2[4 * q + 3]));
                        z0 = make_float2(ex2_approx(z0.x), ex2_approx(z0.y));
                        z1 = make_float2(ex2_approx(z1.x), ex2_approx(z1.y));
                    } else {
                        z0 = make_float2(expf(dd.x * A2[4 * q]), expf(dd.x * A2[4 * q + 1]));
                        z1 = make_float2(expf(dd.x * A2[4 * q + 2]), expf(dd.x * A2[4 * q + 3]));
                    }
                    const float2 u0 = mul2(dx2, make_float2(bv.x, bv.y));
                    const float2 u1 = mul2(dx2, make_float2(bv.z, bv.w));
                    const float2 h0 = fma2(z0, make_float2(h[4 * q], h[4 * q + 1]), u0);
                    const float2 h1 = fma2(z1, make_float2(h[4 * q + 2], h[4 * q + 3]), u1);
                    h[4 * q] = h0.x;
                    h[4 * q + 1] = h0.y;
                    h[4 * q + 2] = h1.x;
                    h[4 * q + 3] = h1.y;
                    acc = fma2(make_float2(cv.x, cv.y), h0, acc);
                    acc = fma2(make_float2(cv.z, cv.w), h1, acc);
                }
                part[t] = acc.x + acc.y;
            }
        }

        // (3) reduce-scatter the partial outputs across the channel's TPC threads; in each
        // round the kept half moves to the front so that indices stay compile-time.
#pragma unroll
        for (int r = 0; r < LOG2TPC; ++r) {
            const int half = T >> (r + 1);
            const int bit = TPC >> (r + 1);
            const bool keep_lo = (gi & bit) == 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float lo = part[i], hi = part[i + half];
                const float send = keep_lo ? hi : lo;
                const float recv = __shfl_xor_sync(0xffffffffu, send, bit);
                part[i] = (keep_lo ? lo : hi) + recv;
            }
        }
        // this thread now owns steps tb .. tb+TO-1 of channel c: skip term, gate, store
        if (active) {
            float yv[TO];
#pragma unroll
            for (int i0 = 0; i0 < TO; i0 += VEC) {
                float xv[VEC], zv[VEC];
                load_f32<VEC>(Xs + c * T + tb + i0, xv);
                if (has_z) load_f32<VEC>(Zs + c * T + tb + i0, zv);
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    float v = part[i0 + i] + Dd * xv[i];
                    if (has_z) v *= FAST ? silu_fast(zv[i]) : silu_accurate(zv[i]);
                    yv[i0 + i] = v;
                }
            }
            Tout* yrow = static_cast<Tout*>(a.y) + static_cast<size_t>(ch) * L + t0 + tb;
            store_row<TO>(yrow, yv, L - (t0 + tb));
        }
        __syncthreads();  // stage k and the dtx/Bf/Cf buffers are free again
    }

    if (active && a.h_final) {
#pragma unroll
        for (int j = 0; j < NS; ++j) a.h_final[static_cast<size_t>(ch) * N + gi * NS + j] = h[j];
    }
}

// --------------------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------------------
template <typename Tin, typename Tout>
static cudaError_t launch_generic(const M1Args& a, cudaStream_t s) {
    const long long warps = static_cast<long long>(a.batch) * a.dim;
    const int threads = 128;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    m1_scan_generic<Tin, Tout><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
    return cudaGetLastError();
}

int m1_tile_steps(ssm_dtype in_dtype) { return in_dtype == SSM_BF16 ? 64 : 32; }

size_t m1_tiled_smem_bytes(int cpb, int N, int T, size_t es) {
    const size_t rowb = static_cast<size_t>(T) * es;
    const size_t stage = (3 * static_cast<size_t>(cpb) + 2 * kM1MaxPairs * N) * rowb;
    const size_t dtx = (static_cast<size_t>(cpb) * (T + 1) * sizeof(float2) + 15) & ~size_t(15);
    const size_t bcf = 2 * static_cast<size_t>(kM1MaxPairs) * T * N * sizeof(float);
    return 2 * stage + dtx + bcf;
}

template <typename Tin, typename Tout, int TPC, int NS, int T, bool FAST>
struct TiledKernel {
    static void* fn() { return reinterpret_cast<void*>(m1_scan_tiled<Tin, Tout, TPC, NS, T, FAST>); }
    static cudaError_t launch(const M1Args& a, const M1Plan& p, cudaStream_t s) {
        m1_scan_tiled<Tin, Tout, TPC, NS, T, FAST>
            <<<p.grid, ((p.cpb_max * TPC + 31) / 32) * 32, p.smem, s>>>(a);
        return cudaGetLastError();
    }
};

// Dispatch on (in dtype, out dtype, threads per channel); F gets the TiledKernel type.
template <typename F>
static cudaError_t dispatch_tiled(const M1Args& a, int tpc, F&& f) {
    if (a.in_dtype == SSM_BF16) {
        if (a.out_dtype == SSM_BF16) {
            if (tpc == 1) return f(TiledKernel<bf16_t, bf16_t, 1, 16, 64, true>{});
            if (tpc == 2) return f(TiledKernel<bf16_t, bf16_t, 2, 8, 64, true>{});
            if (tpc == 4) return f(TiledKernel<bf16_t, bf16_t, 4, 4, 64, true>{});
        } else {
            if (tpc == 1) return f(TiledKernel<bf16_t, float, 1, 16, 64, true>{});
            if (tpc == 2) return f(TiledKernel<bf16_t, float, 2, 8, 64, true>{});
            if (tpc == 4) return f(TiledKernel<bf16_t, float, 4, 4, 64, true>{});
        }
    } else {
        if (a.out_dtype == SSM_BF16) {
            if (tpc == 2) return f(TiledKernel<float, bf16_t, 2, 8, 32, false>{});
            if (tpc == 4) return f(TiledKernel<float, bf16_t, 4, 4, 32, false>{});
        } else {
            if (tpc == 2) return f(TiledKernel<float, float, 2, 8, 32, false>{});
            if (tpc == 4) return f(TiledKernel<float, float, 4, 4, 32, false>{});
        }
    }
    return cudaErrorInvalidValue;
}


// Chooses the kernel and its launch.  The tiled path needs dstate = 16, the default
// discretisation, 16-byte aligned rows and at most kM1MaxPairs B/C rows per CTA; it runs
// as one wave: grid = (co-resident CTAs per SM) x SMs, channels split evenly.
cudaError_t m1_plan(const M1Args& a, M1Plan* plan) {
    plan->kind = M1Plan::kGeneric;
    plan->tpc = 0;
    plan->grid = 0;
    plan->cpb_max = 0;
    plan->smem = 0;
    const size_t es = a.in_dtype == SSM_BF16 ? 2 : 4;
    const size_t es_out = a.out_dtype == SSM_BF16 ? 2 : 4;
    // rows of every input and of y must be whole 16-byte vectors (cp.async copies in,
    // 16-byte stores out)
    const bool aligned = (static_cast<size_t>(a.seqlen) * es) % 16 == 0 &&
                         (static_cast<size_t>(a.seqlen) * es_out) % 16 == 0;
    if (a.dstate != 16 || a.disc != SSM_DISC_EXP_EULER || !aligned || a.seqlen == 0 ||
        (a.kernel != SSM_SCAN_KERNEL_AUTO && a.kernel != SSM_SCAN_KERNEL_TILED))
        return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int nch = a.batch * a.dim;
    const int T = m1_tile_steps(a.in_dtype);
    int tpc = a.tpc ? a.tpc : (a.in_dtype == SSM_BF16 ? 2 : 4);
    if (a.in_dtype != SSM_BF16 && tpc == 1) tpc = 2;
    int per_sm = 2;
    const int per_group = a.dim / a.ngroups;
    for (; per_sm >= 1; --per_sm) {
        int grid = per_sm * sms;
        if (grid > nch) grid = nch;
        int cpb = (nch + grid - 1) / grid;
        if (cpb * tpc > kM1MaxThreads) continue;
        // cpb consecutive channels cross at most one (batch, group) boundary when
        // cpb <= per_group, so a CTA then touches at most kM1MaxPairs B/C rows
        if (cpb > per_group) continue;
        const size_t smem = m1_tiled_smem_bytes(cpb, 16, T, es);
        M1Plan p{M1Plan::kTiled, tpc, grid, cpb, smem};
        int max_smem = 0;
        e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        if (smem > static_cast<size_t>(max_smem)) continue;
        int resident = 0;
        M1Args dummy = a;
        e = dispatch_tiled(dummy, tpc, [&](auto k) -> cudaError_t {
            using K = decltype(k);
            cudaError_t r = set_smem_attr(reinterpret_cast<const void*>(K::fn()), static_cast<int>(smem));
            if (r != cudaSuccess) return r;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &resident, K::fn(), ((cpb * tpc + 31) / 32) * 32, smem);
        });
        if (e != cudaSuccess) return e;
        if (resident < per_sm) continue;
        *plan = p;
        return cudaSuccess;
    }
    return cudaSuccess;  // nothing fits: generic path
}

cudaError_t m1_launch(const M1Args& a, const M1Plan& plan, cudaStream_t s) {
    if (plan.kind == M1Plan::kGeneric) {
        if (a.in_dtype == SSM_BF16)
            return a.out_dtype == SSM_BF16 ? launch_generic<bf16_t, bf16_t>(a, s)
                                           : launch_generic<bf16_t, float>(a, s);
        return a.out_dtype == SSM_BF16 ? launch_generic<float, bf16_t>(a, s)
                                       : launch_generic<float, float>(a, s);
    }
    M1Args b = a;
    b.cpb_max = plan.cpb_max;
    return dispatch_tiled(b, plan.tpc, [&](auto k) { return decltype(k)::launch(b, plan, s); });
}

}  // namespace ssm
