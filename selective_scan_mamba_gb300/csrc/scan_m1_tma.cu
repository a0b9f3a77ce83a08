// scan_m1_tma.cu -- Mamba-1 selective scan, bf16-input fast path with TMA staging.
//
// Same mathematics as scan_m1.cu ("From S4 to Mamba-3", 03/System, mamba_minimal.py):
//   h_t[n] = exp(Delta_t A[d,n]) h_{t-1}[n] + Delta_t B_t[n] x_t,
//   y_t = (C_t . h_t + D x_t) * SiLU(z_t),  Delta_t = softplus(delta_t + bias_d).
//
// Work split: one wave of CTAs, each owning a balanced, contiguous range of channels
// (b, d) for the whole sequence; TPC threads per channel with NS = 16 / TPC states
// each in fp32 registers.  Time advances in tiles of 64 steps:
//   * one thread issues 2-D TMA copies of the tile (x, delta, z rows of the CTA's
//     channels; B, C rows of the (batch, group) pairs they use) into a 128-byte
//     swizzled, double-buffered shared stage; completion is an mbarrier transaction
//     count, so the tile after next is already in flight while this one is computed;
//   * each channel's threads compute (Delta, Delta, Delta*x, Delta*x) for their share
//     of the steps (softplus once per (b, d, t)), and B, C are widened to fp32 once
//     per CTA;
//   * each thread runs the recurrence with f32x2 arithmetic and one MUFU.EX2 per state
//     update, keeping its partial C.h per step in registers;
//   * partials are reduce-scattered across the channel's threads with shuffles; each
//     thread adds the skip term, applies the gate and stores 16-byte vectors of y.
// Every input byte is read from HBM once; y is written once.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdlib.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kT = 64;          // steps per tile (128 bytes of bf16 per row)
constexpr int kN = 16;          // dstate of this path
constexpr int kStages = 2;
constexpr int kRowB = kT * 2;   // bytes per staged row
constexpr int kDtxS = kT + 1;   // float2 row stride of (dt, dt*x)

struct TmaMaps {
    CUtensorMap x, dl, z, b, c;
};

__host__ __device__ inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

// shared-memory layout (bytes), all offsets 1024-byte aligned where TMA writes
struct Layout {
    int cb;        // staged rows per tensor (cpb rounded up to 8)
    int x, dl, z, b, c, stage;
    int dtx, bars, total;
    __host__ __device__ Layout(int cpb) {
        cb = round_up(cpb, 8);
        x = 0;
        dl = x + cb * kRowB;
        z = dl + cb * kRowB;
        b = z + cb * kRowB;
        c = b + kM1MaxPairs * kN * kRowB;
        stage = c + kM1MaxPairs * kN * kRowB;
        dtx = kStages * stage;
        bars = dtx + round_up(cpb * kDtxS * 8, 16);
        total = bars + 64;
    }
};

// (dt, dt*x) pairs: element (c, t) at c * kDtxS + dtx_col(t).  The XOR of bits 2-3 of t
// with t / 16 spreads the four 16-step blocks written by a channel's four threads over
// different banks; with the odd row stride, the channels of a half-warp never collide.
__device__ __forceinline__ int dtx_col(int t) { return t ^ (((t >> 4) & 3) << 2); }

// 8 bf16 values of row `row`, 16-byte chunk `chunk` of a swizzled tile
__device__ __forceinline__ void load8(const unsigned char* tile, int row, int chunk, float* out) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128(row, chunk * 16));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        out[2 * j] = lo_bf16(w[j]);
        out[2 * j + 1] = hi_bf16(w[j]);
    }
}

template <typename Tout, int TPC, int NS>
__global__ void __launch_bounds__(kM1MaxThreads) m1_scan_tma(const __grid_constant__ TmaMaps maps,
                                                             M1Args a) {
    constexpr int TO = kT / TPC;  // steps owned per thread in the prologue/epilogue
    constexpr int LOG2TPC = TPC == 1 ? 0 : (TPC == 2 ? 1 : (TPC == 4 ? 2 : 3));
    static_assert(TPC * NS == kN && NS % 4 == 0 && TO % 8 == 0, "tile shape");

    const int nch_total = a.batch * a.dim;
    const int c0 = static_cast<int>((static_cast<long long>(blockIdx.x) * nch_total) / gridDim.x);
    const int c1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * nch_total) / gridDim.x);
    const int nch = c1 - c0;
    const Layout lay(a.cpb_max);
    const int per_group = a.dim / a.ngroups;
    const int pair0 = (c0 / a.dim) * a.ngroups + (c0 % a.dim) / per_group;
    const int pair_last = ((c1 - 1) / a.dim) * a.ngroups + ((c1 - 1) % a.dim) / per_group;
    const int npairs = pair_last - pair0 + 1;
    const bool has_z = a.z != nullptr;

    extern __shared__ unsigned char smem_raw[];
    // align to 1024 bytes by an offset from the shared array itself, so that the compiler
    // still sees shared-memory pointers (and emits shared loads, not generic ones)
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float2* dtx = reinterpret_cast<float2*>(smem + lay.dtx);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);

    const int tid = threadIdx.x;
    const int gi = tid % TPC;
    const bool active = tid / TPC < nch;
    const int c = active ? tid / TPC : 0;
    const int ch = c0 + c;
    const int b = ch / a.dim, d = ch % a.dim;
    const int pr = (b * a.ngroups + d / per_group) - pair0;
    const int L = a.seqlen;
    const int ntiles = (L + kT - 1) / kT;
    const uint32_t stage_tx =
        static_cast<uint32_t>(((has_z ? 3 : 2) * lay.cb + 2 * npairs * kN) * kRowB);

    auto issue = [&](int k) {
        unsigned char* st = smem + (k % kStages) * lay.stage;
        uint64_t* bar = &full[k % kStages];
        const int t0 = k * kT;
        mbar_arrive_expect_tx(bar, stage_tx);
        tma_load_2d(st + lay.x, &maps.x, t0, c0, bar);
        tma_load_2d(st + lay.dl, &maps.dl, t0, c0, bar);
        if (has_z) tma_load_2d(st + lay.z, &maps.z, t0, c0, bar);
        for (int p = 0; p < npairs; ++p) {
            tma_load_2d(st + lay.b + p * kN * kRowB, &maps.b, t0, (pair0 + p) * kN, bar);
            tma_load_2d(st + lay.c + p * kN * kRowB, &maps.c, t0, (pair0 + p) * kN, bar);
        }
    };

    if (tid == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.dl);
        if (has_z) prefetch_tmap(&maps.z);
        prefetch_tmap(&maps.b);
        prefetch_tmap(&maps.c);
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        wait_setup(a.wait_limit);
    }
    __syncthreads();
    int last_issued = -1;  // thread 0: the last tile whose copy went out
    if (tid == 0)
        for (int k = 0; k < kStages && k < ntiles; ++k) {
            issue(k);
            last_issued = k;
        }

    // per-thread constants
    // Thread gi owns states n = gi + TPC * i (i < NS): strided, so that the B/C chunk rows
    // read by a channel's threads at one step fall in distinct 128B-swizzle phases.
    // State and A * log2(e) are kept as f32x2 pairs (i = 2k, 2k + 1).
    float2 hp[NS / 2], A2p[NS / 2];
#pragma unroll
    for (int k = 0; k < NS / 2; ++k) {
        const int n0 = gi + TPC * (2 * k), n1 = gi + TPC * (2 * k + 1);
        hp[k] = (active && a.h0) ? make_float2(a.h0[static_cast<size_t>(ch) * kN + n0],
                                               a.h0[static_cast<size_t>(ch) * kN + n1])
                                 : make_float2(0.f, 0.f);
        // exp(dt A) = exp2(dt A log2 e)
        A2p[k] = make_float2(a.A[static_cast<size_t>(d) * kN + n0] * SSM_LOG2E,
                             a.A[static_cast<size_t>(d) * kN + n1] * SSM_LOG2E);
    }
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    const float Dd = a.D ? a.D[d] : 0.f;

    for (int k = 0; k < ntiles; ++k) {
        const int s = k % kStages;
        const unsigned char* st = smem + s * lay.stage;
        mbar_wait(&full[s], (k / kStages) & 1);
        const int t0 = k * kT;
        const int tb = gi * TO;

        // (1a) (dt, dt, dt*x, dt*x) for this thread's steps of its channel
        if (active) {
#pragma unroll
            for (int q = 0; q < TO / 8; ++q) {
                float dv[8], xv[8];
                load8(st + lay.dl, c, tb / 8 + q, dv);
                load8(st + lay.x, c, tb / 8 + q, xv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = tb + 8 * q + i;
                    const float v = dv[i] + bias;
                    float dt = a.delta_softplus ? softplus_fast(v) : v;
                    dt = (t0 + t < L) ? dt : 0.f;  // padded steps leave the state unchanged
                    const float dx = dt * xv[i];
                    dtx[c * kDtxS + dtx_col(t)] = make_float2(dt, dx);
                }
            }
        }
        __syncthreads();

        // (2) recurrence over the tile.  B and C are read straight from the bf16 tile:
        // one 16-byte chunk holds 8 consecutive steps of one state, so a thread loads its
        // NS states' chunks once per 8 steps and widens each value when it is used.  The
        // (dt, dt*x) pair of step t+1 and the decays of step t+1 are produced before the
        // state update of step t (manual software pipelining).
        float part[kT];
        {
            const float2* drow = dtx + c * kDtxS;
            const unsigned char* Bt = st + lay.b;
            const unsigned char* Ct = st + lay.c;
            const int row0 = pr * kN + gi;  // state rows of this thread: row0 + TPC * i
            float2 dd = drow[dtx_col(0)];
            float2 zz[NS / 2];
#pragma unroll
            for (int j = 0; j < NS / 2; ++j) {
                const float2 e = mul2(make_float2(dd.x, dd.x), A2p[j]);
                zz[j] = make_float2(ex2_approx(e.x), ex2_approx(e.y));
            }
#pragma unroll
            for (int g8 = 0; g8 < kT / 8; ++g8) {
                uint4 bq[NS], cq[NS];
#pragma unroll
                for (int i = 0; i < NS; ++i) {
                    bq[i] = *reinterpret_cast<const uint4*>(Bt + sw128(row0 + TPC * i, g8 * 16));
                    cq[i] = *reinterpret_cast<const uint4*>(Ct + sw128(row0 + TPC * i, g8 * 16));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = g8 * 8 + j;
                    float2 ddn = dd;
                    float2 zzn[NS / 2];
                    if (t + 1 < kT) {
                        ddn = drow[dtx_col(t + 1)];
#pragma unroll
                        for (int k = 0; k < NS / 2; ++k) {
                            const float2 e = mul2(make_float2(ddn.x, ddn.x), A2p[k]);
                            zzn[k] = make_float2(ex2_approx(e.x), ex2_approx(e.y));
                        }
                    }
                    const float2 dx2 = make_float2(dd.y, dd.y);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < NS / 2; ++k) {
                        const uint32_t wb0 = (&bq[2 * k].x)[j >> 1], wb1 = (&bq[2 * k + 1].x)[j >> 1];
                        const uint32_t wc0 = (&cq[2 * k].x)[j >> 1], wc1 = (&cq[2 * k + 1].x)[j >> 1];
                        const float2 bv = (j & 1) ? make_float2(hi_bf16(wb0), hi_bf16(wb1))
                                                  : make_float2(lo_bf16(wb0), lo_bf16(wb1));
                        const float2 cv = (j & 1) ? make_float2(hi_bf16(wc0), hi_bf16(wc1))
                                                  : make_float2(lo_bf16(wc0), lo_bf16(wc1));
                        hp[k] = fma2(zz[k], hp[k], mul2(dx2, bv));
                        if (k & 1) acc1 = fma2(cv, hp[k], acc1);
                        else acc0 = fma2(cv, hp[k], acc0);
                    }
                    part[t] = (acc0.x + acc1.x) + (acc0.y + acc1.y);
                    dd = ddn;
#pragma unroll
                    for (int k = 0; k < NS / 2; ++k) zz[k] = zzn[k];
                }
            }
        }

        // (3) reduce-scatter across the channel's threads (kept half moves to the front)
#pragma unroll
        for (int r = 0; r < LOG2TPC; ++r) {
            const int half = kT >> (r + 1);
            const int bit = TPC >> (r + 1);
            const bool keep_lo = (gi & bit) == 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float lo = part[i], hi = part[i + half];
                const float recv = __shfl_xor_sync(0xffffffffu, keep_lo ? hi : lo, bit);
                part[i] = (keep_lo ? lo : hi) + recv;
            }
        }
        if (active) {
            float yv[TO];
#pragma unroll
            for (int q = 0; q < TO / 8; ++q) {
                float xv[8], zv[8];
                load8(st + lay.x, c, tb / 8 + q, xv);
                if (has_z) load8(st + lay.z, c, tb / 8 + q, zv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float v = part[8 * q + i] + Dd * xv[i];
                    if (has_z) v *= silu_fast(zv[i]);
                    yv[8 * q + i] = v;
                }
            }
            Tout* yrow = static_cast<Tout*>(a.y) + static_cast<size_t>(ch) * L + t0 + tb;
            store_row<TO>(yrow, yv, L - (t0 + tb));
        }
        __syncthreads();  // stage s and the (dt, dt*x) buffer are free again
        if (tid == 0 && k + kStages < ntiles && !wait_aborted()) {
            issue(k + kStages);
            last_issued = k + kStages;
        }
    }
    // a CTA whose waits gave up lets its copies in flight land before it exits
    if (tid == 0 && wait_aborted()) drain_ring(full, kStages, last_issued);

    if (active && a.h_final) {
#pragma unroll
        for (int k = 0; k < NS / 2; ++k) {
            a.h_final[static_cast<size_t>(ch) * kN + gi + TPC * (2 * k)] = hp[k].x;
            a.h_final[static_cast<size_t>(ch) * kN + gi + TPC * (2 * k + 1)] = hp[k].y;
        }
    }
}

template <typename Tout, int TPC>
struct TmaKernel {
    static constexpr int NS = kN / TPC;
    static const void* fn() { return reinterpret_cast<const void*>(m1_scan_tma<Tout, TPC, NS>); }
};

template <typename F>
cudaError_t dispatch(ssm_dtype out, int tpc, F&& f) {
    if (out == SSM_BF16) {
        if (tpc == 2) return f(TmaKernel<bf16_t, 2>{});
        if (tpc == 4) return f(TmaKernel<bf16_t, 4>{});
    } else {
        if (tpc == 2) return f(TmaKernel<float, 2>{});
        if (tpc == 4) return f(TmaKernel<float, 4>{});
    }
    return cudaErrorInvalidValue;
}


}  // namespace

size_t m1_tma_smem_bytes(int cpb) { return static_cast<size_t>(Layout(cpb).total) + 1024; }

// Plan for the TMA path: bf16 inputs, dstate 16, exp-Euler, rows of whole 16-byte
// vectors.  Returns kGeneric in `plan->kind` when it does not apply.
cudaError_t m1_tma_plan(const M1Args& a, M1Plan* plan) {
    plan->kind = M1Plan::kGeneric;
    const size_t es_out = a.out_dtype == SSM_BF16 ? 2 : 4;
    if (a.in_dtype != SSM_BF16 || a.dstate != kN || a.disc != SSM_DISC_EXP_EULER || a.seqlen <= 0 ||
        (static_cast<size_t>(a.seqlen) * 2) % 16 != 0 ||
        (static_cast<size_t>(a.seqlen) * es_out) % 16 != 0 ||
        (a.kernel != SSM_SCAN_KERNEL_AUTO && a.kernel != SSM_SCAN_KERNEL_TMA))
        return cudaSuccess;
    int dev = 0, sms = 0, max_smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
        return e;
    const int nch = a.batch * a.dim;
    const int tpc = a.tpc ? a.tpc : 4;
    if (tpc != 2 && tpc != 4) return cudaSuccess;  // built for 2 or 4 threads per channel
    const int per_group = a.dim / a.ngroups;
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        int grid = per_sm * sms;
        if (grid > nch) grid = nch;
        const int cpb = (nch + grid - 1) / grid;
        if (cpb * tpc > kM1MaxThreads || cpb > per_group || cpb > 256) continue;
        const size_t smem = m1_tma_smem_bytes(cpb);
        if (smem > static_cast<size_t>(max_smem)) continue;
        int resident = 0;
        const int threads = round_up(cpb * tpc, 32);
        e = dispatch(a.out_dtype, tpc, [&](auto k) -> cudaError_t {
            cudaError_t r = set_smem_attr(reinterpret_cast<const void*>(decltype(k)::fn()), static_cast<int>(smem));
            if (r != cudaSuccess) return r;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, decltype(k)::fn(),
                                                                 threads, smem);
        });
        if (e != cudaSuccess) return e;
        if (resident < per_sm && per_sm > 1) continue;
        plan->kind = M1Plan::kTma;
        plan->tpc = tpc;
        plan->grid = grid;
        plan->cpb_max = cpb;
        plan->smem = smem;
        return cudaSuccess;
    }
    return cudaSuccess;
}

cudaError_t m1_tma_launch(const M1Args& a_in, const M1Plan& plan, cudaStream_t s) {
    M1Args a = a_in;
    a.cpb_max = plan.cpb_max;
    const Layout lay(plan.cpb_max);
    const uint64_t rows = static_cast<uint64_t>(a.batch) * a.dim;
    const uint64_t bcrows = static_cast<uint64_t>(a.batch) * a.ngroups * kN;
    TmaMaps maps;
    cudaError_t e;
    if ((e = encode_tmap_2d(&maps.x, a.x, 2, a.seqlen, rows, kT, lay.cb, true)) != cudaSuccess) return e;
    if ((e = encode_tmap_2d(&maps.dl, a.delta, 2, a.seqlen, rows, kT, lay.cb, true)) != cudaSuccess)
        return e;
    if ((e = encode_tmap_2d(&maps.z, a.z ? a.z : a.x, 2, a.seqlen, rows, kT, lay.cb, true)) !=
        cudaSuccess)
        return e;
    if ((e = encode_tmap_2d(&maps.b, a.B, 2, a.seqlen, bcrows, kT, kN, true)) != cudaSuccess) return e;
    if ((e = encode_tmap_2d(&maps.c, a.C, 2, a.seqlen, bcrows, kT, kN, true)) != cudaSuccess) return e;
    const int threads = round_up(plan.cpb_max * plan.tpc, 32);
    if (a.out_dtype == SSM_BF16) {
        if (plan.tpc == 2) m1_scan_tma<bf16_t, 2, 8><<<plan.grid, threads, plan.smem, s>>>(maps, a);
        else m1_scan_tma<bf16_t, 4, 4><<<plan.grid, threads, plan.smem, s>>>(maps, a);
    } else {
        if (plan.tpc == 2) m1_scan_tma<float, 2, 8><<<plan.grid, threads, plan.smem, s>>>(maps, a);
        else m1_scan_tma<float, 4, 4><<<plan.grid, threads, plan.smem, s>>>(maps, a);
    }
    return cudaGetLastError();
}

cudaError_t m1_tma_take_wait_timeouts(unsigned int* count) {
    return take_wait_timeouts(count);
}

}  // namespace ssm
