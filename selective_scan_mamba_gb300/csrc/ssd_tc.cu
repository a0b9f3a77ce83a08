// ssd_tc.cu -- Mamba-2 chunked SSD scan on the 5th-generation tensor cores (sm_103a).
//
// ("From S4 to Mamba-3", 03/System, mamba2_minimal.py: with a scalar A per head the
// recurrence is computed as chunked decayed-attention matmuls with a carried (N, P)
// state; 04/Approach: it equals the sequential scan.)  For a chunk of Q = 64 steps and
// s_t = running sum of Delta*A_h inside the chunk:
//   Y_diag[t,p] = sum_{s<=t} (C_t . B_s) exp(s_t - s_s) w_s x_s[p]          (decayed attention)
//   Y_off[t,p]  = exp(s_t) sum_n C_t[n] h_in[p,n]                           (carried state)
//   S[n,p]      = sum_s B_s[n] exp(s_end - s_s) w_s x_s[p]                  (chunk state)
//   h_out       = exp(s_end) h_in + S^T,   y = Y_diag + Y_off + D x, gated.
//
// One CTA walks a run ("segment") of consecutive chunks of one (batch, head) and keeps
// the state in fp32 registers.  Per chunk, TMA brings the x, B, C tiles (bf16, 128-byte
// swizzle); the threads build the remaining operand tiles with 16-byte vector stores; one
// thread issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulators in TMEM).  x and B are
// used straight from the TMA tiles, as MN-major operands where the contraction runs over
// their rows:
//   MMA1  CB = C . B^T                        M=64  N=64 K=128  C, B K-major (exact bf16)
//   MMA2  Yd = M_hi . X + M_lo . X            M=64  N=64 K=64   M = CB o decay o w, split
//                                                               into two bf16 parts; X
//                                                               MN-major
//   MMA3  Yo = C . H^T                        M=64  N=64 K=128  state rounded to bf16, held
//                                                               as [n][p] (MN-major); the
//                                                               exp(s_t) row scale is
//                                                               applied in fp32 afterwards
//   MMA4  S  = B^T . F_hi + B^T . F_lo        M=128 N=64 K=64   B MN-major; F = f o X,
//                                                               f_s = exp(s_end - s_s) w_s,
//                                                               split into two bf16 parts
// A first launch ("states" mode) runs the state part only over every segment but the
// last and leaves each segment's local end state and total decay in the workspace; the
// main launch then starts segment k from h0 combined with those (state passing), so
// segments of the same sequence run in parallel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kQ = 64, kP = 64, kNs = 128;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColYd = 0, kColYo = 64, kColS = 128, kColCB = 192;

struct SsdMaps {
    CUtensorMap x, b, c;
};

// shared-memory layout (bytes); every tile 1024-byte aligned, rows of 128 bytes
constexpr int kOffX = 0;                 // [64 s][64 p] bf16 (TMA)
constexpr int kOffB = kOffX + 8192;      // [64 s][128 n] bf16, two 64-column slabs (TMA)
constexpr int kOffC = kOffB + 16384;     // [64 t][128 n] bf16, two slabs (TMA)
constexpr int kOffMh = kOffC + 16384;    // [64 t][64 s] bf16: masked decayed CB, high part
constexpr int kOffMl = kOffMh + 8192;    // [64 t][64 s] bf16: low part
constexpr int kOffHm = kOffMl + 8192;    // [128 n][64 p] bf16: carried state
constexpr int kOffFh = kOffHm + 16384;   // [64 s][64 p] bf16: f_s x_s, high part
constexpr int kOffFl = kOffFh + 8192;    // [64 s][64 p] bf16: low part
constexpr int kOffArr = kOffFl + 8192;   // cum, w, f, e: 4 x 64 floats
constexpr int kOffBar = kOffArr + 4 * kQ * 4;
constexpr int kSmemBytes = kOffBar + 64;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // + alignment slack
constexpr uint32_t kTxFull = 8192 + 2 * 16384;
constexpr uint32_t kTxState = 8192 + 16384;

// 16-byte chunk `cq` (8 bf16) of row `r` in a 128-byte-row swizzled tile
__device__ __forceinline__ int chunk_off(int r, int cq) { return r * 128 + (((cq ^ (r & 7))) << 4); }

// v = hi + lo with hi, lo bf16 (8 values -> two packed 16-byte chunks)
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        h[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        l[j] = pack_bf16x2(v[2 * j] - lo_bf16(h[j]), v[2 * j + 1] - hi_bf16(h[j]));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void unpack8(uint4 w, float* v) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = lo_bf16(a[j]);
        v[2 * j + 1] = hi_bf16(a[j]);
    }
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}


template <typename Tin, typename Tout, bool STATES>
__global__ void __launch_bounds__(kThreads, 2)
    ssd_tc_kernel(const __grid_constant__ SsdMaps maps, SsdArgs a, int nseg, float* seg_state,
                  float* seg_decay) {
    const int seg = blockIdx.x, hd = blockIdx.y, b = blockIdx.z;
    const int L = a.seqlen;
    const int nch = (L + kQ - 1) / kQ;
    const int per = (nch + nseg - 1) / nseg;
    const int cb = seg * per;
    const int ce = min(nch, cb + per);
    const int g = hd / (a.nheads / a.ngroups);
    const float Ah = a.A[hd];
    const float bias = a.dt_bias ? a.dt_bias[hd] : 0.f;
    const Tin* DT = static_cast<const Tin*>(a.dt);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* cum = reinterpret_cast<float*>(sm + kOffArr);
    float* wv = cum + kQ;
    float* fv = wv + kQ;
    float* ev = fv + kQ;
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint64_t* mma_bar = tma_bar + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, hf = warp >> 2;

    if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (tid == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.b);
        if (!STATES) prefetch_tmap(&maps.c);
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_fence_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * qd) << 16);

    // state held by this thread: h[p][n] for n = 32 qd + lane, p = 32 hf .. 32 hf + 31
    const int hn = 32 * qd + lane;
    const size_t PN = static_cast<size_t>(kP) * kNs;
    const size_t bh = static_cast<size_t>(b) * a.nheads + hd;
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = 0.f;
    if (!STATES) {
        if (a.h0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = a.h0[bh * PN + static_cast<size_t>(32 * hf + i) * kNs + hn];
        }
        // state passing over the segments before this one
        for (int j = 0; j < seg; ++j) {
            const float dec = seg_decay[bh * (nseg - 1) + j];
            const float* sl = seg_state + (bh * (nseg - 1) + j) * PN;
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = dec * h[i] + sl[static_cast<size_t>(32 * hf + i) * kNs + hn];
        }
        // carried state as the bf16 operand of MMA3: row n of Hm holds h[., n]
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 w = make_uint4(pack_bf16x2(h[8 * j], h[8 * j + 1]), pack_bf16x2(h[8 * j + 2], h[8 * j + 3]),
                                       pack_bf16x2(h[8 * j + 4], h[8 * j + 5]), pack_bf16x2(h[8 * j + 6], h[8 * j + 7]));
            *reinterpret_cast<uint4*>(sm + kOffHm + chunk_off(hn, 4 * hf + j)) = w;
        }
    }

    auto issue = [&](int c) {
        mbar_arrive_expect_tx(tma_bar, STATES ? kTxState : kTxFull);
        tma_load_4d(sm + kOffX, &maps.x, 0, hd, c * kQ, b, tma_bar);
        tma_load_4d(sm + kOffB, &maps.b, 0, g, c * kQ, b, tma_bar);
        tma_load_4d(sm + kOffB + 8192, &maps.b, 64, g, c * kQ, b, tma_bar);
        if (!STATES) {
            tma_load_4d(sm + kOffC, &maps.c, 0, g, c * kQ, b, tma_bar);
            tma_load_4d(sm + kOffC + 8192, &maps.c, 64, g, c * kQ, b, tma_bar);
        }
    };
    if (tid == 0 && cb < ce) issue(cb);

    uint32_t tma_phase = 0, mma_phase = 0;
    float log_decay = 0.f;  // sum of Delta*A over the segment (states mode)
    const float Dh = a.D ? a.D[hd] : 0.f;
    const Tin* Z = static_cast<const Tin*>(a.z);

    // raw time steps of the next chunk, fetched one chunk ahead (warp 0, two per lane)
    float dt_next[2] = {0.f, 0.f};
    auto fetch_dt = [&](int c) {
        const int t0 = c * kQ, q = min(kQ, L - t0);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int s = 2 * lane + j;
            dt_next[j] = s < q ? to_f32(DT[(static_cast<size_t>(b) * L + t0 + s) * a.nheads + hd]) : 0.f;
        }
    };
    if (warp == 0 && cb < ce) fetch_dt(cb);

    for (int c = cb; c < ce; ++c) {
        const int t0 = c * kQ;
        const int q = min(kQ, L - t0);
        float dt_raw[2] = {dt_next[0], dt_next[1]};
        if (warp == 0 && c + 1 < ce) fetch_dt(c + 1);
        mbar_wait(tma_bar, tma_phase);
        tma_phase ^= 1;

        // (a) Delta, running sums and weights of the chunk (warp 0: two steps per lane)
        if (warp == 0) {
            float d2[2], w2[2], c2[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int s = 2 * lane + j;
                float dt = 0.f;
                if (s < q) {
                    const float v = dt_raw[j] + bias;
                    dt = a.dt_softplus ? softplus_accurate(v) : v;
                }
                d2[j] = dt * Ah;
                w2[j] = a.disc == SSM_DISC_ZOH ? dt * phi1f(dt * Ah) : dt;
            }
            c2[0] = d2[0];
            c2[1] = d2[0] + d2[1];
            float run = c2[1];  // inclusive prefix of lane sums
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run += o;
            }
            const float excl = run - c2[1];
            const float last = __shfl_sync(0xffffffffu, run, 31);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int s = 2 * lane + j;
                const float cs = excl + c2[j];
                cum[s] = cs;
                wv[s] = w2[j];
                fv[s] = expf(last - cs) * w2[j];
                ev[s] = expf(cs);
            }
            if (lane == 0) log_decay += last;
        }
        __syncthreads();

        // x values this thread needs in the output epilogue (row t, 32 columns), kept in
        // registers so the stage can take the next chunk's tiles before the epilogue
        uint4 xkeep[4];
        if (!STATES) {
            const int t = 16 * qd + (lane & 15);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                xkeep[j] = *reinterpret_cast<const uint4*>(sm + kOffX + chunk_off(t, 4 * hf + j));
        }

        if (!STATES && tid == 0) {  // MMA1: CB = C . B^T
            tc::fence_after();
            const uint32_t sc = smem_u32(sm + kOffC), sb = smem_u32(sm + kOffB);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 8192 + (k & 3) * 32;
                tc::mma_bf16(tmem + kColCB, tc::desc_sw128(sc + off), tc::desc_sw128(sb + off),
                             tc::idesc_bf16(64, 64), k > 0);
            }
            tc::mma_commit(mma_bar);
        }
        // (b) F[s][p] = f_s x_s[p] as bf16 hi + lo (row s, 16 columns per thread)
        {
            const int s = tid >> 2, pq = tid & 3;
            const float f = fv[s];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int cq = 2 * pq + j;
                float v[8];
                unpack8(*reinterpret_cast<const uint4*>(sm + kOffX + chunk_off(s, cq)), v);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] *= f;
                uint4 hi, lo;
                split8(v, hi, lo);
                *reinterpret_cast<uint4*>(sm + kOffFh + chunk_off(s, cq)) = hi;
                *reinterpret_cast<uint4*>(sm + kOffFl + chunk_off(s, cq)) = lo;
            }
        }
        if (!STATES) {
            // (c) masked, decayed, weighted CB -> M_hi, M_lo (row t = 16 qd + lane for
            //     lane < 16; columns s = 32 hf .. 32 hf + 31)
            mbar_wait(mma_bar, mma_phase);
            mma_phase ^= 1;
            tc::fence_after();
            const int t = 16 * qd + (lane & 15);
            float cbv[32];
            tc::tmem_ld16(tlane + kColCB + 32 * hf, cbv);
            tc::tmem_ld16(tlane + kColCB + 32 * hf + 16, cbv + 16);
            if (lane < 16) {
                const float ct = cum[t];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float m[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = 32 * hf + 8 * j + e;
                        m[e] = (s <= t && t < q) ? cbv[8 * j + e] * expf(ct - cum[s]) * wv[s] : 0.f;
                    }
                    uint4 hi, lo;
                    split8(m, hi, lo);
                    *reinterpret_cast<uint4*>(sm + kOffMh + chunk_off(t, 4 * hf + j)) = hi;
                    *reinterpret_cast<uint4*>(sm + kOffMl + chunk_off(t, 4 * hf + j)) = lo;
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();

        if (tid == 0) {
            tc::fence_after();
            const uint32_t sx = smem_u32(sm + kOffX), sbm = smem_u32(sm + kOffB);
            if (!STATES) {
                const uint32_t smh = smem_u32(sm + kOffMh), sml = smem_u32(sm + kOffMl);
                const uint32_t idn = tc::idesc_bf16_mn(64, 64, false, true);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // MMA2: Yd = M_hi X + M_lo X
                    tc::mma_bf16(tmem + kColYd, tc::desc_sw128(smh + k * 32),
                                 tc::desc_sw128_mn(sx + k * 2048, 8192), idn, k > 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc::mma_bf16(tmem + kColYd, tc::desc_sw128(sml + k * 32),
                                 tc::desc_sw128_mn(sx + k * 2048, 8192), idn, 1);
                const uint32_t sc = smem_u32(sm + kOffC), sh = smem_u32(sm + kOffHm);
#pragma unroll
                for (int k = 0; k < 8; ++k)  // MMA3: Yo = C H^T
                    tc::mma_bf16(tmem + kColYo, tc::desc_sw128(sc + (k >> 2) * 8192 + (k & 3) * 32),
                                 tc::desc_sw128_mn(sh + k * 2048, 16384), idn, k > 0);
            }
            const uint32_t sfh = smem_u32(sm + kOffFh), sfl = smem_u32(sm + kOffFl);
            const uint32_t id4 = tc::idesc_bf16_mn(128, 64, true, true);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // MMA4: S = B^T F_hi + B^T F_lo
                tc::mma_bf16(tmem + kColS, tc::desc_sw128_mn(sbm + k * 2048, 8192),
                             tc::desc_sw128_mn(sfh + k * 2048, 8192), id4, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                tc::mma_bf16(tmem + kColS, tc::desc_sw128_mn(sbm + k * 2048, 8192),
                             tc::desc_sw128_mn(sfl + k * 2048, 8192), id4, 1);
            tc::mma_commit(mma_bar);
        }
        mbar_wait(mma_bar, mma_phase);
        mma_phase ^= 1;
        tc::fence_after();
        // every read of the stage is done: bring in the next chunk while the epilogues run
        if (tid == 0 && c + 1 < ce) issue(c + 1);

        if (!STATES) {  // (d) outputs: row t = 16 qd + lane (lane < 16), p = 32 hf .. + 31
            const int t = 16 * qd + (lane & 15);
            float yd[32], yo[32];
            tc::tmem_ld16(tlane + kColYd + 32 * hf, yd);
            tc::tmem_ld16(tlane + kColYd + 32 * hf + 16, yd + 16);
            tc::tmem_ld16(tlane + kColYo + 32 * hf, yo);
            tc::tmem_ld16(tlane + kColYo + 32 * hf + 16, yo + 16);
            if (lane < 16 && t < q) {
                const float et = ev[t];
                const size_t row = ((static_cast<size_t>(b) * L + t0 + t) * a.nheads + hd) * kP + 32 * hf;
                float out[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float xv[8];
                    unpack8(xkeep[j], xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * j + e;
                        float v = yd[i] + et * yo[i] + Dh * xv[e];
                        if (Z) v *= silu_accurate(to_f32(Z[row + i]));
                        out[i] = v;
                    }
                }
                store_row<32>(static_cast<Tout*>(a.y) + row, out, 32);
            }
        }
        {  // (e) state update: row n = 32 qd + lane, p = 32 hf .. + 31
            float sv[32];
            tc::tmem_ld16(tlane + kColS + 32 * hf, sv);
            tc::tmem_ld16(tlane + kColS + 32 * hf + 16, sv + 16);
            const float dec = expf(cum[kQ - 1]);
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = dec * h[i] + sv[i];
            if (!STATES) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 w = make_uint4(pack_bf16x2(h[8 * j], h[8 * j + 1]), pack_bf16x2(h[8 * j + 2], h[8 * j + 3]),
                                               pack_bf16x2(h[8 * j + 4], h[8 * j + 5]), pack_bf16x2(h[8 * j + 6], h[8 * j + 7]));
                    *reinterpret_cast<uint4*>(sm + kOffHm + chunk_off(hn, 4 * hf + j)) = w;
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
    }

    if (STATES) {
        float* sl = seg_state + (bh * (nseg - 1) + seg) * PN;
#pragma unroll
        for (int i = 0; i < 32; ++i) sl[static_cast<size_t>(32 * hf + i) * kNs + hn] = h[i];
        if (tid == 0) seg_decay[bh * (nseg - 1) + seg] = expf(log_decay);
    } else if (a.h_final && seg == nseg - 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) a.h_final[bh * PN + static_cast<size_t>(32 * hf + i) * kNs + hn] = h[i];
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

cudaError_t encode_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t d3);

}  // namespace

// The tensor-core path covers the Mamba-2 130m/780m layer shapes: chunk 64, headdim 64,
// dstate 128, bf16 inputs; other shapes use the CUDA-core kernels in ssd.cu.
bool ssd_tc_supported(const SsdArgs& a) {
    return a.chunk == kQ && a.headdim == kP && a.dstate == kNs && a.in_dtype == SSM_BF16 &&
           a.seqlen > 0;
}

int ssd_tc_segments(const SsdArgs& a) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int nch = (a.seqlen + kQ - 1) / kQ;
    const long long units = static_cast<long long>(a.batch) * a.nheads;
    int S = static_cast<int>((2LL * sms) / units);  // one wave at two CTAs per SM
    if (S < 1) S = 1;
    if (S > nch) S = nch;
    if (S > 64) S = 64;
    return S;
}

size_t ssd_tc_workspace_bytes(const SsdArgs& a) {
    const int S = ssd_tc_segments(a);
    const size_t units = static_cast<size_t>(a.batch) * a.nheads * (S > 1 ? S - 1 : 0);
    return ((units * kP * kNs * sizeof(float) + 255) / 256) * 256 + ((units * 4 + 255) / 256) * 256;
}

cudaError_t ssd_tc_launch(const SsdArgs& a, void* workspace, cudaStream_t s) {
    const int S = ssd_tc_segments(a);
    SsdMaps maps;
    cudaError_t e;
    const uint64_t H = a.nheads, G = a.ngroups, L = a.seqlen, Bt = a.batch;
    if ((e = encode_4d(&maps.x, a.x, kP, H, L, Bt)) != cudaSuccess) return e;
    if ((e = encode_4d(&maps.b, a.B, kNs, G, L, Bt)) != cudaSuccess) return e;
    if ((e = encode_4d(&maps.c, a.C, kNs, G, L, Bt)) != cudaSuccess) return e;
    const size_t units = static_cast<size_t>(a.batch) * a.nheads * (S > 1 ? S - 1 : 0);
    float* seg_state = static_cast<float*>(workspace);
    float* seg_decay = reinterpret_cast<float*>(
        static_cast<char*>(workspace) + ((units * kP * kNs * sizeof(float) + 255) / 256) * 256);
    auto set = [](const void* fn) {
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    };
    if (S > 1) {
        auto k = ssd_tc_kernel<bf16_t, bf16_t, true>;
        if ((e = set(reinterpret_cast<const void*>(k))) != cudaSuccess) return e;
        k<<<dim3(S - 1, a.nheads, a.batch), kThreads, kSmemAlloc, s>>>(maps, a, S, seg_state, seg_decay);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.out_dtype == SSM_BF16) {
        auto k = ssd_tc_kernel<bf16_t, bf16_t, false>;
        if ((e = set(reinterpret_cast<const void*>(k))) != cudaSuccess) return e;
        k<<<dim3(S, a.nheads, a.batch), kThreads, kSmemAlloc, s>>>(maps, a, S, seg_state, seg_decay);
    } else {
        auto k = ssd_tc_kernel<bf16_t, float, false>;
        if ((e = set(reinterpret_cast<const void*>(k))) != cudaSuccess) return e;
        k<<<dim3(S, a.nheads, a.batch), kThreads, kSmemAlloc, s>>>(maps, a, S, seg_state, seg_decay);
    }
    return cudaGetLastError();
}

namespace {
cudaError_t encode_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t d3) {
    // [d3][d2][d1][d0] bf16, box {64, 1, 64, 1}, 128-byte swizzle
    const unsigned long long dims[4] = {d0, d1, d2, d3};
    const unsigned box[4] = {64, 1, 64, 1};
    return encode_tmap_nd(map, base, 2, 4, dims, box, true);
}
}  // namespace

}  // namespace ssm
