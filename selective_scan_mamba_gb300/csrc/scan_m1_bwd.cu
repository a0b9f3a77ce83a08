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
// One launch computes everything per CTA, then a small launch sums the per-row partials:
//   - a CTA of NT threads (128; 256 at 32 threads per channel) owns NT / TPC channels of one
//     (batch, group) (TPC threads per channel, four
//     consecutive states per thread);
//   - the sequence is cut into 16-step chunks and the chunks into blocks of K chunks:
//     K = 1 while a checkpoint per chunk takes no more room than x and dy (N <= 16 in
//     bf16), else K ~ sqrt(chunks); pass 1 runs the recurrence forwards and keeps h at
//     the start of every block (coarse checkpoints, in the workspace);
//   - pass 2 takes the blocks last to first: when K > 1 it reruns the block forwards
//     from its checkpoint, keeping h at the start of each of its chunks (fine
//     checkpoints, one block's worth in the workspace), then walks the block's chunks
//     last to first: it
//     stages the chunk's inputs in shared memory, recomputes h_t over the chunk from its
//     checkpoint into a shared buffer (with the pre-gate output o_t), sums dC over the
//     CTA's channels from that buffer, walks the chunk backwards overwriting h_t by G_t
//     (h_t is dead once step t+1 has used it), then sums dB over the channels from the
//     same buffer;
//   - the CTA adds its dB, dC sums into the outputs (zeroed before the launch) with
//     float32 atomic adds, so their last bits depend on the order in which CTAs arrive;
//     dA, dD, dbias partial sums per batch row go to the workspace and the second
//     launch adds them in a fixed order.
// So the workspace is at most x plus dy in size, or two sets of checkpoints of about
// sqrt(L / 16) states per channel each, for one extra forward pass.
// The same kernels serve the Mamba-2 SSD backward: with a scalar A per head its
// recurrence is this scan over the H*P channels of the heads, A tied over a head's
// channels and states and Delta, D and the bias shared by its P channels.  A BwdView
// carries the element strides of either layout and `hp`, the channels per head; with
// hp > 1 the per-channel d(delta) is added into the head's ddt (zeroed before the
// launch) with atomic adds, and the second launch sums A over the head's channels and
// states.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kBT = 16;          // steps per chunk
// threads per CTA: 128 (four CTAs per SM); 256 at 32 threads per channel (the SSD view at
// dstate 128), where each CTA's dB/dC atomic adds then cover twice the channels
__host__ __device__ constexpr int bwd_threads(int tpc) { return tpc == 32 ? 256 : 128; }
constexpr int kBS = 4;           // states per thread
constexpr int kRow = kBT + 1;    // padded row of the per-(channel, step) tiles

struct BwdLayout {  // float offsets into dynamic shared memory (16-byte aligned blocks)
    int h, bs, cs, red, dl, dlx, xs, dout, o, sg, zz, gx, gd, total;
    __host__ __device__ BwdLayout(int cpb, int n, int nt) {
        h = 0;                                  // [kBT][nt][kBS]: h_t, then G_t
        bs = h + kBT * nt * kBS;                // [kBT][n] B
        cs = bs + kBT * n;                      // [kBT][n] C
        red = cs + kBT * n;                     // [nt][4] partial sums over channels
        dl = red + nt * 4;                      // [cpb][kRow] Delta
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
    size_t ckpt, fine, part_a, part_d, part_bias, bytes;
};

// chunks per checkpoint block: one (a checkpoint per chunk, no rerun) while those
// checkpoints, N floats per 16 steps and channel, take no more room than x and dy;
// else about the square root of the chunk count, which keeps the coarse ([row][blocks]
// [N]) and fine ([row][K][N]) checkpoints together smallest
inline int bwd_block_chunks(int nch, int N, int L, int in_bytes, int dy_bytes) {
    if (static_cast<long long>(nch) * N * 4 <= static_cast<long long>(L) * (in_bytes + dy_bytes)) return 1;
    int k = 1;
    while (k * k < nch) ++k;
    return k;
}

// float32 atomic adds into dB / dC: four consecutive states as one vector add when they
// are contiguous (16-byte aligned there: N % 4 == 0 and 16-byte aligned outputs)
__device__ __forceinline__ void red_add4(float* p, long long stride, float4 v) {
    if (stride == 1) {
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                     "f"(v.w)
                     : "memory");
    } else {
        atomicAdd(p, v.x);
        atomicAdd(p + stride, v.y);
        atomicAdd(p + 2 * stride, v.z);
        atomicAdd(p + 3 * stride, v.w);
    }
}

__host__ __device__ inline int bwd_cpb(int tpc) { return bwd_threads(tpc) / tpc; }

template <typename T>
__device__ __forceinline__ float ldf(const T* p, size_t i) {
    return io<T>::load(p, i);
}

__device__ __forceinline__ float sigmoid_fast(float v) { return rcp_approx(1.f + ex2_approx(-v * SSM_LOG2E)); }

}  // namespace

// Operands of one backward call in either layout (element strides; see the file comment).
struct BwdView {
    const void *x, *delta, *z, *B, *C, *dy;
    const float *delta_bias, *A, *D_skip, *h0, *dh_final;
    float *dx, *ddelta, *dz, *dh0;             // per (b, channel, t) / per state outputs
    float *dA, *dB, *dC, *dD, *dbias;          // reduced outputs
    int batch, dim, dstate, seqlen, ngroups, softplus;
    ssm_dtype in_dtype, dy_dtype;
    int hp;                                    // channels per head (1: Mamba-1)
    long long sxb, sxd, sxt;                   // x, z, dy, dx, dz: batch, channel, step
    long long sdb, sdh, sdt;                   // delta and its gradient: batch, head, step
    long long sbb, sbg, sbn, sbt;              // B, C, dB, dC: batch, group, state, step
    long long sah, san;                        // A: head, state (san = 0: one A per head)
};

namespace {

template <typename Tin, typename Tdy, int TPC, int NT = bwd_threads(TPC)>
__global__ void __launch_bounds__(NT, 512 / NT)
    m1_scan_bwd(BwdView a, int cps, int kb, float* ckpt, float* fine, float* part_a, float* part_d,
                float* part_bias) {
    constexpr int N = TPC * kBS;
    constexpr int CPB = NT / TPC;
    constexpr int NQ = kBT * N / 4;         // (step, 4 states) cells of a chunk
    // channel slices summed in parallel per cell (1: each thread sums whole cells)
    constexpr int SPLIT = NQ < NT ? NT / NQ : 1;
    const int L = a.seqlen, Dm = a.dim, G = a.ngroups;
    const int per_group = Dm / G;
    const int pair = blockIdx.x / cps, part_i = blockIdx.x % cps;
    const int b = pair / G, g = pair % G;
    const int l0 = static_cast<int>((static_cast<long long>(part_i) * per_group) / cps);
    const int l1 = static_cast<int>((static_cast<long long>(part_i + 1) * per_group) / cps);
    const int nchan = l1 - l0;
    const int d0 = g * per_group + l0;
    const int nch = (L + kBT - 1) / kBT;
    const int nblk = (nch + kb - 1) / kb;  // kb: chunks per checkpoint block

    extern __shared__ __align__(16) float sm[];
    const BwdLayout lay(CPB, N, NT);
    float* hbuf = sm + lay.h;
    const int tid = threadIdx.x;
    const int c = tid / TPC, gi = tid % TPC;
    const bool active = c < nchan;
    const int d = d0 + (active ? c : 0);
    const size_t row = static_cast<size_t>(b) * Dm + d;  // (b, d)
    const Tin* X = static_cast<const Tin*>(a.x);
    const Tin* DL = static_cast<const Tin*>(a.delta);
    const Tin* Z = static_cast<const Tin*>(a.z);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const Tdy* DY = static_cast<const Tdy*>(a.dy);
    const long long bc_base = b * a.sbb + g * a.sbg;
    // element (b, channel cc of the CTA, step t) of x, z, dy, dx, dz and of delta
    // head of each of the CTA's channels (the channel itself when hp = 1), once
    __shared__ int s_head[CPB];
    for (int cc = tid; cc < CPB; cc += NT) s_head[cc] = (d0 + cc) / a.hp;
    __syncthreads();
    auto xi = [&](int cc, int t) { return b * a.sxb + (d0 + cc) * a.sxd + t * a.sxt; };
    auto di = [&](int cc, int t) { return b * a.sdb + s_head[cc] * a.sdh + t * a.sdt; };
    // staging order: consecutive threads take consecutive addresses of the layout
    const bool tfast = a.sxt == 1, bt_fast = a.sbt == 1;

    float Av[kBS], A2[kBS];  // A, and A log2(e) for the exponentials
#pragma unroll
    for (int i = 0; i < kBS; ++i) {
        Av[i] = a.A[(d / a.hp) * a.sah + (kBS * gi + i) * a.san];
        A2[i] = Av[i] * SSM_LOG2E;
    }
    const float Dd = a.D_skip ? a.D_skip[d / a.hp] : 0.f;

    // stage Delta (and Delta x, x, sigmoid, dL/do, z) of the CTA's channels and B (C)
    // for a chunk
    auto stage = [&](int t0, int tl, bool full) {
        for (int j = tid; j < CPB * kBT; j += NT) {
            const int cc = tfast ? j / kBT : j % CPB, t = tfast ? j % kBT : j / CPB;
            float dl = 0.f, xv = 0.f, sgv = 1.f, dov = 0.f, zv = 0.f;
            if (cc < nchan && t < tl) {
                const long long i = xi(cc, t0 + t);
                const float v = ldf(DL, di(cc, t0 + t)) + (a.delta_bias ? a.delta_bias[s_head[cc]] : 0.f);
                dl = a.softplus ? softplus_fast(v) : v;
                xv = ldf(X, i);
                if (full) {
                    sgv = a.softplus ? sigmoid_fast(v) : 1.f;
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
        for (int j = tid; j < N * kBT; j += NT) {
            const int n = bt_fast ? j / kBT : j % N, t = bt_fast ? j % kBT : j / N;
            const long long i = bc_base + n * a.sbn + (t0 + t) * a.sbt;
            sm[lay.bs + t * N + n] = t < tl ? ldf(Bp, i) : 0.f;
            if (full) sm[lay.cs + t * N + n] = t < tl ? ldf(Cp, i) : 0.f;
        }
    };
    // sum over the CTA's channels of w[channel][t] * buf[t][channel][n] for every (t, n) of
    // the chunk, added into dst (dB or dC) at step t0 + t: cell q = (t, 4 states) per
    // thread slice, SPLIT slices of the channels, then the slices added
    auto channel_sum = [&](int wofs, float* dst, int t0, int tl) {
      for (int q0 = 0; q0 < (NQ > NT ? NQ : 1); q0 += NT) {
        const int q = NQ > NT ? q0 + tid : tid % NQ, sl = NQ > NT ? 0 : tid / NQ;
        const int t = q / (N / 4), n4 = q % (N / 4);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < tl) {
            for (int cc = sl; cc < nchan; cc += SPLIT) {
                const float w = sm[wofs + cc * kRow + t];
                const float4 v = *reinterpret_cast<const float4*>(hbuf + (t * NT + cc * TPC + n4) * kBS);
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
        if (sl == 0 && t < tl) red_add4(dst + bc_base + 4 * n4 * a.sbn + (t0 + t) * a.sbt, a.sbn, s);
      }
    };

    // forward over chunks [c0, c1) from h, storing h at the start of chunk ch in
    // dst + (ch - c0) * every N when (ch - c0) % every == 0, dst rows [row][.][N]
    float h[kBS];
    auto forward = [&](int c0, int c1, float* dst, int per_row, int every) {
      for (int ch = c0; ch < c1; ++ch) {
        const int t0 = ch * kBT, tl = min(kBT, L - t0);
        if (active && (ch - c0) % every == 0)
            *reinterpret_cast<float4*>(dst + (row * per_row + (ch - c0) / every) * N + kBS * gi) =
                make_float4(h[0], h[1], h[2], h[3]);
        __syncthreads();
        stage(t0, tl, false);
        __syncthreads();
        for (int t = 0; t < tl; ++t) {
            const float dl = sm[lay.dl + c * kRow + t], dlx = sm[lay.dlx + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float2 dl2 = make_float2(dl, dl), dx2 = make_float2(dlx, dlx);
            const float2 b01 = make_float2(bv.x, bv.y), b23 = make_float2(bv.z, bv.w);
            const float2 e01 = mul2(dl2, make_float2(A2[0], A2[1])), e23 = mul2(dl2, make_float2(A2[2], A2[3]));
            float2 h01 = make_float2(h[0], h[1]), h23 = make_float2(h[2], h[3]);
            h01 = fma2(make_float2(ex2_approx(e01.x), ex2_approx(e01.y)), h01, mul2(dx2, b01));
            h23 = fma2(make_float2(ex2_approx(e23.x), ex2_approx(e23.y)), h23, mul2(dx2, b23));
            h[0] = h01.x; h[1] = h01.y; h[2] = h23.x; h[3] = h23.y;
        }
      }
    };
    // pass 1: coarse checkpoints, h at the start of every block
#pragma unroll
    for (int i = 0; i < kBS; ++i) h[i] = (active && a.h0) ? a.h0[row * N + kBS * gi + i] : 0.f;
    forward(0, nch, ckpt, nblk, kb);

    // pass 2: blocks last to first, and in each the chunks last to first
    float gcar[kBS], dAacc[kBS];
#pragma unroll
    for (int i = 0; i < kBS; ++i) {
        gcar[i] = (active && a.dh_final) ? a.dh_final[row * N + kBS * gi + i] : 0.f;
        dAacc[i] = 0.f;
    }
    float dDacc = 0.f, dbacc = 0.f;
    for (int blk = nblk - 1; blk >= 0; --blk) {
      const int cb0 = blk * kb, cb1 = min(nch, cb0 + kb);
      {  // fine checkpoints of the block, from its coarse one
          const float4 v = active ? *reinterpret_cast<const float4*>(ckpt + (row * nblk + blk) * N + kBS * gi)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
      }
      if (kb > 1) forward(cb0, cb1, fine, kb, 1);  // one chunk: its coarse checkpoint is h
      for (int ch = cb1 - 1; ch >= cb0; --ch) {
        const int t0 = ch * kBT, tl = min(kBT, L - t0);
        __syncthreads();  // the previous chunk's tiles are no longer read
        stage(t0, tl, true);
        float hs[kBS];
        if (kb > 1) {  // written by this thread in forward(): program order suffices
            const float4 v = active ? *reinterpret_cast<const float4*>(fine + (row * kb + (ch - cb0)) * N + kBS * gi)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            hs[0] = v.x; hs[1] = v.y; hs[2] = v.z; hs[3] = v.w;
        } else {
#pragma unroll
            for (int i = 0; i < kBS; ++i) hs[i] = h[i];
        }
        __syncthreads();
        // recompute h_t over the chunk, and the pre-gate output
#pragma unroll
        for (int i = 0; i < kBS; ++i) h[i] = hs[i];
        for (int t = 0; t < tl; ++t) {
            const float dl = sm[lay.dl + c * kRow + t], dlx = sm[lay.dlx + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float4 cv = *reinterpret_cast<const float4*>(sm + lay.cs + t * N + kBS * gi);
            const float2 dl2 = make_float2(dl, dl), dx2 = make_float2(dlx, dlx);
            const float2 e01 = mul2(dl2, make_float2(A2[0], A2[1])), e23 = mul2(dl2, make_float2(A2[2], A2[3]));
            float2 h01 = make_float2(h[0], h[1]), h23 = make_float2(h[2], h[3]);
            h01 = fma2(make_float2(ex2_approx(e01.x), ex2_approx(e01.y)), h01, mul2(dx2, make_float2(bv.x, bv.y)));
            h23 = fma2(make_float2(ex2_approx(e23.x), ex2_approx(e23.y)), h23, mul2(dx2, make_float2(bv.z, bv.w)));
            h[0] = h01.x; h[1] = h01.y; h[2] = h23.x; h[3] = h23.y;
            const float2 ac = fma2(make_float2(cv.z, cv.w), h23, mul2(make_float2(cv.x, cv.y), h01));
            float acc = ac.x + ac.y;
            *reinterpret_cast<float4*>(hbuf + (t * NT + tid) * kBS) = make_float4(h[0], h[1], h[2], h[3]);
            if constexpr (TPC >= 8) {
                // two butterfly rounds here, the rest summed once per chunk below: the
                // step loop does not wait on a 32-lane reduction tree every step
                if (gi == 0) acc += Dd * sm[lay.xs + c * kRow + t];
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if ((gi & 3) == 0) sm[lay.red + (c * kBT + t) * (TPC / 4) + (gi >> 2)] = acc;
            } else {
#pragma unroll
                for (int off = 1; off < TPC; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (gi == 0) sm[lay.o + c * kRow + t] = acc + Dd * sm[lay.xs + c * kRow + t];
            }
        }
        __syncthreads();
        if constexpr (TPC >= 8) {  // o_t of every (channel, step) from its TPC / 4 partial sums
            for (int j = tid; j < CPB * kBT; j += NT) {
                const int cc = j / kBT, t = j % kBT;
                if (t >= tl) continue;
                const float* pr = sm + lay.red + j * (TPC / 4);
                float sum = 0.f;
#pragma unroll
                for (int q = 0; q < TPC / 4; ++q) sum += pr[q];
                sm[lay.o + cc * kRow + t] = sum;
            }
            __syncthreads();
        }
        // dC_t[n] = sum over the CTA's channels of do_t h_t[n]; dz from the pre-gate output
        channel_sum(lay.dout, a.dC, t0, tl);
        if (a.dz) {
            for (int j = tid; j < CPB * kBT; j += NT) {
                const int cc = tfast ? j / kBT : j % CPB, t = tfast ? j % kBT : j / CPB;
                if (cc >= nchan || t >= tl) continue;
                const long long i = xi(cc, t0 + t);
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
                const float4 v = *reinterpret_cast<const float4*>(hbuf + ((t - 1) * NT + tid) * kBS);
                hp[0] = v.x; hp[1] = v.y; hp[2] = v.z; hp[3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < kBS; ++i) hp[i] = hs[i];
            }
            const float dl = sm[lay.dl + c * kRow + t], xv = sm[lay.xs + c * kRow + t];
            const float dov = sm[lay.dout + c * kRow + t];
            const float4 bv = *reinterpret_cast<const float4*>(sm + lay.bs + t * N + kBS * gi);
            const float4 cv = *reinterpret_cast<const float4*>(sm + lay.cs + t * N + kBS * gi);
            // states in pairs (f32x2): E = exp(Delta A), G = g + do C, dx += G B,
            // dDelta += G (B x + h_{t-1} E A), dA += G h_{t-1} E Delta, g <- G E
            const float2 dl2 = make_float2(dl, dl), do2 = make_float2(dov, dov), xv2 = make_float2(xv, xv);
            float2 gx2 = make_float2(0.f, 0.f), gd2 = make_float2(0.f, 0.f), G2[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float2 bq = q ? make_float2(bv.z, bv.w) : make_float2(bv.x, bv.y);
                const float2 cq = q ? make_float2(cv.z, cv.w) : make_float2(cv.x, cv.y);
                const float2 ea = mul2(dl2, make_float2(A2[2 * q], A2[2 * q + 1]));
                const float2 E = make_float2(ex2_approx(ea.x), ex2_approx(ea.y));
                const float2 G = fma2(do2, cq, make_float2(gcar[2 * q], gcar[2 * q + 1]));
                gx2 = fma2(G, bq, gx2);
                const float2 hE = mul2(make_float2(hp[2 * q], hp[2 * q + 1]), E);
                gd2 = fma2(G, fma2(hE, make_float2(Av[2 * q], Av[2 * q + 1]), mul2(bq, xv2)), gd2);
                const float2 da = fma2(mul2(G, hE), dl2, make_float2(dAacc[2 * q], dAacc[2 * q + 1]));
                dAacc[2 * q] = da.x;
                dAacc[2 * q + 1] = da.y;
                const float2 gn = mul2(G, E);
                gcar[2 * q] = gn.x;
                gcar[2 * q + 1] = gn.y;
                G2[q] = G;
            }
            float gx = (gx2.x + gx2.y) * dl, gd = gd2.x + gd2.y;
            const float Gt[kBS] = {G2[0].x, G2[0].y, G2[1].x, G2[1].y};
            *reinterpret_cast<float4*>(hbuf + (t * NT + tid) * kBS) = make_float4(Gt[0], Gt[1], Gt[2], Gt[3]);
            if constexpr (TPC >= 8) {
                // three butterfly rounds here, the rest summed once per chunk below
                if (gi == 0) gx += dov * Dd;
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) {
                    gx += __shfl_xor_sync(0xffffffffu, gx, off);
                    gd += __shfl_xor_sync(0xffffffffu, gd, off);
                }
                if ((gi & 7) == 0)
                    *reinterpret_cast<float2*>(sm + lay.red + ((c * kBT + t) * (TPC / 8) + (gi >> 3)) * 2) =
                        make_float2(gx, gd);
            } else {
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
        }
        __syncthreads();
        if constexpr (TPC >= 8) {  // dx and d(delta) of every (channel, step) from the partials
            for (int j = tid; j < CPB * kBT; j += NT) {
                const int cc = j / kBT, t = j % kBT;
                if (t >= tl) continue;
                const float2* pr = reinterpret_cast<const float2*>(sm + lay.red) + j * (TPC / 8);
                float sx = 0.f, sd = 0.f;
#pragma unroll
                for (int q = 0; q < TPC / 8; ++q) {
                    sx += pr[q].x;
                    sd += pr[q].y;
                }
                sm[lay.gx + cc * kRow + t] = sx;
                sm[lay.gd + cc * kRow + t] = sd * sm[lay.sg + cc * kRow + t];
            }
            __syncthreads();
            if (gi == 0)  // the channel's dD and d(bias) terms of this chunk
                for (int t = 0; t < tl; ++t) {
                    dDacc += sm[lay.dout + c * kRow + t] * sm[lay.xs + c * kRow + t];
                    dbacc += sm[lay.gd + c * kRow + t];
                }
        }
        // dB_t[n] = sum over the CTA's channels of G_t[n] Delta_t x_t
        channel_sum(lay.dlx, a.dB, t0, tl);
        for (int j = tid; j < CPB * kBT; j += NT) {
            const int cc = tfast ? j / kBT : j % CPB, t = tfast ? j % kBT : j / CPB;
            if (cc >= nchan || t >= tl) continue;
            a.dx[xi(cc, t0 + t)] = sm[lay.gx + cc * kRow + t];
            // one channel per head: the gradient of delta directly; else the channel's
            // share added into the head's (zeroed before the launch)
            if (a.hp == 1)
                a.ddelta[di(cc, t0 + t)] = sm[lay.gd + cc * kRow + t];
            else
                atomicAdd(a.ddelta + di(cc, t0 + t), sm[lay.gd + cc * kRow + t]);
        }
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

// dA, dD, dbias: sums over the batch (and over a head's channels and, for A, states when
// hp > 1).  One thread per output element, fixed summation order.
__global__ void m1_scan_bwd_reduce(BwdView a, const float* part_a, const float* part_d, const float* part_bias) {
    const int Dm = a.dim, N = a.dstate, Bt = a.batch, hp = a.hp;
    const int heads = Dm / hp;
    const size_t na = a.san ? static_cast<size_t>(Dm) * N : static_cast<size_t>(heads);
    const size_t total = na + 2 * static_cast<size_t>(heads);
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (i < na) {
            const size_t e = i;  // (d, n), or the head
            float sum = 0.f;
            if (a.san) {
                for (int bb = 0; bb < Bt; ++bb) sum += part_a[static_cast<size_t>(bb) * Dm * N + e];
            } else {
                for (int bb = 0; bb < Bt; ++bb)
                    for (int q = 0; q < hp * N; ++q)
                        sum += part_a[(static_cast<size_t>(bb) * Dm + e * hp) * N + q];
            }
            a.dA[e] = sum;
        } else {
            const size_t e = i - na;
            const int hh = static_cast<int>(e % heads);
            const float* src = e < static_cast<size_t>(heads) ? part_d : part_bias;
            float* dst = e < static_cast<size_t>(heads) ? a.dD : a.dbias;
            if (!dst) continue;
            float sum = 0.f;
            for (int bb = 0; bb < Bt; ++bb)
                for (int q = 0; q < hp; ++q) sum += src[static_cast<size_t>(bb) * Dm + hh * hp + q];
            dst[hh] = sum;
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
        case 128: return 32;
        default: return 0;
    }
}

int bwd_kb(const BwdView& a) {
    const int nch = (a.seqlen + kBT - 1) / kBT;
    return bwd_block_chunks(nch, a.dstate, a.seqlen, a.in_dtype == SSM_BF16 ? 2 : 4, a.dy_dtype == SSM_BF16 ? 2 : 4);
}

BwdWs bwd_ws(const BwdView& a) {
    const size_t rows = static_cast<size_t>(a.batch) * a.dim;
    const int nch = (a.seqlen + kBT - 1) / kBT;
    const int kb = bwd_kb(a);
    const size_t nblk = (static_cast<size_t>(nch) + kb - 1) / kb;
    auto r256 = [](size_t v) { return (v + 255) / 256 * 256; };
    BwdWs w;
    w.ckpt = 0;
    w.fine = r256(rows * nblk * a.dstate * 4);
    w.part_a = w.fine + (kb > 1 ? r256(rows * static_cast<size_t>(kb) * a.dstate * 4) : 0);
    w.part_d = w.part_a + r256(rows * a.dstate * 4);
    w.part_bias = w.part_d + r256(rows * 4);
    w.bytes = w.part_bias + r256(rows * 4);
    return w;
}

int bwd_cps(const BwdView& a) {
    const int cpb = bwd_cpb(bwd_tpc(a.dstate));
    const int per_group = a.dim / a.ngroups;
    return (per_group + cpb - 1) / cpb;
}

template <typename Tin, typename Tdy, int TPC>
cudaError_t launch_bwd(const BwdView& a, void* ws, cudaStream_t s) {
    const int cps = bwd_cps(a);
    const BwdWs w = bwd_ws(a);
    unsigned char* base = static_cast<unsigned char*>(ws);
    const BwdLayout lay(bwd_cpb(TPC), TPC * kBS, bwd_threads(TPC));
    const size_t smem = static_cast<size_t>(lay.total) * sizeof(float);
    auto k = m1_scan_bwd<Tin, Tdy, TPC>;
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(k), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // the atomic sums start from zero: dB, dC (dense in either layout) and, with shared
    // delta, the head's gradient
    const size_t nbc = static_cast<size_t>(a.batch) * a.ngroups * a.dstate * a.seqlen;
    if ((e = cudaMemsetAsync(a.dB, 0, nbc * sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dC, 0, nbc * sizeof(float), s)) != cudaSuccess) return e;
    if (a.hp > 1) {
        const size_t ndt = static_cast<size_t>(a.batch) * (a.dim / a.hp) * a.seqlen;
        if ((e = cudaMemsetAsync(a.ddelta, 0, ndt * sizeof(float), s)) != cudaSuccess) return e;
    }
    const int grid = a.batch * a.ngroups * cps;
    float* part_a = reinterpret_cast<float*>(base + w.part_a);
    float* part_d = reinterpret_cast<float*>(base + w.part_d);
    float* part_bias = reinterpret_cast<float*>(base + w.part_bias);
    if (grid > 0)
        k<<<grid, bwd_threads(TPC), smem, s>>>(a, cps, bwd_kb(a), reinterpret_cast<float*>(base + w.ckpt),
                                        reinterpret_cast<float*>(base + w.fine), part_a, part_d, part_bias);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    m1_scan_bwd_reduce<<<2 * 152, 256, 0, s>>>(a, part_a, part_d, part_bias);
    return cudaGetLastError();
}

template <typename Tin, typename Tdy>
cudaError_t dispatch_tpc(const BwdView& a, void* ws, cudaStream_t s) {
    switch (bwd_tpc(a.dstate)) {
        case 4: return launch_bwd<Tin, Tdy, 4>(a, ws, s);
        case 8: return launch_bwd<Tin, Tdy, 8>(a, ws, s);
        case 16: return launch_bwd<Tin, Tdy, 16>(a, ws, s);
        case 32: return launch_bwd<Tin, Tdy, 32>(a, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t bwd_launch(const BwdView& a, void* workspace, cudaStream_t s) {
    const bool in_bf = a.in_dtype == SSM_BF16, dy_bf = a.dy_dtype == SSM_BF16;
    if (in_bf && dy_bf) return dispatch_tpc<bf16_t, bf16_t>(a, workspace, s);
    if (in_bf) return dispatch_tpc<bf16_t, float>(a, workspace, s);
    if (dy_bf) return dispatch_tpc<float, bf16_t>(a, workspace, s);
    return dispatch_tpc<float, float>(a, workspace, s);
}

// Mamba-1 layouts: x, z, dy, delta [Bt, D, L]; B, C [Bt, G, N, L]; A [D, N]
BwdView view_m1(const M1BwdArgs& a) {
    const ssm_scan_params& f = a.fwd;
    BwdView v{};
    v.x = f.x; v.delta = f.delta; v.z = f.z; v.B = f.B; v.C = f.C; v.dy = a.dy;
    v.delta_bias = f.delta_bias; v.A = f.A; v.D_skip = f.D_skip; v.h0 = f.h0; v.dh_final = a.dh_final;
    v.dx = a.dx; v.ddelta = a.ddelta; v.dz = a.dz; v.dh0 = a.dh0;
    v.dA = a.dA; v.dB = a.dB; v.dC = a.dC; v.dD = a.dD_skip; v.dbias = a.ddelta_bias;
    v.batch = f.batch; v.dim = f.dim; v.dstate = f.dstate; v.seqlen = f.seqlen; v.ngroups = f.ngroups;
    v.softplus = f.delta_softplus; v.in_dtype = f.in_dtype; v.dy_dtype = f.out_dtype;
    const long long L = f.seqlen, D = f.dim, N = f.dstate, G = f.ngroups;
    v.hp = 1;
    v.sxb = D * L; v.sxd = L; v.sxt = 1;
    v.sdb = D * L; v.sdh = L; v.sdt = 1;
    v.sbb = G * N * L; v.sbg = N * L; v.sbn = L; v.sbt = 1;
    v.sah = N; v.san = 1;
    return v;
}

// SSD layouts: x, z, dy [Bt, L, H, P] (channel d = h P + p); dt [Bt, L, H]; B, C
// [Bt, L, G, N]; A, D, dt_bias [H]
BwdView view_ssd(const ssd_bwd_params& a) {
    const ssd_params& f = a.fwd;
    BwdView v{};
    v.x = f.x; v.delta = f.dt; v.z = f.z; v.B = f.B; v.C = f.C; v.dy = a.dy;
    v.delta_bias = f.dt_bias; v.A = f.A; v.D_skip = f.D_skip; v.h0 = f.h0; v.dh_final = a.dh_final;
    v.dx = a.dx; v.ddelta = a.ddt; v.dz = a.dz; v.dh0 = a.dh0;
    v.dA = a.dA; v.dB = a.dB; v.dC = a.dC; v.dD = a.dD_skip; v.dbias = a.ddt_bias;
    const long long L = f.seqlen, H = f.nheads, P = f.headdim, N = f.dstate, G = f.ngroups;
    v.batch = f.batch; v.dim = static_cast<int>(H * P); v.dstate = f.dstate; v.seqlen = f.seqlen;
    v.ngroups = f.ngroups; v.softplus = f.dt_softplus; v.in_dtype = f.in_dtype; v.dy_dtype = f.out_dtype;
    v.hp = f.headdim;
    v.sxb = L * H * P; v.sxd = 1; v.sxt = H * P;
    v.sdb = L * H; v.sdh = 1; v.sdt = H;
    v.sbb = L * G * N; v.sbg = N; v.sbn = 1; v.sbt = G * N;
    v.sah = 1; v.san = 0;
    return v;
}

}  // namespace

bool m1_bwd_supported(const M1BwdArgs& a) {
    return a.fwd.disc == SSM_DISC_EXP_EULER && bwd_tpc(a.fwd.dstate) > 0;
}

size_t m1_bwd_workspace_size(const M1BwdArgs& a) {
    if (!m1_bwd_supported(a)) return 0;
    return bwd_ws(view_m1(a)).bytes;
}

cudaError_t m1_bwd_launch(const M1BwdArgs& a, void* workspace, cudaStream_t s) {
    return bwd_launch(view_m1(a), workspace, s);
}

bool ssd_bwd_supported(const ssd_bwd_params& a) {
    return a.fwd.disc == SSM_DISC_EXP_EULER && bwd_tpc(a.fwd.dstate) > 0;
}

// The chunked form (ssd_bwd.cu) where it covers the shape, else the tied recurrence.
size_t ssd_bwd_workspace_size(const ssd_bwd_params& a) {
    if (!ssd_bwd_supported(a)) return 0;
    if (ssd_chunked_bwd_supported(a)) return ssd_chunked_bwd_workspace_size(a);
    return bwd_ws(view_ssd(a)).bytes;
}

cudaError_t ssd_bwd_launch(const ssd_bwd_params& a, void* workspace, cudaStream_t s) {
    if (ssd_chunked_bwd_supported(a)) return ssd_chunked_bwd_launch(a, workspace, s);
    return bwd_launch(view_ssd(a), workspace, s);
}

}  // namespace ssm
