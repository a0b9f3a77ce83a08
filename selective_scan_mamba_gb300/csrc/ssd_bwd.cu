// ssd_bwd.cu -- Mamba-2 SSD backward in chunked form (float32 on the CUDA cores).
//
// The forward is the chunked SSD ("From S4 to Mamba-3", 03/System, mamba2_minimal.py;
// 04/Approach, "Chunked SSD"): per (batch b, head h), with a_t = dt_t A_h, the input
// weight dt_t (exponential-Euler) and, inside a chunk of Q steps, the running sums
// cum_t = a_0 + ... + a_t (tot = cum_{Q-1}) and the state h_p entering the chunk,
//   h_t = e^{cum_t} h_p + sum_{s<=t} e^{cum_t - cum_s} dt_s B_s x_s^T      [N x P]
//   y_t = sum_{s<=t} (C_t . B_s) e^{cum_t - cum_s} dt_s x_s + e^{cum_t} C_t^T h_p
//   o_t = y_t + D x_t,   out_t = o_t SiLU(z_t)
// and the state leaving the chunk is e^{tot} h_p + S with S = sum_s F_s B_s x_s^T,
// F_s = e^{tot - cum_s} dt_s.  Its reverse-mode derivative, with do_t = dout_t SiLU(z_t)
// and G = dL/d(state leaving the chunk), splits into products of chunk-sized matrices:
//   T[t][s] = do_t . x_s,  CB[t][s] = C_t . B_s,  E[t][s] = e^{cum_t - cum_s} (s <= t)
//   dx_s = D do_s + sum_t CB E dt_s do_t + F_s G^T B_s
//   dB_s = sum_t T E dt_s C_t + F_s G x_s,     dC_t = sum_s T E dt_s B_s + e^{cum_t} h_p do_t
//   d(dt)_s from dt_s as input weight: sum_t CB E T + e^{tot - cum_s} B_s^T G x_s
//   d cum_t = sum_s dt_s (CB E T)[t][s] - dt_t sum_u (CB E T)[u][t] + C_t . (e^{cum_t} h_p do_t)
//             - F_t B_t^T G x_t,    d tot = sum_s F_s B_s^T G x_s + e^{tot} <G, h_p>
//   d a_s = sum_{t>=s} d cum_t + d tot,   d(dt)_s += d a_s A_h,   dA_h += d a_s dt_s
// and the chunk boundaries chain the states forwards (h_p of chunk c+1 = e^{tot_c} h_p
// of chunk c + S_c) and the adjoints backwards (G_{c-1} = e^{tot_c} G_c + R_c with
// R_c = sum_t e^{cum_t} C_t do_t^T, the chunk's outputs' dependence on its h_p).
//
// Launches, per slice of (batch, head) sequences (the slice bounds the workspace):
//   1. ssd_bwd_chunk_states: S_c and tot_c of every chunk;
//   2. ssd_bwd_pass<false>: walks each sequence's chunks forwards, replacing S_c by the
//      state entering chunk c (h0 first);
//   3. ssd_bwd_chunk_outputs: recomputes o_t, writes dz and do_t (into dx, as scratch)
//      and R_c;
//   4. ssd_bwd_pass<true>: walks the chunks backwards, replacing R_c by the adjoint of
//      the state leaving chunk c (dh_final first), and writes dh0;
//   5. ssd_bwd_chunk_grads: every gradient of the chunk from the products above; dB and
//      dC are summed over a group's heads with float32 atomic adds (zeroed first), ddt
//      and dx are written once, dA, dD and ddt_bias per-chunk partials go to the
//      workspace; after the last slice a small launch sums them in a fixed order.
// Each chunk launch runs one CTA of 256 threads per chunk with the chunk's operands in
// shared memory as float32 (rows padded to an odd length so that row and column walks
// are free of bank conflicts); a product of an I x K by a K x J operand gives each thread
// a tile of I J / 256 outputs.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kQ = 64;     // steps per chunk
#ifndef SSD_BWD_THREADS
#define SSD_BWD_THREADS 256
#endif
#ifndef SSD_BWD_UNROLL
#define SSD_BWD_UNROLL 8
#endif
constexpr int kNT = SSD_BWD_THREADS;  // threads per CTA of the chunk launches
constexpr int kUnroll = SSD_BWD_UNROLL;  // unrolling of the products' inner loop
constexpr int kSQ = kQ + 1;

struct CkArgs {
    int batch, seqlen, nheads, hpg, ngroups, nch;  // hpg: heads per group
    int softplus;
    const void* x;
    const void* dt;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* h0;
    const void* dy;
    const float* dh_final;
    float* dx;
    float* ddt;
    float* dz;
    float* dB;
    float* dC;
    float* dh0;
    float* st;    // [slice][nch][P][N]: S_c, then the state entering chunk c
    float* adj;   // [slice][nch][P][N]: R_c, then the adjoint of the state leaving chunk c
    float* tot;   // [batch * H][nch]
    float* part;  // [3][batch * H * nch]: dA, dD, ddt_bias per chunk
    int q0;       // first sequence (b H + h) of the slice
    int nq;       // sequences in the slice
};

template <typename T>
__device__ __forceinline__ float ld(const void* p, size_t i) {
    return to_f32(static_cast<const T*>(p)[i]);
}

__device__ __forceinline__ float sigmoid_accurate(float v) { return 1.f / (1.f + expf(-v)); }

// The chunk's steps: the softplus argument u (raw dt + bias), dt (0 past the sequence
// end, which leaves the state unchanged) and the inclusive running sums cum of dt A.
// Warp 0; lane j holds steps j and j + 32.
template <typename Tin>
__device__ __forceinline__ void chunk_steps(const CkArgs& a, int b, int hd, int c, float* su, float* sdt,
                                            float* scum) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const float Ah = a.A[hd];
    const float bias = a.dt_bias ? a.dt_bias[hd] : 0.f;
    float v[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int s = lane + 32 * j;
        const long long tau = static_cast<long long>(c) * kQ + s;
        float u = 0.f, dt = 0.f;
        if (tau < a.seqlen) {
            u = ld<Tin>(a.dt, (static_cast<size_t>(b) * a.seqlen + tau) * a.nheads + hd) + bias;
            dt = a.softplus ? softplus_accurate(u) : u;
        }
        su[s] = u;
        sdt[s] = dt;
        v[j] = dt * Ah;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float o = __shfl_up_sync(0xffffffffu, v[j], off);
            if (lane >= off) v[j] += o;
        }
    }
    const float first = __shfl_sync(0xffffffffu, v[0], 31);
    scum[lane] = v[0];
    scum[lane + 32] = first + v[1];
}

// A thread's share of an I x J product: rows i0 .. i0 + TI - 1, columns j0 + q NJ
// (q < TJ), so that the threads of a warp cover consecutive columns.
template <int I, int J>
struct Tile {
    static constexpr int C = I * J / kNT;
    static constexpr int TI = C >= 4 ? 4 : C;
    static constexpr int TJ = C / TI;
    static constexpr int NJ = J / TJ;
    static_assert(I * J % kNT == 0 && C >= 1 && I % TI == 0 && J % TJ == 0 && (I / TI) * NJ == kNT,
                  "tile shape");
    int i0, j0;
    __device__ __forceinline__ Tile() : i0((static_cast<int>(threadIdx.x) / NJ) * TI), j0(threadIdx.x % NJ) {}
    __device__ __forceinline__ int row(int r) const { return i0 + r; }
    __device__ __forceinline__ int col(int q) const { return j0 + q * NJ; }
};

// acc[r][q] += sum_k a(row r, k) b(k, col q)
template <int I, int J, int K, typename FA, typename FB>
__device__ __forceinline__ void mac(const Tile<I, J>& t, float (&acc)[Tile<I, J>::TI][Tile<I, J>::TJ], FA a,
                                    FB b) {
    constexpr int TI = Tile<I, J>::TI, TJ = Tile<I, J>::TJ;
#pragma unroll kUnroll
    for (int k = 0; k < K; ++k) {
        float av[TI], bv[TJ];
#pragma unroll
        for (int r = 0; r < TI; ++r) av[r] = a(t.row(r), k);
#pragma unroll
        for (int q = 0; q < TJ; ++q) bv[q] = b(k, t.col(q));
#pragma unroll
        for (int r = 0; r < TI; ++r)
#pragma unroll
            for (int q = 0; q < TJ; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
    }
}

template <int I, int J>
__device__ __forceinline__ void zero(float (&acc)[Tile<I, J>::TI][Tile<I, J>::TJ]) {
#pragma unroll
    for (int r = 0; r < Tile<I, J>::TI; ++r)
#pragma unroll
        for (int q = 0; q < Tile<I, J>::TJ; ++q) acc[r][q] = 0.f;
}

// rows [Q][ld] of a [Bt, L, ., W] tensor (row stride `stride` elements), zero past L
template <typename T, int W>
__device__ __forceinline__ void load_rows(float* dst, int ldst, const void* src, size_t base, size_t stride,
                                          int rows_valid) {
    for (int i = threadIdx.x; i < kQ * W; i += kNT) {
        const int t = i / W, w = i % W;
        dst[t * ldst + w] = t < rows_valid ? ld<T>(src, base + t * stride + w) : 0.f;
    }
}

// block sum in a fixed order (every thread calls it; the result is returned to all)
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kNT / 32; ++w) s += red[w];
    return s;
}

struct ChunkId {
    int ql, c, q, b, hd, g, valid;
    size_t row0;  // (b L + c Q): the first time row of the chunk
    __device__ __forceinline__ ChunkId(const CkArgs& a) {
        ql = blockIdx.x / a.nch;
        c = blockIdx.x % a.nch;
        q = a.q0 + ql;
        b = q / a.nheads;
        hd = q % a.nheads;
        g = hd / a.hpg;
        valid = min(kQ, a.seqlen - c * kQ);
        row0 = static_cast<size_t>(b) * a.seqlen + static_cast<size_t>(c) * kQ;
    }
};

// ---------------------------------------------------------------------------------------
// 1. chunk states S_c[p][n] = sum_s x_s[p] F_s B_s[n] and tot_c
// ---------------------------------------------------------------------------------------
template <typename Tin, int N, int P>
__global__ void __launch_bounds__(kNT) ssd_bwd_chunk_states(CkArgs a) {
    constexpr int SX = P + 1, SN = N + 1;
    extern __shared__ float sm[];
    float* xs = sm;                // [Q][SX] x_s F_s
    float* Bs = xs + kQ * SX;      // [Q][SN]
    float* su = Bs + kQ * SN;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, N>(Bs, SN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    __syncthreads();
    const float tot = scum[kQ - 1];
    for (int i = threadIdx.x; i < kQ * P; i += kNT) {
        const int s = i / P, p = i % P;
        const float f = expf(tot - scum[s]) * sdt[s];
        xs[s * SX + p] = s < id.valid ? ld<Tin>(a.x, ((id.row0 + s) * H + id.hd) * P + p) * f : 0.f;
    }
    __syncthreads();
    const Tile<P, N> t;
    float acc[Tile<P, N>::TI][Tile<P, N>::TJ];
    zero<P, N>(acc);
    mac<P, N, kQ>(t, acc, [&](int p, int s) { return xs[s * SX + p]; }, [&](int s, int n) { return Bs[s * SN + n]; });
    float* out = a.st + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N;
#pragma unroll
    for (int r = 0; r < Tile<P, N>::TI; ++r)
#pragma unroll
        for (int q = 0; q < Tile<P, N>::TJ; ++q) out[t.row(r) * N + t.col(q)] = acc[r][q];
    if (threadIdx.x == 0) a.tot[static_cast<size_t>(id.q) * a.nch + id.c] = tot;
}

// ---------------------------------------------------------------------------------------
// 2. / 4. the chunk-boundary chains, one thread per (sequence, p, n), chunks prefetched
// eight at a time.  Forwards: v_c <- carry, carry <- e^{tot_c} carry + v_c (carry = h0).
// Backwards: the same from the last chunk (carry = dh_final), the final carry is dh0.
// ---------------------------------------------------------------------------------------
template <bool REVERSE>
__global__ void __launch_bounds__(256) ssd_bwd_pass(CkArgs a, int PN) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(a.nq) * PN) return;
    const int ql = static_cast<int>(i / PN), e = static_cast<int>(i % PN);
    const size_t qg = static_cast<size_t>(a.q0 + ql) * PN + e;  // [Bt, H, P, N] index
    float* v = (REVERSE ? a.adj : a.st) + static_cast<size_t>(ql) * a.nch * PN + e;
    const float* tot = a.tot + static_cast<size_t>(a.q0 + ql) * a.nch;
    const float* init = REVERSE ? a.dh_final : a.h0;
    float carry = init ? init[qg] : 0.f;
    constexpr int kG = 8;
    for (int c0 = 0; c0 < a.nch; c0 += kG) {
        float val[kG], dec[kG];
#pragma unroll
        for (int j = 0; j < kG; ++j) {
            const int c = REVERSE ? a.nch - 1 - (c0 + j) : c0 + j;
            if (c0 + j < a.nch) {
                val[j] = v[static_cast<size_t>(c) * PN];
                dec[j] = expf(tot[c]);
            }
        }
#pragma unroll
        for (int j = 0; j < kG; ++j) {
            const int c = REVERSE ? a.nch - 1 - (c0 + j) : c0 + j;
            if (c0 + j < a.nch) {
                v[static_cast<size_t>(c) * PN] = carry;
                carry = dec[j] * carry + val[j];
            }
        }
    }
    if (REVERSE && a.dh0) a.dh0[qg] = carry;
}

// ---------------------------------------------------------------------------------------
// 3. outputs: o_t, dz_t, do_t (into dx) and R_c[p][n] = sum_t do_t[p] e^{cum_t} C_t[n]
// ---------------------------------------------------------------------------------------
template <typename Tin, int N, int P>
__global__ void __launch_bounds__(kNT, 1) ssd_bwd_chunk_outputs(CkArgs a) {
    constexpr int SX = P + 1, SN = N + 1;
    extern __shared__ float sm[];
    float* xs = sm;                // [Q][SX]
    float* ds = xs + kQ * SX;      // [Q][SX] do_t e^{cum_t}
    float* Bs = ds + kQ * SX;      // [Q][SN]
    float* Cs = Bs + kQ * SN;      // [Q][SN]
    float* Hs = Cs + kQ * SN;      // [P][SN] state entering the chunk
    float* Wa = Hs + P * SN;       // [Q][kSQ]
    float* su = Wa + kQ * kSQ;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, P>(xs, SX, a.x, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                      id.valid);
    load_rows<Tin, N>(Bs, SN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    load_rows<Tin, N>(Cs, SN, a.C, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    {
        const float* hp = a.st + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N;
        for (int i = threadIdx.x; i < P * N; i += kNT) Hs[(i / N) * SN + i % N] = hp[i];
    }
    __syncthreads();
    {  // Wa = (C B^T) E dt_s, lower triangle
        const Tile<kQ, kQ> t;
        float acc[Tile<kQ, kQ>::TI][Tile<kQ, kQ>::TJ];
        zero<kQ, kQ>(acc);
        mac<kQ, kQ, N>(t, acc, [&](int i, int n) { return Cs[i * SN + n]; }, [&](int n, int s) { return Bs[s * SN + n]; });
#pragma unroll
        for (int r = 0; r < Tile<kQ, kQ>::TI; ++r)
#pragma unroll
            for (int q = 0; q < Tile<kQ, kQ>::TJ; ++q) {
                const int i = t.row(r), s = t.col(q);
                Wa[i * kSQ + s] = s <= i ? acc[r][q] * expf(scum[i] - scum[s]) * sdt[s] : 0.f;
            }
    }
    __syncthreads();
    {  // o = Wa x + e^{cum_t} C h_p + D x, then the gate
        const Tile<kQ, P> t;
        float a1[Tile<kQ, P>::TI][Tile<kQ, P>::TJ], a2[Tile<kQ, P>::TI][Tile<kQ, P>::TJ];
        zero<kQ, P>(a1);
        zero<kQ, P>(a2);
        mac<kQ, P, kQ>(t, a1, [&](int i, int s) { return Wa[i * kSQ + s]; }, [&](int s, int p) { return xs[s * SX + p]; });
        mac<kQ, P, N>(t, a2, [&](int i, int n) { return Cs[i * SN + n]; }, [&](int n, int p) { return Hs[p * SN + n]; });
        const float Dh = a.D ? a.D[id.hd] : 0.f;
#pragma unroll
        for (int r = 0; r < Tile<kQ, P>::TI; ++r) {
            const int i = t.row(r);
            const float ec = expf(scum[i]);
#pragma unroll
            for (int q = 0; q < Tile<kQ, P>::TJ; ++q) {
                const int p = t.col(q);
                float dov = 0.f;
                if (i < id.valid) {
                    const size_t gi = ((id.row0 + i) * H + id.hd) * P + p;
                    const float o = a1[r][q] + ec * a2[r][q] + Dh * xs[i * SX + p];
                    const float dout = ld<Tin>(a.dy, gi);
                    if (a.z) {
                        const float zz = ld<Tin>(a.z, gi);
                        const float sg = sigmoid_accurate(zz);
                        dov = dout * zz * sg;
                        a.dz[gi] = dout * o * sg * (1.f + zz * (1.f - sg));
                    } else {
                        dov = dout;
                    }
                    a.dx[gi] = dov;
                }
                ds[i * SX + p] = dov * ec;
            }
        }
    }
    __syncthreads();
    {  // R[p][n] = sum_t ds[t][p] C[t][n]
        const Tile<P, N> t;
        float acc[Tile<P, N>::TI][Tile<P, N>::TJ];
        zero<P, N>(acc);
        mac<P, N, kQ>(t, acc, [&](int p, int s) { return ds[s * SX + p]; }, [&](int s, int n) { return Cs[s * SN + n]; });
        float* out = a.adj + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N;
#pragma unroll
        for (int r = 0; r < Tile<P, N>::TI; ++r)
#pragma unroll
            for (int q = 0; q < Tile<P, N>::TJ; ++q) out[t.row(r) * N + t.col(q)] = acc[r][q];
    }
}

// ---------------------------------------------------------------------------------------
// 5. gradients of the chunk
// ---------------------------------------------------------------------------------------
template <typename Tin, int N, int P>
__global__ void __launch_bounds__(kNT, 1) ssd_bwd_chunk_grads(CkArgs a) {
    constexpr int SX = P + 1, SN = N + 1;
    extern __shared__ float sm[];
    float* xs = sm;                // [Q][SX]
    float* ds = xs + kQ * SX;      // [Q][SX] do
    float* Bs = ds + kQ * SX;      // [Q][SN]
    float* Cs = Bs + kQ * SN;      // [Q][SN]
    float* Hs = Cs + kQ * SN;      // [P][SN] adjoint leaving the chunk, then state entering it
    float* Wa = Hs + P * SN;       // [Q][kSQ] C B^T, then C B^T E dt_s
    float* Wb = Wa + kQ * kSQ;     // [Q][kSQ] T, then T E dt_s
    float* Vb = Wb + kQ * kSQ;     // [Q][kSQ] C B^T E T
    float* su = Vb + kQ * kSQ;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    float* sdw = scum + kQ;        // dt_s as input weight: intra-chunk part
    float* sdc = sdw + kQ;         // d cum, intra-chunk part
    float* sdc2 = sdc + kQ;        // d cum, through the state entering the chunk
    float* sdF = sdc2 + kQ;        // B_s^T G x_s
    float* red = sdF + kQ;         // [32]
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    const size_t PN = static_cast<size_t>(P) * N;
    const size_t cidx = static_cast<size_t>(id.ql) * a.nch + id.c;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, P>(xs, SX, a.x, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                      id.valid);
    load_rows<float, P>(ds, SX, a.dx, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                        id.valid);
    load_rows<Tin, N>(Bs, SN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    load_rows<Tin, N>(Cs, SN, a.C, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    if (threadIdx.x < kQ) {
        sdc2[threadIdx.x] = 0.f;
        sdF[threadIdx.x] = 0.f;
    }
    __syncthreads();
    {  // Wa = C B^T, Wb = T = do x^T
        const Tile<kQ, kQ> t;
        float a1[Tile<kQ, kQ>::TI][Tile<kQ, kQ>::TJ], a2[Tile<kQ, kQ>::TI][Tile<kQ, kQ>::TJ];
        zero<kQ, kQ>(a1);
        zero<kQ, kQ>(a2);
        mac<kQ, kQ, N>(t, a1, [&](int i, int n) { return Cs[i * SN + n]; }, [&](int n, int s) { return Bs[s * SN + n]; });
        mac<kQ, kQ, P>(t, a2, [&](int i, int p) { return ds[i * SX + p]; }, [&](int p, int s) { return xs[s * SX + p]; });
#pragma unroll
        for (int r = 0; r < Tile<kQ, kQ>::TI; ++r)
#pragma unroll
            for (int q = 0; q < Tile<kQ, kQ>::TJ; ++q) {
                const int i = t.row(r), s = t.col(q);
                float w1 = 0.f, w2 = 0.f, v = 0.f;
                if (s <= i) {
                    const float e = expf(scum[i] - scum[s]);
                    v = a1[r][q] * e * a2[r][q];
                    w1 = a1[r][q] * e * sdt[s];
                    w2 = a2[r][q] * e * sdt[s];
                }
                Wa[i * kSQ + s] = w1;
                Wb[i * kSQ + s] = w2;
                Vb[i * kSQ + s] = v;
            }
    }
    __syncthreads();
    // column sums (dt_s as weight) and dt-weighted row sums (d cum) of C B^T E T; the
    // adjoint leaving the chunk into Hs, and <adjoint, state entering the chunk>
    if (threadIdx.x < kQ) {
        const int s = threadIdx.x;
        float cs = 0.f;
        for (int i = 0; i < kQ; ++i) cs += Vb[i * kSQ + s];
        sdw[s] = cs;
    } else if (threadIdx.x < 2 * kQ) {
        const int i = threadIdx.x - kQ;
        float rs = 0.f;
        for (int s = 0; s < kQ; ++s) rs += sdt[s] * Vb[i * kSQ + s];
        sdc[i] = rs;
    }
    float dot = 0.f;
    {
        const float* gh = a.adj + cidx * PN;
        const float* hp = a.st + cidx * PN;
        for (int i = threadIdx.x; i < P * N; i += kNT) {
            const float gv = gh[i];
            Hs[(i / N) * SN + i % N] = gv;
            dot = fmaf(gv, hp[i], dot);
        }
    }
    dot = block_sum(dot, red);  // includes the barrier that publishes Hs, sdw, sdc
    const float tot = scum[kQ - 1];
    const float Dh = a.D ? a.D[id.hd] : 0.f;
    float ddsum = 0.f;  // sum do x (dD)
    {  // dx = D do + Wa^T do + F_s B G
        const Tile<kQ, P> t;
        float a1[Tile<kQ, P>::TI][Tile<kQ, P>::TJ], a2[Tile<kQ, P>::TI][Tile<kQ, P>::TJ];
        zero<kQ, P>(a1);
        zero<kQ, P>(a2);
        mac<kQ, P, kQ>(t, a1, [&](int s, int i) { return Wa[i * kSQ + s]; }, [&](int i, int p) { return ds[i * SX + p]; });
        mac<kQ, P, N>(t, a2, [&](int s, int n) { return Bs[s * SN + n]; }, [&](int n, int p) { return Hs[p * SN + n]; });
#pragma unroll
        for (int r = 0; r < Tile<kQ, P>::TI; ++r) {
            const int s = t.row(r);
            if (s >= id.valid) continue;
            const float F = expf(tot - scum[s]) * sdt[s];
#pragma unroll
            for (int q = 0; q < Tile<kQ, P>::TJ; ++q) {
                const int p = t.col(q);
                const float dov = ds[s * SX + p];
                ddsum = fmaf(dov, xs[s * SX + p], ddsum);
                a.dx[((id.row0 + s) * H + id.hd) * P + p] = Dh * dov + a1[r][q] + F * a2[r][q];
            }
        }
    }
    {  // dB = Wb^T C + F_s x G^T, and B_s^T G x_s
        const Tile<kQ, N> t;
        float a1[Tile<kQ, N>::TI][Tile<kQ, N>::TJ], a2[Tile<kQ, N>::TI][Tile<kQ, N>::TJ];
        zero<kQ, N>(a1);
        zero<kQ, N>(a2);
        mac<kQ, N, kQ>(t, a1, [&](int s, int i) { return Wb[i * kSQ + s]; }, [&](int i, int n) { return Cs[i * SN + n]; });
        mac<kQ, N, P>(t, a2, [&](int s, int p) { return xs[s * SX + p]; }, [&](int p, int n) { return Hs[p * SN + n]; });
#pragma unroll
        for (int r = 0; r < Tile<kQ, N>::TI; ++r) {
            const int s = t.row(r);
            const float F = expf(tot - scum[s]) * sdt[s];
            float fsum = 0.f;
#pragma unroll
            for (int q = 0; q < Tile<kQ, N>::TJ; ++q) {
                const int n = t.col(q);
                fsum = fmaf(Bs[s * SN + n], a2[r][q], fsum);
                if (s < id.valid) atomicAdd(&a.dB[((id.row0 + s) * G + id.g) * N + n], a1[r][q] + F * a2[r][q]);
            }
            atomicAdd(&sdF[s], fsum);
        }
    }
    __syncthreads();  // Hs is read by every thread above
    {
        const float* hp = a.st + cidx * PN;
        for (int i = threadIdx.x; i < P * N; i += kNT) Hs[(i / N) * SN + i % N] = hp[i];
    }
    __syncthreads();
    {  // dC = Wb B + e^{cum_t} do h_p^T, and C_t . (e^{cum_t} h_p do_t)
        const Tile<kQ, N> t;
        float a1[Tile<kQ, N>::TI][Tile<kQ, N>::TJ], a2[Tile<kQ, N>::TI][Tile<kQ, N>::TJ];
        zero<kQ, N>(a1);
        zero<kQ, N>(a2);
        mac<kQ, N, kQ>(t, a1, [&](int i, int s) { return Wb[i * kSQ + s]; }, [&](int s, int n) { return Bs[s * SN + n]; });
        mac<kQ, N, P>(t, a2, [&](int i, int p) { return ds[i * SX + p]; }, [&](int p, int n) { return Hs[p * SN + n]; });
#pragma unroll
        for (int r = 0; r < Tile<kQ, N>::TI; ++r) {
            const int i = t.row(r);
            const float ec = expf(scum[i]);
            float csum = 0.f;
#pragma unroll
            for (int q = 0; q < Tile<kQ, N>::TJ; ++q) {
                const int n = t.col(q);
                const float u = ec * a2[r][q];
                csum = fmaf(Cs[i * SN + n], u, csum);
                if (i < id.valid) atomicAdd(&a.dC[((id.row0 + i) * G + id.g) * N + n], a1[r][q] + u);
            }
            atomicAdd(&sdc2[i], csum);
        }
    }
    ddsum = block_sum(ddsum, red);  // also publishes sdF, sdc2
    // per step: d cum, then d a by a reverse running sum, then d(dt) through softplus
    float* fdf = Vb;  // F_s B_s^T G x_s, reusing the free Q x Q buffer
    if (threadIdx.x < kQ) {
        const int s = threadIdx.x;
        const float eT = expf(tot - scum[s]);
        const float F = eT * sdt[s];
        fdf[s] = F * sdF[s];
        sdc[s] = sdc[s] - sdt[s] * sdw[s] + sdc2[s] - F * sdF[s];
        sdw[s] += eT * sdF[s];
    }
    __syncthreads();
    float pa = 0.f, pb = 0.f;
    if (threadIdx.x < kQ) {
        const int s = threadIdx.x;
        float dtot = expf(tot) * dot;
        for (int j = 0; j < kQ; ++j) dtot += fdf[j];
        float da = dtot;
        for (int j = s; j < kQ; ++j) da += sdc[j];
        const float ddt = da * a.A[id.hd] + sdw[s];
        const float raw = a.softplus ? ddt * sigmoid_accurate(su[s]) : ddt;
        if (s < id.valid) {
            a.ddt[(id.row0 + s) * H + id.hd] = raw;
            pa = da * sdt[s];
            pb = raw;
        }
    }
    pa = block_sum(pa, red);
    pb = block_sum(pb, red);
    if (threadIdx.x == 0) {
        const size_t gc = static_cast<size_t>(id.q) * a.nch + id.c;
        const size_t all = static_cast<size_t>(a.batch) * H * a.nch;
        a.part[gc] = pa;
        a.part[all + gc] = ddsum;
        a.part[2 * all + gc] = pb;
    }
}

// dA, dD, ddt_bias of head h: sums of the per-chunk partials in a fixed order
__global__ void __launch_bounds__(256) ssd_bwd_reduce(CkArgs a, float* dA, float* dD, float* dbias) {
    __shared__ float red[32];
    const int hd = blockIdx.x % a.nheads, k = blockIdx.x / a.nheads;
    float* out = k == 0 ? dA : (k == 1 ? dD : dbias);
    if (out == nullptr) return;
    const size_t all = static_cast<size_t>(a.batch) * a.nheads * a.nch;
    const float* p = a.part + k * all;
    const int per = a.batch * a.nch;
    float v = 0.f;
    for (int i = threadIdx.x; i < per; i += blockDim.x) {
        const int b = i / a.nch, c = i % a.nch;
        v += p[(static_cast<size_t>(b) * a.nheads + hd) * a.nch + c];
    }
    v = block_sum(v, red);
    if (threadIdx.x == 0) out[hd] = v;
}

template <int N, int P>
constexpr size_t smem_outputs() {
    return sizeof(float) * (2 * kQ * (P + 1) + 2 * kQ * (N + 1) + P * (N + 1) + kQ * kSQ + 3 * kQ);
}
template <int N, int P>
constexpr size_t smem_grads() {
    return sizeof(float) * (2 * kQ * (P + 1) + 2 * kQ * (N + 1) + P * (N + 1) + 3 * kQ * kSQ + 7 * kQ + 32);
}
template <int N, int P>
constexpr size_t smem_states() {
    return sizeof(float) * (kQ * (P + 1) + kQ * (N + 1) + 3 * kQ);
}

// the supported (dstate, headdim) pairs
bool shape_ok(int N, int P) {
    return (N == 128 && P == 64) || (N == 64 && P == 64) || (N == 128 && P == 32) || (N == 64 && P == 32);
}

struct CkWs {
    size_t st, adj, tot, part, bytes;
    int nq;  // sequences per slice
};

size_t al256(size_t v) { return (v + 255) / 256 * 256; }

CkWs ck_ws(const ssd_bwd_params& p) {
    const ssd_params& f = p.fwd;
    const size_t nch = (static_cast<size_t>(f.seqlen) + kQ - 1) / kQ;
    const size_t seqs = static_cast<size_t>(f.batch) * f.nheads;
    const size_t per_seq = 2 * nch * f.headdim * f.dstate * sizeof(float);
    // the chunk states and adjoints of a slice take at most the room of x and dy; the
    // slices are made equal
    const size_t es = f.in_dtype == SSM_BF16 ? 2 : 4;
    const size_t budget = 2 * static_cast<size_t>(f.batch) * f.seqlen * f.nheads * f.headdim * es;
    size_t nq = budget / per_seq;
    if (nq < 1) nq = 1;
    if (nq > seqs) nq = seqs;
    const size_t slices = (seqs + nq - 1) / nq;
    nq = (seqs + slices - 1) / slices;
    CkWs w;
    w.nq = static_cast<int>(nq);
    const size_t slice = al256(nq * nch * f.headdim * f.dstate * sizeof(float));
    w.st = 0;
    w.adj = slice;
    w.tot = 2 * slice;
    w.part = w.tot + al256(seqs * nch * sizeof(float));
    w.bytes = w.part + al256(3 * seqs * nch * sizeof(float));
    return w;
}

template <typename Tin, int N, int P>
cudaError_t launch_shape(const ssd_bwd_params& p, void* ws, cudaStream_t s) {
    const ssd_params& f = p.fwd;
    const CkWs w = ck_ws(p);
    unsigned char* base = static_cast<unsigned char*>(ws);
    CkArgs a{};
    a.batch = f.batch;
    a.seqlen = f.seqlen;
    a.nheads = f.nheads;
    a.ngroups = f.ngroups;
    a.hpg = f.nheads / f.ngroups;
    a.nch = (f.seqlen + kQ - 1) / kQ;
    a.softplus = f.dt_softplus;
    a.x = f.x; a.dt = f.dt; a.dt_bias = f.dt_bias; a.A = f.A; a.B = f.B; a.C = f.C; a.D = f.D_skip; a.z = f.z;
    a.h0 = f.h0; a.dy = p.dy; a.dh_final = p.dh_final;
    a.dx = p.dx; a.ddt = p.ddt; a.dz = p.dz; a.dB = p.dB; a.dC = p.dC; a.dh0 = p.dh0;
    a.st = reinterpret_cast<float*>(base + w.st);
    a.adj = reinterpret_cast<float*>(base + w.adj);
    a.tot = reinterpret_cast<float*>(base + w.tot);
    a.part = reinterpret_cast<float*>(base + w.part);
    cudaError_t e;
    const size_t nbc = static_cast<size_t>(f.batch) * f.seqlen * f.ngroups * f.dstate;
    if ((e = cudaMemsetAsync(p.dB, 0, nbc * sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(p.dC, 0, nbc * sizeof(float), s)) != cudaSuccess) return e;
    auto k1 = ssd_bwd_chunk_states<Tin, N, P>;
    auto k3 = ssd_bwd_chunk_outputs<Tin, N, P>;
    auto k5 = ssd_bwd_chunk_grads<Tin, N, P>;
    if ((e = set_smem_attr(reinterpret_cast<const void*>(k1), static_cast<int>(smem_states<N, P>()))) != cudaSuccess)
        return e;
    if ((e = set_smem_attr(reinterpret_cast<const void*>(k3), static_cast<int>(smem_outputs<N, P>()))) != cudaSuccess)
        return e;
    if ((e = set_smem_attr(reinterpret_cast<const void*>(k5), static_cast<int>(smem_grads<N, P>()))) != cudaSuccess)
        return e;
    const int seqs = f.batch * f.nheads, PN = P * N;
    for (int q0 = 0; q0 < seqs; q0 += w.nq) {
        a.q0 = q0;
        a.nq = seqs - q0 < w.nq ? seqs - q0 : w.nq;
        const unsigned chunks = static_cast<unsigned>(a.nq) * a.nch;
        const unsigned pass_grid = static_cast<unsigned>((static_cast<long long>(a.nq) * PN + 255) / 256);
        k1<<<chunks, kNT, smem_states<N, P>(), s>>>(a);
        ssd_bwd_pass<false><<<pass_grid, 256, 0, s>>>(a, PN);
        k3<<<chunks, kNT, smem_outputs<N, P>(), s>>>(a);
        ssd_bwd_pass<true><<<pass_grid, 256, 0, s>>>(a, PN);
        k5<<<chunks, kNT, smem_grads<N, P>(), s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ssd_bwd_reduce<<<3 * f.nheads, 256, 0, s>>>(a, p.dA, p.dD_skip, p.ddt_bias);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t dispatch_shape(const ssd_bwd_params& p, void* ws, cudaStream_t s) {
    const int N = p.fwd.dstate, P = p.fwd.headdim;
    if (N == 128 && P == 64) return launch_shape<Tin, 128, 64>(p, ws, s);
    if (N == 64 && P == 64) return launch_shape<Tin, 64, 64>(p, ws, s);
    if (N == 128 && P == 32) return launch_shape<Tin, 128, 32>(p, ws, s);
    if (N == 64 && P == 32) return launch_shape<Tin, 64, 32>(p, ws, s);
    return cudaErrorInvalidValue;
}

}  // namespace

bool ssd_chunked_bwd_supported(const ssd_bwd_params& p) {
    const ssd_params& f = p.fwd;
    return f.disc == SSM_DISC_EXP_EULER && f.seqlen >= 1 && f.in_dtype == f.out_dtype &&
           shape_ok(f.dstate, f.headdim) && static_cast<long long>(f.batch) * f.nheads <= (1 << 20);
}

size_t ssd_chunked_bwd_workspace_size(const ssd_bwd_params& p) {
    return ssd_chunked_bwd_supported(p) ? ck_ws(p).bytes : 0;
}

cudaError_t ssd_chunked_bwd_launch(const ssd_bwd_params& p, void* workspace, cudaStream_t s) {
    return p.fwd.in_dtype == SSM_BF16 ? dispatch_shape<bf16_t>(p, workspace, s)
                                      : dispatch_shape<float>(p, workspace, s);
}

}  // namespace ssm
