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
// shared memory as float32.  Each product is laid out so that both of its operands are
// read with 16-byte loads: every operand is stored with either the contraction index or
// the output index contiguous, whichever the product needs (the adjoint is kept both ways
// in the gradient launch); a thread computes a 4 x TJ tile (4 x 8 lanes per warp) and takes
// four steps of the contraction per load.  Global loads are issued in batches before their
// stores to shared memory (the state entering the chunk by asynchronous copies, the
// adjoint while the dC products run), and dB, dC are added with 16-byte vector atomics.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kQ = 64;     // steps per chunk
// threads per CTA of the chunk launches (512 measured slower: smaller tiles per thread)
constexpr int kNT = 256;
// unrolling of the products' four-step inner loop: 2 measured fastest (1: 2.84, 2: 2.76,
// 8: 3.23 ms per call on the 130m SSD shape; 8 overflows the instruction cache)
constexpr int kUnroll = 2;
constexpr int kLQ = kQ + 4;  // row length of the Q x Q operands

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

// Operand layouts in shared memory, rows padded to width + 4 floats (16-byte aligned, and
// successive rows start four banks apart):
//   KC: the contraction index k is contiguous (element (x, k) at x * ld + k);
//   XC: the other index is contiguous (element (x, k) at k * ld + x).
enum Lay { KC = 0, XC = 1 };

// A thread's share of an I x J product.  Warp w covers rows 16 (w / WJ) .. + 15 and
// columns 8 TJ (w % WJ) .. + 8 TJ - 1; lane 8 ti + tj holds 4 rows and TJ columns, spread
// so that every 16-byte load of a warp touches each bank at most once: rows ti + 4 r (A
// in KC) or 4 ti + r (A in XC), columns tj + 8 q (B in KC) or 4 tj + 32 (q / 4) + q % 4
// (B in XC; 2 tj + q when TJ = 2).
template <int I, int J, Lay LA, Lay LB>
struct Frag {
    static constexpr int TJ = I * J / (kNT * 4);
    static constexpr int WJ = J / (8 * TJ);
    static_assert(I % 16 == 0 && (TJ == 2 || TJ % 4 == 0) && (I / 16) * WJ * 32 == kNT, "fragment shape");
    int ib, jb, ti, tj;
    __device__ __forceinline__ Frag() {
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        ib = (w / WJ) * 16;
        jb = (w % WJ) * 8 * TJ;
        ti = l >> 3;
        tj = l & 7;
    }
    __device__ __forceinline__ int row(int r) const { return LA == KC ? ib + ti + 4 * r : ib + 4 * ti + r; }
    __device__ __forceinline__ int col(int q) const {
        if (LB == KC) return jb + tj + 8 * q;
        if (TJ == 2) return jb + 2 * tj + q;
        return jb + 4 * tj + 32 * (q / 4) + q % 4;
    }
};

// acc[r][q] += sum_k A(row r, k) B(col q, k), four k per step, 16-byte (8-byte) loads
template <int K, int I, int J, Lay LA, Lay LB>
__device__ __forceinline__ void mac(const Frag<I, J, LA, LB>& f, float (&acc)[4][Frag<I, J, LA, LB>::TJ],
                                    const float* A, int lda, const float* B, int ldb) {
    constexpr int TJ = Frag<I, J, LA, LB>::TJ;
    static_assert(K % 4 == 0, "contraction length");
#pragma unroll kUnroll
    for (int k0 = 0; k0 < K; k0 += 4) {
        float a[4][4], b[4][TJ];  // [k - k0][r], [k - k0][q]
        if constexpr (LA == KC) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 v = *reinterpret_cast<const float4*>(A + f.row(r) * lda + k0);
                a[0][r] = v.x;
                a[1][r] = v.y;
                a[2][r] = v.z;
                a[3][r] = v.w;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 v = *reinterpret_cast<const float4*>(A + (k0 + kk) * lda + f.row(0));
                a[kk][0] = v.x;
                a[kk][1] = v.y;
                a[kk][2] = v.z;
                a[kk][3] = v.w;
            }
        }
        if constexpr (LB == KC) {
#pragma unroll
            for (int q = 0; q < TJ; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(B + f.col(q) * ldb + k0);
                b[0][q] = v.x;
                b[1][q] = v.y;
                b[2][q] = v.z;
                b[3][q] = v.w;
            }
        } else if constexpr (TJ == 2) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float2 v = *reinterpret_cast<const float2*>(B + (k0 + kk) * ldb + f.col(0));
                b[kk][0] = v.x;
                b[kk][1] = v.y;
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int q4 = 0; q4 < TJ / 4; ++q4) {
                    const float4 v = *reinterpret_cast<const float4*>(B + (k0 + kk) * ldb + f.col(4 * q4));
                    b[kk][4 * q4] = v.x;
                    b[kk][4 * q4 + 1] = v.y;
                    b[kk][4 * q4 + 2] = v.z;
                    b[kk][4 * q4 + 3] = v.w;
                }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < TJ; ++q) acc[r][q] = fmaf(a[kk][r], b[kk][q], acc[r][q]);
    }
}

template <int TJ>
__device__ __forceinline__ void zero(float (&acc)[4][TJ]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < TJ; ++q) acc[r][q] = 0.f;
}

// acc into a global [I][ld] float32 array (columns of a thread contiguous by fours in XC)
template <int I, int J, Lay LA, Lay LB>
__device__ __forceinline__ void store_tile(const Frag<I, J, LA, LB>& f,
                                           const float (&acc)[4][Frag<I, J, LA, LB>::TJ], float* out, int ld) {
    constexpr int TJ = Frag<I, J, LA, LB>::TJ;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if constexpr (LB == XC && TJ % 4 == 0) {
#pragma unroll
            for (int q4 = 0; q4 < TJ / 4; ++q4)
                *reinterpret_cast<float4*>(out + static_cast<size_t>(f.row(r)) * ld + f.col(4 * q4)) =
                    make_float4(acc[r][4 * q4], acc[r][4 * q4 + 1], acc[r][4 * q4 + 2], acc[r][4 * q4 + 3]);
        } else {
#pragma unroll
            for (int q = 0; q < TJ; ++q) out[static_cast<size_t>(f.row(r)) * ld + f.col(q)] = acc[r][q];
        }
    }
}

// 16-byte vector of T as float32
__device__ __forceinline__ void unpack16(const uint4& v, float* f, float) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float* f, bf16_t) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = lo_bf16(w[j]);
        f[2 * j + 1] = hi_bf16(w[j]);
    }
}

// Rows t < Q of a tensor (row t at element base + t * stride, W contiguous elements of T)
// into shared memory as float32 rows of length ldst, zero from row `rows_valid` on.
// Every thread issues all of its 16-byte loads before its first store, so their
// latencies overlap.  With CT, also the transpose: element (t, w) at ct[w * ldct + t].
template <typename T, int W, bool CT = false>
__device__ __forceinline__ void load_rows(float* dst, int ldst, const void* src, size_t base, size_t stride,
                                          int rows_valid, float* ct = nullptr, int ldct = 0) {
    constexpr int V = 16 / sizeof(T);  // elements per load
    constexpr int RV = W / V;          // loads per row
    constexpr int PER = kQ * RV / kNT;
    static_assert(W % V == 0 && (kQ * RV) % kNT == 0, "load shape");
    const T* g = static_cast<const T*>(src) + base;
    uint4 v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = threadIdx.x + j * kNT, t = i / RV, w = (i % RV) * V;
        v[j] = t < rows_valid ? *reinterpret_cast<const uint4*>(g + t * stride + w) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = threadIdx.x + j * kNT, t = i / RV, w = (i % RV) * V;
        float f[V];
        unpack16(v[j], f, T{});
#pragma unroll
        for (int e = 0; e < V; e += 4)
            *reinterpret_cast<float4*>(dst + t * ldst + w + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        if constexpr (CT) {
#pragma unroll
            for (int e = 0; e < V; ++e) ct[(w + e) * ldct + t] = f[e];
        }
    }
}

// The thread's j-th 16-byte piece (p, n .. n + 3) of a P x N state block [p][n]: a warp
// takes 16 rows and 8 columns, lane l row 16 rb + l % 16 and columns 4 (2 nb + l / 16)
// .. + 3, so that the 32 lanes of a transposed store (n * ld + p, ld = 4 mod 32) fall in
// distinct banks and each global load still reads whole 32-byte sectors.
template <int N, int P>
__device__ __forceinline__ void state_elem(int j, int& p, int& n) {
    static_assert(P % 16 == 0 && N % 8 == 0, "state shape");
    const int g = static_cast<int>(threadIdx.x) + j * kNT, c = g >> 5, l = g & 31;
    p = (c % (P / 16)) * 16 + (l & 15);
    n = ((c / (P / 16)) * 2 + (l >> 4)) * 4;
}

// The P x N float32 block src ([p][n]) into shared memory: as (n, p) at dst[n * ld + p]
// (TR) or as (p, n) at dst[p * ld + n]; with `other` (the same shape), also returns the
// thread's part of sum(src * other).  Loads first, then stores.
template <int N, int P, bool TR>
__device__ __forceinline__ float load_state(float* dst, int ld, const float* src, const float* other = nullptr) {
    constexpr int PER = P * N / 4 / kNT;
    static_assert((P * N / 4) % kNT == 0, "state shape");
    float4 v[PER], o[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        int p, n;
        state_elem<N, P>(j, p, n);
        v[j] = *reinterpret_cast<const float4*>(src + p * N + n);
        if (other) o[j] = *reinterpret_cast<const float4*>(other + p * N + n);
    }
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        int p, n;
        state_elem<N, P>(j, p, n);
        if (other) dot += v[j].x * o[j].x + v[j].y * o[j].y + v[j].z * o[j].z + v[j].w * o[j].w;
        if constexpr (TR) {
            dst[n * ld + p] = v[j].x;
            dst[(n + 1) * ld + p] = v[j].y;
            dst[(n + 2) * ld + p] = v[j].z;
            dst[(n + 3) * ld + p] = v[j].w;
        } else {
            *reinterpret_cast<float4*>(dst + p * ld + n) = v[j];
        }
    }
    return dot;
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
    constexpr int LX = P + 4, LN = N + 4;
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                // [Q][LX] x_s F_s
    float* Bs = xs + kQ * LX;      // [Q][LN]
    float* su = Bs + kQ * LN;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, P>(xs, LX, a.x, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                      id.valid);
    load_rows<Tin, N>(Bs, LN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    __syncthreads();
    const float tot = scum[kQ - 1];
    for (int i = threadIdx.x; i < kQ * P; i += kNT) {
        const int s = i / P, p = i % P;
        xs[s * LX + p] *= expf(tot - scum[s]) * sdt[s];
    }
    __syncthreads();
    const Frag<P, N, XC, XC> f;
    float acc[4][Frag<P, N, XC, XC>::TJ];
    zero(acc);
    mac<kQ>(f, acc, xs, LX, Bs, LN);
    store_tile(f, acc, a.st + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N, N);
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
    constexpr int LX = P + 4, LN = N + 4;
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                // [Q][LX]
    float* ds = xs + kQ * LX;      // [Q][LX] do_t e^{cum_t}
    float* Bs = ds + kQ * LX;      // [Q][LN]
    float* Cs = Bs + kQ * LN;      // [Q][LN]
    float* Hs = Cs + kQ * LN;      // [N][LX] state entering the chunk, element (n, p)
    float* Wa = Hs + N * LX;       // [Q][kLQ]
    float* su = Wa + kQ * kLQ;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, P>(xs, LX, a.x, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                      id.valid);
    load_rows<Tin, N>(Bs, LN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    load_rows<Tin, N>(Cs, LN, a.C, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    load_state<N, P, true>(Hs, LX, a.st + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N);
    // dy and z of this thread's outputs, in flight during the first product
    using FY = Frag<kQ, P, KC, XC>;
    const FY fy;
    float dyv[4][FY::TJ], zv[4][FY::TJ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < FY::TJ; ++q) {
            const int i = fy.row(r);
            const size_t gi = ((id.row0 + i) * H + id.hd) * P + fy.col(q);
            dyv[r][q] = i < id.valid ? ld<Tin>(a.dy, gi) : 0.f;
            zv[r][q] = (a.z && i < id.valid) ? ld<Tin>(a.z, gi) : 0.f;
        }
    __syncthreads();
    {  // Wa = (C B^T) E dt_s, lower triangle
        const Frag<kQ, kQ, KC, KC> f;
        float acc[4][Frag<kQ, kQ, KC, KC>::TJ];
        zero(acc);
        mac<N>(f, acc, Cs, LN, Bs, LN);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < Frag<kQ, kQ, KC, KC>::TJ; ++q) {
                const int i = f.row(r), s = f.col(q);
                Wa[i * kLQ + s] = s <= i ? acc[r][q] * expf(scum[i] - scum[s]) * sdt[s] : 0.f;
            }
    }
    __syncthreads();
    {  // o = Wa x + e^{cum_t} C h_p + D x, then the gate
        using F = FY;
        const F& f = fy;
        float a1[4][F::TJ], a2[4][F::TJ];
        zero(a1);
        zero(a2);
        mac<kQ>(f, a1, Wa, kLQ, xs, LX);
        mac<N>(f, a2, Cs, LN, Hs, LX);
        const float Dh = a.D ? a.D[id.hd] : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = f.row(r);
            const float ec = expf(scum[i]);
#pragma unroll
            for (int q = 0; q < F::TJ; ++q) {
                const int p = f.col(q);
                float dov = 0.f;
                if (i < id.valid) {
                    const size_t gi = ((id.row0 + i) * H + id.hd) * P + p;
                    const float o = a1[r][q] + ec * a2[r][q] + Dh * xs[i * LX + p];
                    const float dout = dyv[r][q];
                    if (a.z) {
                        const float zz = zv[r][q];
                        const float sg = sigmoid_accurate(zz);
                        dov = dout * zz * sg;
                        a.dz[gi] = dout * o * sg * (1.f + zz * (1.f - sg));
                    } else {
                        dov = dout;
                    }
                    a.dx[gi] = dov;
                }
                ds[i * LX + p] = dov * ec;
            }
        }
    }
    __syncthreads();
    {  // R[p][n] = sum_t ds[t][p] C[t][n]
        const Frag<P, N, XC, XC> f;
        float acc[4][Frag<P, N, XC, XC>::TJ];
        zero(acc);
        mac<kQ>(f, acc, ds, LX, Cs, LN);
        store_tile(f, acc, a.adj + (static_cast<size_t>(id.ql) * a.nch + id.c) * P * N, N);
    }
}

// ---------------------------------------------------------------------------------------
// 5. gradients of the chunk
// ---------------------------------------------------------------------------------------
template <typename Tin, int N, int P>
__global__ void __launch_bounds__(kNT, 1) ssd_bwd_chunk_grads(CkArgs a) {
    constexpr int LX = P + 4, LN = N + 4;
    constexpr int GB = N * LX > P * LN ? N * LX : P * LN;
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                // [Q][LX]
    float* ds = xs + kQ * LX;      // [Q][LX] do
    float* Bs = ds + kQ * LX;      // [Q][LN]
    float* Cs = Bs + kQ * LN;      // [Q][LN]
    float* Gn = Cs + kQ * LN;      // [P][LN] adjoint leaving the chunk, element (p, n)
    float* Gb = Gn + P * LN;       // state entering the chunk [P][LN], then the adjoint as (n, p) [N][LX]
    float* WaT = Gb + GB;          // [Q][kLQ] (C B^T E dt_s)[t][s] at s * kLQ + t
    float* Wb = WaT + kQ * kLQ;    // [Q][kLQ] (T E dt_s)[t][s] at t * kLQ + s
    float* WbT = Wb + kQ * kLQ;    // [Q][kLQ] the same at s * kLQ + t
    float* su = WbT + kQ * kLQ;
    float* sdt = su + kQ;
    float* scum = sdt + kQ;
    float* sdw = scum + kQ;        // dt_s as input weight: intra-chunk part
    float* sdc = sdw + kQ;         // d cum, intra-chunk part (dt-weighted row sums)
    float* sdc2 = sdc + kQ;        // d cum, through the state entering the chunk
    float* sdF = sdc2 + kQ;        // B_s^T G x_s
    float* colp = sdF + kQ;        // [4][Q] column sums of C B^T E T per warp row
    float* red = colp + 4 * kQ;    // [32]
    const ChunkId id(a);
    const int H = a.nheads, G = a.ngroups;
    const size_t PN = static_cast<size_t>(P) * N;
    const size_t cidx = static_cast<size_t>(id.ql) * a.nch + id.c;
    chunk_steps<Tin>(a, id.b, id.hd, id.c, su, sdt, scum);
    load_rows<Tin, P>(xs, LX, a.x, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                      id.valid);
    load_rows<float, P>(ds, LX, a.dx, id.row0 * H * P + static_cast<size_t>(id.hd) * P, static_cast<size_t>(H) * P,
                        id.valid);
    load_rows<Tin, N>(Bs, LN, a.B, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    load_rows<Tin, N>(Cs, LN, a.C, (id.row0 * G + id.g) * N, static_cast<size_t>(G) * N, id.valid);
    {  // the state entering the chunk into Gb as (p, n), asynchronously
        const float* hp = a.st + cidx * PN;
        for (int i4 = threadIdx.x; i4 < P * N / 4; i4 += kNT) {
            const int i = 4 * i4;
            cp_async16(Gb + (i / N) * LN + i % N, hp + i, 16);
        }
        cp_async_commit();
    }
    if (threadIdx.x < kQ) {
        sdc[threadIdx.x] = 0.f;
        sdc2[threadIdx.x] = 0.f;
        sdF[threadIdx.x] = 0.f;
    }
    __syncthreads();
    {  // C B^T and T = do x^T; the masked, decayed, weighted forms; sums of C B^T E T
        using F = Frag<kQ, kQ, KC, KC>;
        const F f;
        float a1[4][F::TJ], a2[4][F::TJ];
        zero(a1);
        zero(a2);
        mac<N>(f, a1, Cs, LN, Bs, LN);
        mac<P>(f, a2, ds, LX, xs, LX);
        float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[F::TJ];
#pragma unroll
        for (int q = 0; q < F::TJ; ++q) cp[q] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < F::TJ; ++q) {
                const int i = f.row(r), s = f.col(q);
                float w1 = 0.f, w2 = 0.f, v = 0.f;
                if (s <= i) {
                    const float e = expf(scum[i] - scum[s]);
                    v = a1[r][q] * e * a2[r][q];
                    w1 = a1[r][q] * e * sdt[s];
                    w2 = a2[r][q] * e * sdt[s];
                }
                WaT[s * kLQ + i] = w1;
                Wb[i * kLQ + s] = w2;
                WbT[s * kLQ + i] = w2;
                rp[r] = fmaf(sdt[s], v, rp[r]);
                cp[q] += v;
            }
        // rows: the 8 lanes of a row, then the two warps of a row (atomic adds of two
        // terms onto zero, so the order does not matter); columns: the 4 lanes of a
        // column, then the four warp rows in a fixed order below
#pragma unroll
        for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) rp[r] += __shfl_xor_sync(0xffffffffu, rp[r], off);
            if (f.tj == 0) atomicAdd(&sdc[f.row(r)], rp[r]);
        }
#pragma unroll
        for (int q = 0; q < F::TJ; ++q) {
            cp[q] += __shfl_xor_sync(0xffffffffu, cp[q], 8);
            cp[q] += __shfl_xor_sync(0xffffffffu, cp[q], 16);
            if (f.ti == 0) colp[(f.ib / 16) * kQ + f.col(q)] = cp[q];
        }
    }
    __syncthreads();
    if (threadIdx.x < kQ) {
        const int s = threadIdx.x;
        sdw[s] = ((colp[s] + colp[kQ + s]) + colp[2 * kQ + s]) + colp[3 * kQ + s];
    }
    cp_async_wait<0>();
    __syncthreads();  // the state entering the chunk is in Gb
    // the adjoint leaving the chunk, in flight during the dC products
    constexpr int GPER = P * N / 4 / kNT;
    float4 gv[GPER];
#pragma unroll
    for (int j = 0; j < GPER; ++j) {
        int pp, n;
        state_elem<N, P>(j, pp, n);
        gv[j] = *reinterpret_cast<const float4*>(a.adj + cidx * PN + pp * N + n);
    }
    const float tot = scum[kQ - 1];
    const float Dh = a.D ? a.D[id.hd] : 0.f;
    {  // dC = (T E dt) B + e^{cum_t} h_p do, and C_t . (e^{cum_t} h_p do_t)
        using F = Frag<kQ, N, KC, XC>;
        const F f;
        float a1[4][F::TJ], a2[4][F::TJ];
        zero(a1);
        zero(a2);
        mac<kQ>(f, a1, Wb, kLQ, Bs, LN);
        mac<P>(f, a2, ds, LX, Gb, LN);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = f.row(r);
            const float ec = expf(scum[i]);
            float csum = 0.f, u[F::TJ];
#pragma unroll
            for (int q = 0; q < F::TJ; ++q) {
                u[q] = ec * a2[r][q];
                csum = fmaf(Cs[i * LN + f.col(q)], u[q], csum);
            }
            if (i < id.valid) {
                float* dst = a.dC + ((id.row0 + i) * G + id.g) * N;
#pragma unroll
                for (int q = 0; q < F::TJ; q += 4)
                    atomicAdd(reinterpret_cast<float4*>(dst + f.col(q)),
                              make_float4(a1[r][q] + u[q], a1[r][q + 1] + u[q + 1], a1[r][q + 2] + u[q + 2],
                                          a1[r][q + 3] + u[q + 3]));
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) csum += __shfl_xor_sync(0xffffffffu, csum, off);
            if (f.tj == 0) atomicAdd(&sdc2[i], csum);  // two warps per row
        }
    }
    // <adjoint, state entering the chunk>, then the adjoint into Gb as (n, p)
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < GPER; ++j) {
        int pp, n;
        state_elem<N, P>(j, pp, n);
        const float4 h = *reinterpret_cast<const float4*>(Gb + pp * LN + n);
        dot += gv[j].x * h.x + gv[j].y * h.y + gv[j].z * h.z + gv[j].w * h.w;
    }
    __syncthreads();  // every read of the state in Gb is done
#pragma unroll
    for (int j = 0; j < GPER; ++j) {
        int pp, n;
        state_elem<N, P>(j, pp, n);
        *reinterpret_cast<float4*>(Gn + pp * LN + n) = gv[j];
        Gb[n * LX + pp] = gv[j].x;
        Gb[(n + 1) * LX + pp] = gv[j].y;
        Gb[(n + 2) * LX + pp] = gv[j].z;
        Gb[(n + 3) * LX + pp] = gv[j].w;
    }
    dot = block_sum(dot, red);  // includes the barrier that publishes Gb and Gn
    float ddsum = 0.f;  // sum do x (dD)
    {  // dx = D do + (C B^T E dt)^T do + F_s B G
        using F = Frag<kQ, P, KC, XC>;
        const F f;
        float a1[4][F::TJ], a2[4][F::TJ];
        zero(a1);
        zero(a2);
        mac<kQ>(f, a1, WaT, kLQ, ds, LX);
        mac<N>(f, a2, Bs, LN, Gb, LX);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int s = f.row(r);
            if (s >= id.valid) continue;
            const float Fs = expf(tot - scum[s]) * sdt[s];
#pragma unroll
            for (int q = 0; q < F::TJ; ++q) {
                const int p = f.col(q);
                const float dov = ds[s * LX + p];
                ddsum = fmaf(dov, xs[s * LX + p], ddsum);
                a.dx[((id.row0 + s) * H + id.hd) * P + p] = Dh * dov + a1[r][q] + Fs * a2[r][q];
            }
        }
    }
    {  // dB = (T E dt)^T C + F_s G x, and B_s^T G x_s
        using F = Frag<kQ, N, KC, XC>;
        const F f;
        float a1[4][F::TJ], a2[4][F::TJ];
        zero(a1);
        zero(a2);
        mac<kQ>(f, a1, WbT, kLQ, Cs, LN);
        mac<P>(f, a2, xs, LX, Gn, LN);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int s = f.row(r);
            const float Fs = expf(tot - scum[s]) * sdt[s];
            float fsum = 0.f;
#pragma unroll
            for (int q = 0; q < F::TJ; ++q) fsum = fmaf(Bs[s * LN + f.col(q)], a2[r][q], fsum);
            if (s < id.valid) {
                float* dst = a.dB + ((id.row0 + s) * G + id.g) * N;
#pragma unroll
                for (int q = 0; q < F::TJ; q += 4)
                    atomicAdd(reinterpret_cast<float4*>(dst + f.col(q)),
                              make_float4(a1[r][q] + Fs * a2[r][q], a1[r][q + 1] + Fs * a2[r][q + 1],
                                          a1[r][q + 2] + Fs * a2[r][q + 2], a1[r][q + 3] + Fs * a2[r][q + 3]));
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) fsum += __shfl_xor_sync(0xffffffffu, fsum, off);
            if (f.tj == 0) atomicAdd(&sdF[s], fsum);  // two warps per row
        }
    }
    ddsum = block_sum(ddsum, red);  // also publishes sdF, sdc2
    // per step: d cum, then d a by a reverse running sum, then d(dt) through softplus
    float* fdf = colp;  // F_s B_s^T G x_s
    if (threadIdx.x < kQ) {
        const int s = threadIdx.x;
        const float eT = expf(tot - scum[s]);
        const float Fs = eT * sdt[s];
        fdf[s] = Fs * sdF[s];
        sdc[s] = sdc[s] - sdt[s] * sdw[s] + sdc2[s] - Fs * sdF[s];
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
    return sizeof(float) * (2 * kQ * (P + 4) + 2 * kQ * (N + 4) + N * (P + 4) + kQ * kLQ + 3 * kQ);
}
template <int N, int P>
constexpr size_t smem_grads() {
    constexpr int GB = N * (P + 4) > P * (N + 4) ? N * (P + 4) : P * (N + 4);
    return sizeof(float) * (2 * kQ * (P + 4) + 2 * kQ * (N + 4) + P * (N + 4) + GB + 3 * kQ * kLQ + 11 * kQ + 32);
}
template <int N, int P>
constexpr size_t smem_states() {
    return sizeof(float) * (kQ * (P + 4) + kQ * (N + 4) + 3 * kQ);
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
