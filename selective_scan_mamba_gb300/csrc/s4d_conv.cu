// s4d_conv.cu -- S4D convolution form on the GPU: y = K * u + D u by FFT (sm_103a).
//
// ("From S4 to Mamba-3", 03/System, s4_minimal.py: S4D trains as one FFT convolution with
// its kernel K_l = Re sum_n C Bbar Abar^l; 09/Validation: the convolution equals the
// recurrent form from a zero state.)  The causal convolution of a length-L row with the
// length-L kernel is the first L points of the cyclic convolution of both, zero-padded
// to N = 2^ceil(log2 2L): y = IFFT(FFT(K) . FFT(u)) restricted to t < L.
//
// Two launches:
//   1. s4d_kspec, one CTA per channel: K_l = Re sum_n w_n z_n^l (w = C Bbar, z = Delta A)
//      for l < L, with e^(l z) = e^(64 q z) e^(i z) (l = 64 q + i) from two small power
//      tables per state, so each (l, n) costs two FMAs.  A power's phase l Im z is taken
//      as a 64-bit fixed-point fraction of a turn, l times frac(Im z / 2 pi) modulo 2^64
//      (exact integer wrap-around; Delta and that fraction are formed in double), then
//      evaluated in float.  Then Khat = FFT(K zero-padded) / N into the workspace,
//      [dim, N] complex; CTA 0 also stores the twiddle tables there.
//   2. s4d_conv, per channel and pair of batch rows (b, b + 1): one complex sequence
//      u_b + i u_{b+1} (zero-padded) is transformed, multiplied by Khat and transformed
//      back.  K is real, so Khat is Hermitian and IFFT(Khat FFT(u_b + i u_{b+1})) =
//      y_b + i y_{b+1}: two rows per transform pair.  The inverse is conj(FFT(conj(.))),
//      so one forward routine serves both.  The first pass reads u from global memory,
//      the last forward pass multiplies by Khat as it stores, and the last inverse pass
//      adds D u and writes y: the sequence goes through shared memory only between passes.
// The transforms run in shared memory, one CTA of N / 16 threads per sequence: a Stockham
// (autosort) FFT, natural order in and out, in passes of radix 16 (and one of radix 2, 4
// or 8 for the remaining bits).  In a pass each thread loads its butterfly's points into
// registers, the block syncs, each thread twiddles, transforms and stores them, and the
// block syncs again, so one buffer serves in place (one pad slot per 16 elements keeps
// the strided stores off a single bank).  Pass p (after the first) twiddles point r of
// butterfly k by w^(r k), w = exp(-2 pi i / (Ns R)): w^k is read from that pass's own
// table (consecutive k, so no bank conflicts) and its powers are formed by repeated
// multiplication.  Input points past N / 2 are zero and output points past N / 2 are
// never read (L <= N / 2), so the first forward and last inverse passes skip them.
// N is at most 16384 (L <= 8192).
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kMaxLog2N = 14;
constexpr int kMaxThreads = (1 << kMaxLog2N) / 16;  // N / 16 threads: one radix-16 butterfly each
constexpr int kPowChunk = 64;  // l = 64 q + i in the kernel generator
constexpr int kGroup = 8;      // states per power-table round
constexpr int kMaxSteps = 8;   // steps l < L per thread: L <= N / 2 = 8 x threads
constexpr int kMaxStates = 64;

// threads of a block for an N = 2^m point transform
__host__ __device__ inline int fft_threads(int m) { return m >= 9 ? (1 << m) / 16 : 32; }
// passes of an N = 2^m transform: radix 16 while four bits remain, then radix 2, 4 or 8
__host__ __device__ inline int n_passes(int m) { return m / 4 + (m % 4 != 0); }
__host__ __device__ inline int pass_log2_radix(int m, int p) { return p < m / 4 ? 4 : m % 4; }
// pass p >= 1 has Ns = 16^p; its table of Ns twiddles starts at sum_{i=1}^{p-1} 16^i
__host__ __device__ inline int twiddle_offset(int p) { return ((1 << (4 * p)) - 16) / 15; }
__host__ __device__ inline int twiddle_len(int m) { return n_passes(m) > 1 ? twiddle_offset(n_passes(m)) : 0; }

// Shared-memory position of element i: one pad slot per 16 elements, so that the
// stride-16 stores of the first pass (and the stride-Ns ones after it) spread over the
// banks instead of all landing on one.
__device__ __forceinline__ int pad(int i) { return i + (i >> 4); }
__host__ __device__ inline int padded_len(int n) { return n + (n >> 4); }
// the spectrum kernel's sequence region also holds its power tables first
__host__ __device__ inline int power_chunks(int L) { return (L + kPowChunk - 1) / kPowChunk; }
__host__ __device__ inline int kspec_x_len(int m, int L) {
    const int t = kGroup * (power_chunks(L) + kPowChunk), x = padded_len(1 << m);
    return t > x ? t : x;
}

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}

// exp(-2 pi i k / 16), k < 8: cos and -sin of k pi / 8
__device__ __forceinline__ float2 root16(int k) {
    constexpr float c1 = 0.92387953251128674f, s1 = 0.38268343236508978f, h = 0.70710678118654752f;
    switch (k) {
        case 0: return make_float2(1.f, 0.f);
        case 1: return make_float2(c1, -s1);
        case 2: return make_float2(h, -h);
        case 3: return make_float2(s1, -c1);
        case 4: return make_float2(0.f, -1.f);
        case 5: return make_float2(-s1, -c1);
        case 6: return make_float2(-h, -h);
        default: return make_float2(-c1, -s1);
    }
}

// R-point DFT of v in registers (R = 2, 4, 8 or 16), natural order in and out:
// decimation in frequency, then the bit-reversal permutation (all indices compile-time)
template <int R>
__device__ __forceinline__ void dft_reg(float2* v) {
#pragma unroll
    for (int h = R / 2; h >= 1; h >>= 1) {
#pragma unroll
        for (int g = 0; g < R; g += 2 * h) {
#pragma unroll
            for (int j = 0; j < h; ++j) {
                const float2 a = v[g + j], b = v[g + j + h];
                v[g + j] = cadd(a, b);
                const float2 dd = csub(a, b);
                const int k = j * (8 / h);  // exp(-2 pi i j / (2h)) = root16(j 16 / (2h))
                if (k == 0) {
                    v[g + j + h] = dd;
                } else if (k == 4) {
                    v[g + j + h] = make_float2(dd.y, -dd.x);
                } else {
                    v[g + j + h] = cmul(dd, root16(k));
                }
            }
        }
    }
    constexpr int B = R == 2 ? 1 : R == 4 ? 2 : R == 8 ? 3 : 4;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        int rv = 0;
#pragma unroll
        for (int bb = 0; bb < B; ++bb) rv |= ((i >> bb) & 1) << (B - 1 - bb);
        if (i < rv) {
            const float2 t = v[i];
            v[i] = v[rv];
            v[rv] = t;
        }
    }
}

// The twiddle tables of every pass after the first: pass p's entry k is
// exp(-2 pi i k / (Ns R)), k < Ns = 16^p (the argument -2k / (Ns R) is exact in float).
__device__ void make_twiddles(float2* W, int m) {
    for (int p = 1; p < n_passes(m); ++p) {
        const int ns_log2 = 4 * p, Ns = 1 << ns_log2;
        const float inv = 1.0f / static_cast<float>(Ns << pass_log2_radix(m, p));
        float2* T = W + twiddle_offset(p);
        for (int k = threadIdx.x; k < Ns; k += blockDim.x) {
            float s, c;
            sincospif(-2.0f * static_cast<float>(k) * inv, &s, &c);
            T[k] = make_float2(c, s);
        }
    }
}

// point loaders and storers of a pass.  Those of the shared sequence X also take a
// padded address directly (put / the X member), so that a pass can address its points
// as one padded base plus constant strides.
struct LoadX {
    const float2* X;
    __device__ __forceinline__ float2 operator()(int t) const { return X[pad(t)]; }
};
struct StoreX {
    float2* X;
    __device__ __forceinline__ void operator()(int t, float2 v) const { X[pad(t)] = v; }
    __device__ __forceinline__ void put(float2* p, int, float2 v) const { *p = v; }
};
// Y = X Khat (Khat holds 1/N), stored conjugated for the inverse
struct StoreTimesKhat {
    float2* X;
    const float2* kh;
    __device__ __forceinline__ void operator()(int t, float2 v) const { put(X + pad(t), t, v); }
    __device__ __forceinline__ void put(float2* p, int t, float2 v) const {
        const float2 y = cmul(v, __ldg(kh + t));
        *p = make_float2(y.x, -y.y);
    }
};
template <class F> struct padded_load : std::false_type {};
template <> struct padded_load<LoadX> : std::true_type {};
template <class F> struct padded_store : std::false_type {};
template <> struct padded_store<StoreX> : std::true_type {};
template <> struct padded_store<StoreTimesKhat> : std::true_type {};

// One Stockham pass of radix 2^LR over N = 2^m points, Ns = 2^ns_log2 (the product of
// the radices before it), at most BPT butterflies per thread.  load(t) gives point t of
// the pass input, store(t, v) takes point t of its output; with SYNC the block syncs
// between the loads and the stores (both in the same shared buffer).  HALF_IN: input
// points t >= N / 2 are zero and not loaded; HALF_OUT: output points t >= N / 2 are not
// formed (only for a last pass, where they are r >= R / 2).  tw: this pass's table.
template <int LR, int BPT, bool HALF_IN, bool HALF_OUT, bool SYNC, class Load, class Store>
__device__ __forceinline__ void fft_pass(const float2* tw, int m, int ns_log2, Load load, Store store) {
    constexpr int R = 1 << LR;
    const int nb = 1 << (m - LR), Ns = 1 << ns_log2;
    float2 v[BPT][R];
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        const int j = threadIdx.x + q * blockDim.x;
        if (j < nb) {
            bool done = false;
            if constexpr (padded_load<Load>::value) {
                if (nb % 16 == 0) {  // pad(j + r nb) = pad(j) + r (nb + nb / 16)
                    const float2* xb = load.X + pad(j);
                    const int pnb = nb + (nb >> 4);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        v[q][r] = HALF_IN && r >= R / 2 ? make_float2(0.f, 0.f) : xb[r * pnb];
                    done = true;
                }
            }
            if (!done) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    v[q][r] = HALF_IN && r >= R / 2 ? make_float2(0.f, 0.f) : load(j + r * nb);
            }
        }
    }
    if (SYNC) __syncthreads();
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        const int j = threadIdx.x + q * blockDim.x;
        if (j < nb) {
            const int k = j & (Ns - 1);
            if (ns_log2 > 0) {
                const float2 w = tw[k];
                float2 wr = w;
#pragma unroll
                for (int r = 1; r < R; ++r) {
                    v[q][r] = cmul(v[q][r], wr);
                    if (r + 1 < R) wr = cmul(wr, w);
                }
            }
            dft_reg<R>(v[q]);
            const int base = ((j - k) << LR) + k;  // (j / Ns) Ns R + k
            bool done = false;
            if constexpr (padded_store<Store>::value) {
                if (Ns % 16 == 0 || (Ns == 1 && R == 16)) {
                    // pad(base + r Ns) = pad(base) + r (Ns + Ns / 16) when 16 divides Ns, and
                    // pad(base) + r when Ns = 1 (base = 16 j)
                    float2* xb = store.X + pad(base);
                    const int pns = Ns == 1 ? 1 : Ns + (Ns >> 4);
#pragma unroll
                    for (int r = 0; r < (HALF_OUT ? R / 2 : R); ++r) store.put(xb + r * pns, base + r * Ns, v[q][r]);
                    done = true;
                }
            }
            if (!done) {
#pragma unroll
                for (int r = 0; r < (HALF_OUT ? R / 2 : R); ++r) store(base + r * Ns, v[q][r]);
            }
        }
    }
}

// pass p of an N = 2^m transform with its radix chosen at run time
template <bool HALF_IN, bool HALF_OUT, bool SYNC, class Load, class Store>
__device__ __forceinline__ void fft_pass_any(const float2* W, int m, int p, Load load, Store store) {
    const float2* tw = W + (p > 0 ? twiddle_offset(p) : 0);
    const int ns_log2 = 4 * p;
    switch (pass_log2_radix(m, p)) {
        case 4: fft_pass<4, 1, HALF_IN, HALF_OUT, SYNC>(tw, m, ns_log2, load, store); break;
        case 3: fft_pass<3, 2, HALF_IN, HALF_OUT, SYNC>(tw, m, ns_log2, load, store); break;
        case 2: fft_pass<2, 4, HALF_IN, HALF_OUT, SYNC>(tw, m, ns_log2, load, store); break;
        default: fft_pass<1, 8, HALF_IN, HALF_OUT, SYNC>(tw, m, ns_log2, load, store); break;
    }
}


// Forward FFT of N = 2^m points whose second half is zero: the first pass takes its
// input from first(t) (t < N / 2; FIRST_SYNC if that reads X) and stores into X; the
// middle passes run in X; the last pass hands its natural-order output to last(t, v).
// The block syncs after every pass but the last (last may write X: the caller syncs).
template <bool FIRST_SYNC, class First, class Last>
__device__ __forceinline__ void fft_forward(float2* X, const float2* W, int m, First first, Last last) {
    const LoadX ld{X};
    const StoreX st{X};
    const int P = n_passes(m);
    if (P == 1) {
        fft_pass_any<true, false, FIRST_SYNC>(W, m, 0, first, last);
        return;
    }
    // every pass but the last has radix 16
    fft_pass<4, 1, true, false, FIRST_SYNC>(W, m, 0, first, st);
    __syncthreads();
#pragma unroll
    for (int p = 1; p + 1 < P; ++p) {
        fft_pass<4, 1, false, false, true>(W + twiddle_offset(p), m, 4 * p, ld, st);
        __syncthreads();
    }
    fft_pass_any<false, false, true>(W, m, P - 1, ld, last);
}

// FFT of the N = 2^m points in X of which only outputs t < N / 2 are wanted, handed to
// last(t, v); X is overwritten.
template <class Last>
__device__ __forceinline__ void fft_half_out(float2* X, const float2* W, int m, Last last) {
    const LoadX ld{X};
    const StoreX st{X};
    const int P = n_passes(m);
#pragma unroll
    for (int p = 0; p + 1 < P; ++p) {
        fft_pass<4, 1, false, false, true>(W + (p > 0 ? twiddle_offset(p) : 0), m, 4 * p, ld, st);
        __syncthreads();
    }
    fft_pass_any<false, true, false>(W, m, P - 1, ld, last);
}

// One state's w = C Bbar / N (float), Re z = Delta Re A (float) and frac(Im z / 2 pi) as a
// 64-bit fixed-point fraction of a turn, z = Delta A.  Delta and Im z are formed in double:
// the phase l Im z reaches 1e5 rad at long L, so its turn fraction must hold that many
// more bits than a float does.  Bbar = (e^z - 1) / z Delta B (zero-order hold).
struct StateWZ {
    float2 w;
    float zr;
    unsigned long long turn;
};
struct StoreKhat {
    float2* kh;
    __device__ __forceinline__ void operator()(int t, float2 v) const { kh[t] = v; }
};

__device__ StateWZ s4d_wz(const ssm_s4d_params& a, int d, int n, double dt, float inv_n) {
    const size_t k = (static_cast<size_t>(d) * a.dstate + n) * 2;
    const double zi = dt * static_cast<double>(a.A[k + 1]);
    const double x = zi * 0.15915494309189535;  // turns
    const double f = x - floor(x);                // [0, 1)
    StateWZ s;
    // f 2^64 as an integer: f 2^32 splits into high word and remainder (both exact)
    const double hi = floor(f * 4294967296.0);
    const double lo = (f * 4294967296.0 - hi) * 4294967296.0;
    s.turn = (static_cast<unsigned long long>(hi) << 32) + static_cast<unsigned long long>(lo);
    const float dtf = static_cast<float>(dt);
    const float pr0 = dtf * a.A[k], pi0 = static_cast<float>(zi);
    s.zr = pr0;
    float sn, cs;
    sincosf(pi0, &sn, &cs);
    float pr, pi;  // phi1(z) = (e^z - 1) / z, Taylor 1 + z/2 + z^2/6 near 0
    const float den = pr0 * pr0 + pi0 * pi0;
    if (den < 1e-6f) {
        pr = 1.0f + pr0 / 2.0f + (pr0 * pr0 - pi0 * pi0) / 6.0f;
        pi = pi0 / 2.0f + (2.0f * pr0 * pi0) / 6.0f;
    } else {
        const float s2 = sinf(pi0 / 2.0f);
        const float nr = expm1f(pr0) * cs - 2.0f * s2 * s2;  // Re e^z - 1
        const float ni = expf(pr0) * sn;
        pr = (nr * pr0 + ni * pi0) / den;
        pi = (ni * pr0 - nr * pi0) / den;
    }
    const float br = a.B[k], bi = a.B[k + 1];
    const float bbr = dtf * (br * pr - bi * pi), bbi = dtf * (br * pi + bi * pr);
    const float cr = a.C[k], ci = a.C[k + 1];
    s.w = make_float2((cr * bbr - ci * bbi) * inv_n, (cr * bbi + ci * bbr) * inv_n);
    return s;
}

// e^(l z) for an integer l >= 0 in float: the phase from the turn fraction l frac(Im z /
// 2 pi) modulo 1 (exact in 64 bits, then its top 32 bits as a signed turn in [-1/2, 1/2)),
// the magnitude e^(l Re z)
__device__ __forceinline__ float2 pow_z(const StateWZ& s, unsigned int l) {
    const unsigned long long ph = s.turn * static_cast<unsigned long long>(l);
    const int top = static_cast<int>(static_cast<unsigned int>(ph >> 32));
    float sn, cs;
    sincospif(static_cast<float>(top) * 4.656612873077393e-10f, &sn, &cs);  // top / 2^31
    const float mag = expf(static_cast<float>(l) * s.zr);
    return make_float2(mag * cs, mag * sn);
}

// Khat[d] = FFT(K[d] zero-padded to N) / N, K computed here (see the file comment): each
// state's w and z once, then the power tables of kGroup states at a time (in the space of
// X, which is filled only afterwards); each thread keeps the sums of its steps
// l = tid + threads k in registers.  CTA 0 also stores the twiddle tables for s4d_conv.
template <int MT>
__global__ void __launch_bounds__(kMaxThreads) s4d_kspec(ssm_s4d_params a, float2* Khat, float2* Wg, int m_arg) {
    const int m = MT ? MT : m_arg;  // MT: the transform size known when compiled
    extern __shared__ float2 sm[];
    __shared__ StateWZ s_wz[kMaxStates];
    const int N = 1 << m, L = a.seqlen, Ns = a.dstate, nt = blockDim.x;
    float2* X = sm;
    float2* W = sm + kspec_x_len(m, L);
    float2* T = X;  // [kGroup][nq + kPowChunk]: w z^(64 q) / N, then z^i
    const int d = blockIdx.x;
    const int nq = power_chunks(L);
    const int row = nq + kPowChunk;
    make_twiddles(W, m);
    {
        const double dt = exp(static_cast<double>(a.log_dt[d]));
        const float inv_n = 1.0f / static_cast<float>(N);  // a power of two: exact
        for (int n = threadIdx.x; n < Ns; n += nt) s_wz[n] = s4d_wz(a, d, n, dt, inv_n);
    }
    __syncthreads();
    float acc[kMaxSteps];
#pragma unroll
    for (int k = 0; k < kMaxSteps; ++k) acc[k] = 0.f;
    for (int n0 = 0; n0 < Ns; n0 += kGroup) {
        const int ng = min(kGroup, Ns - n0);
        for (int e = threadIdx.x; e < ng * row; e += nt) {
            const int g = e / row, r = e % row;
            const StateWZ& s = s_wz[n0 + g];
            if (r < nq) {
                T[e] = cmul(s.w, pow_z(s, static_cast<unsigned int>(r * kPowChunk)));
            } else {
                T[e] = pow_z(s, static_cast<unsigned int>(r - nq));
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kMaxSteps; ++k) {
            const int l = threadIdx.x + k * nt;
            if (l < L) {
                const int q = l / kPowChunk, i = l % kPowChunk;
                for (int g = 0; g < ng; ++g) {
                    const float2 p = T[g * row + q], z = T[g * row + nq + i];
                    acc[k] = fmaf(p.x, z.x, fmaf(-p.y, z.y, acc[k]));
                }
            }
        }
        __syncthreads();
    }
    // K into X (the first pass reads only t < N / 2, the rest is zero by HALF_IN)
#pragma unroll
    for (int k = 0; k < kMaxSteps; ++k) {
        const int l = threadIdx.x + k * nt;
        if (l < N / 2) X[pad(l)] = make_float2(l < L ? acc[k] : 0.f, 0.f);
    }
    if (d == 0) {
        for (int k = threadIdx.x; k < twiddle_len(m); k += nt) Wg[k] = W[k];
    }
    __syncthreads();
    fft_forward<true>(X, W, m, LoadX{X}, StoreKhat{Khat + static_cast<size_t>(d) * N});
}

// u_b + i u_{b+1}, zero past L
template <typename Tin>
struct LoadRows {
    const Tin* u0;
    const Tin* u1;
    int L;
    bool has_b1;
    __device__ __forceinline__ float2 operator()(int t) const {
        float re = 0.f, im = 0.f;
        if (t < L) {
            re = to_f32(u0[t]);
            if (has_b1) im = to_f32(u1[t]);
        }
        return make_float2(re, im);
    }
};
// the conjugate of the inverse is y_b0 + i y_b1 with D u added; t < L only
template <typename Tin, typename Tout>
struct StoreRows {
    const Tin* u0;
    const Tin* u1;
    Tout* y0;
    Tout* y1;
    float Dd;
    int L;
    bool has_b1;
    __device__ __forceinline__ void operator()(int t, float2 v) const {
        if (t < L) {
            io<Tout>::store(y0, t, v.x + Dd * to_f32(u0[t]));
            if (has_b1) io<Tout>::store(y1, t, -v.y + Dd * to_f32(u1[t]));
        }
    }
};

template <typename Tin, typename Tout, int MT>
__global__ void __launch_bounds__(kMaxThreads) s4d_conv(ssm_s4d_params a, const float2* Khat, const float2* Wg,
                                                       int m_arg) {
    const int m = MT ? MT : m_arg;  // MT: the transform size known when compiled
    extern __shared__ float2 sm[];
    const int N = 1 << m;
    float2* X = sm;
    float2* W = sm + padded_len(N);
    const int d = blockIdx.y;
    const int b0 = 2 * blockIdx.x;
    const bool has_b1 = b0 + 1 < a.batch;
    const int L = a.seqlen;
    const Tin* u0 = static_cast<const Tin*>(a.u) + (static_cast<size_t>(b0) * a.dim + d) * L;
    const Tin* u1 = u0 + static_cast<size_t>(a.dim) * L;  // row b0 + 1 (read only if has_b1)
    for (int k = threadIdx.x; k < twiddle_len(m); k += blockDim.x) W[k] = Wg[k];
    // the first pass stores no twiddles' reader: the sync after it publishes W too
    fft_forward<false>(X, W, m, LoadRows<Tin>{u0, u1, L, has_b1},
                       StoreTimesKhat{X, Khat + static_cast<size_t>(d) * N});
    __syncthreads();
    Tout* y0 = static_cast<Tout*>(a.y) + (static_cast<size_t>(b0) * a.dim + d) * L;
    fft_half_out(X, W, m, StoreRows<Tin, Tout>{u0, u1, y0, y0 + static_cast<size_t>(a.dim) * L,
                                               a.D_skip ? a.D_skip[d] : 0.f, L, has_b1});
}

int log2_fft(int L) {
    int m = 1;
    while ((1 << m) < 2 * L) ++m;
    return m;
}

size_t smem_bytes(int m) {
    return static_cast<size_t>(padded_len(1 << m) + twiddle_len(m)) * sizeof(float2);
}
size_t kspec_smem_bytes(int m, int L) {
    return static_cast<size_t>(kspec_x_len(m, L) + twiddle_len(m)) * sizeof(float2);
}

// the kernels of an N = 2^m transform: compiled for each m of 9 .. 14 (N / 16 threads,
// every stride a constant), one runtime-m kernel for the short ones
template <int MT, typename F>
cudaError_t with_m(int m, F&& f) {
    if constexpr (MT > kMaxLog2N) {
        return f(std::integral_constant<int, 0>{});
    } else {
        if (m == MT) return f(std::integral_constant<int, MT>{});
        return with_m<MT + 1>(m, f);
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_conv(const ssm_s4d_params& a, const float2* Khat, const float2* Wg, int m, cudaStream_t s) {
    return with_m<9>(m, [&](auto mt) -> cudaError_t {
        auto k = s4d_conv<Tin, Tout, decltype(mt)::value>;
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(k), static_cast<int>(smem_bytes(m)));
        if (e != cudaSuccess) return e;
        const dim3 grid((a.batch + 1) / 2, a.dim);
        k<<<grid, fft_threads(m), smem_bytes(m), s>>>(a, Khat, Wg, m);
        return cudaGetLastError();
    });
}

}  // namespace

bool s4d_conv_supported(const ssm_s4d_params& a) {
    return s4d_supported(a.dstate) && a.dstate <= kMaxStates && a.seqlen >= 1 && log2_fft(a.seqlen) <= kMaxLog2N;
}

// [dim, N] complex Khat, then the twiddle tables
size_t s4d_conv_workspace_size(const ssm_s4d_params& a) {
    if (!s4d_conv_supported(a)) return 0;
    const int m = log2_fft(a.seqlen);
    return (static_cast<size_t>(a.dim) * (static_cast<size_t>(1) << m) + twiddle_len(m)) * sizeof(float2);
}

cudaError_t s4d_conv_launch(const ssm_s4d_params& a, void* workspace, cudaStream_t s) {
    const int m = log2_fft(a.seqlen);
    float2* Khat = static_cast<float2*>(workspace);
    float2* Wg = Khat + static_cast<size_t>(a.dim) * (static_cast<size_t>(1) << m);
    const size_t ks = kspec_smem_bytes(m, a.seqlen);
    cudaError_t e = with_m<9>(m, [&](auto mt) -> cudaError_t {
        auto k = s4d_kspec<decltype(mt)::value>;
        cudaError_t r = set_smem_attr(reinterpret_cast<const void*>(k), static_cast<int>(ks));
        if (r != cudaSuccess) return r;
        k<<<a.dim, fft_threads(m), ks, s>>>(a, Khat, Wg, m);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
    const bool ib = a.in_dtype == SSM_BF16, ob = a.out_dtype == SSM_BF16;
    if (ib && ob) return launch_conv<bf16_t, bf16_t>(a, Khat, Wg, m, s);
    if (ib) return launch_conv<bf16_t, float>(a, Khat, Wg, m, s);
    if (ob) return launch_conv<float, bf16_t>(a, Khat, Wg, m, s);
    return launch_conv<float, float>(a, Khat, Wg, m, s);
}

}  // namespace ssm
