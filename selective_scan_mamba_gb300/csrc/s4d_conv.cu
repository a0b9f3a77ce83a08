// s4d_conv.cu -- S4D convolution form on the GPU: y = K * u + D u by FFT (sm_103a).
//
// ("From S4 to Mamba-3", 03/System, s4_minimal.py: S4D trains as one FFT convolution with
// its kernel K_l = Re sum_n C Bbar Abar^l; 09/Validation: the convolution equals the
// recurrent form from a zero state.)  The causal convolution of a length-L row with the
// length-L kernel is the first L points of the cyclic convolution of both, zero-padded
// to N = 2^ceil(log2 2L): y = IFFT(FFT(K) . FFT(u)) restricted to t < L.
//
// Two launches:
//   1. s4d_kspec, one CTA per channel: K_l = Re sum_n w_n z_n^l (w = C Bbar, z = Abar)
//      for l < L, with z^l = z^(64 q) z^i (l = 64 q + i): each power's phase l Im z is
//      formed and reduced modulo 2 pi in double, then evaluated in float; w is folded
//      into the first power, so each (l, n) costs two FMAs.  Then
//      Khat = FFT(K zero-padded) / N into the workspace, [dim, N] complex.
//   2. s4d_conv, per channel and pair of batch rows (b, b + 1): one complex sequence
//      u_b + i u_{b+1} (zero-padded) is transformed, multiplied by Khat and transformed
//      back.  K is real, so Khat is Hermitian and IFFT(Khat FFT(u_b + i u_{b+1})) =
//      y_b + i y_{b+1}: two rows per transform pair.  The inverse is conj(FFT(conj(.))),
//      so one forward routine serves both.  Then D u is added.
// The transforms run in shared memory, one CTA of N / 16 threads per sequence: a Stockham
// (autosort) FFT, natural order in and out, in passes of radix 16 (and one of radix 2, 4
// or 8 for the remaining bits).  In a pass each thread loads its butterfly's 16 points
// into registers, the block syncs, each thread twiddles, transforms and stores them, and
// the block syncs again, so one buffer serves in place (one pad slot per 16 elements
// keeps the strided stores off a single bank).  Twiddles exp(-2 pi i k / N), k < N/2,
// are computed once per CTA with sincospif (the argument -2k/N is exact in float32); the
// radix-16 butterflies use the 16th roots of unity as constants.  N is at most 16384
// (L <= 8192): the sequence and the twiddles take 192 KB of shared memory (204 KB with
// the power tables of the spectrum kernel).
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {

namespace {

constexpr int kMaxLog2N = 14;
constexpr int kMaxThreads = (1 << kMaxLog2N) / 16;  // N / 16 threads: one radix-16 butterfly each
constexpr int kPowChunk = 64;  // l = 64 q + i in the kernel generator
constexpr int kGroup = 8;      // states per power-table round
constexpr int kMaxSteps = 8;   // steps l < L per thread: L <= N / 2 = 8 x threads
constexpr int kTableFloat2 = kGroup * ((1 << (kMaxLog2N - 1)) / kPowChunk + kPowChunk);

// threads of a block for an N = 2^m point transform
__host__ __device__ inline int fft_threads(int m) { return m >= 9 ? (1 << m) / 16 : 32; }

// Shared-memory position of element i: one pad slot per 16 elements, so that the
// stride-16 stores of the first pass (and the stride-Ns ones after it) spread over the
// banks instead of all landing on one.
__device__ __forceinline__ int pad(int i) { return i + (i >> 4); }
__host__ __device__ inline int padded_len(int n) { return n + (n >> 4); }

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

// W[k] = exp(-2 pi i k / N), k < N / 2
__device__ void make_twiddles(float2* W, int m) {
    const int N = 1 << m;
    for (int k = threadIdx.x; k < N / 2; k += blockDim.x) {
        float s, c;
        sincospif(-2.0f * static_cast<float>(k) / static_cast<float>(N), &s, &c);
        W[k] = make_float2(c, s);
    }
}
// exp(-2 pi i k / N) for k < N from the half table
__device__ __forceinline__ float2 twiddle(const float2* W, int k, int half) {
    if (k < half) return W[k];
    const float2 w = W[k - half];
    return make_float2(-w.x, -w.y);
}

// One Stockham pass of radix R over N = 2^m points in place, Ns = product of the
// radices of the passes before it (BPT = butterflies per thread, upper bound).
template <int R, int BPT>
__device__ __forceinline__ void stockham_pass(float2* X, const float2* W, int m, int ns_log2) {
    constexpr int LR = R == 2 ? 1 : R == 4 ? 2 : R == 8 ? 3 : 4;
    const int N = 1 << m, nb = N >> LR, Ns = 1 << ns_log2;
    const int tw_shift = m - ns_log2 - LR;  // N / (Ns R) = 2^tw_shift
    float2 v[BPT][R];
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        const int j = threadIdx.x + q * blockDim.x;
        if (j < nb) {
#pragma unroll
            for (int r = 0; r < R; ++r) v[q][r] = X[pad(j + r * nb)];
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        const int j = threadIdx.x + q * blockDim.x;
        if (j < nb) {
            const int k = j & (Ns - 1);
            if (Ns > 1) {
#pragma unroll
                for (int r = 1; r < R; ++r) v[q][r] = cmul(v[q][r], twiddle(W, (r * k) << tw_shift, N >> 1));
            }
            dft_reg<R>(v[q]);
            const int base = ((j - k) << LR) + k;  // (j / Ns) Ns R + k
#pragma unroll
            for (int r = 0; r < R; ++r) X[pad(base + r * Ns)] = v[q][r];
        }
    }
    __syncthreads();
}

// Forward FFT of N = 2^m (1 <= m <= 14) points in X (padded positions), natural order in
// and out, by a block of fft_threads(m) threads: passes of radix 16, then one of radix 2,
// 4 or 8 if m % 4 != 0.  With N / 16 threads a radix-R pass has 16 / R butterflies per
// thread.
__device__ void fft_stockham(float2* X, const float2* W, int m) {
    int done = 0;
    while (m - done >= 4) {
        stockham_pass<16, 1>(X, W, m, done);
        done += 4;
    }
    switch (m - done) {
        case 1: stockham_pass<2, 8>(X, W, m, done); break;
        case 2: stockham_pass<4, 4>(X, W, m, done); break;
        case 3: stockham_pass<8, 2>(X, W, m, done); break;
        default: break;
    }
}

// one state's w = C Bbar and z = e^(Delta A), the latter as magnitude log and phase (double)
__device__ void s4d_wz(const ssm_s4d_params& a, int d, int n, double* wr, double* wi, double* zr,
                       double* zi) {
    const double dt = exp(static_cast<double>(a.log_dt[d]));
    const size_t k = (static_cast<size_t>(d) * a.dstate + n) * 2;
    const double ar = a.A[k], ai = a.A[k + 1], br = a.B[k], bi = a.B[k + 1];
    const double pr0 = dt * ar, pi0 = dt * ai;  // z = Delta A
    const double ex = exp(pr0);
    double sn, cs;
    sincos(pi0, &sn, &cs);
    double pr, pi;  // phi1(z) = (e^z - 1) / z, Taylor 1 + z/2 + z^2/6 near 0
    if (sqrt(pr0 * pr0 + pi0 * pi0) < 1e-4) {
        pr = 1.0 + pr0 / 2.0 + (pr0 * pr0 - pi0 * pi0) / 6.0;
        pi = pi0 / 2.0 + (2.0 * pr0 * pi0) / 6.0;
    } else {
        const double s2 = sin(pi0 / 2.0);
        const double nr = expm1(pr0) * cs - 2.0 * s2 * s2;
        const double ni = ex * sn;
        const double den = pr0 * pr0 + pi0 * pi0;
        pr = (nr * pr0 + ni * pi0) / den;
        pi = (ni * pr0 - nr * pi0) / den;
    }
    const double bbr = dt * (br * pr - bi * pi), bbi = dt * (br * pi + bi * pr);
    const double cr = a.C[k], ci = a.C[k + 1];
    *wr = cr * bbr - ci * bbi;
    *wi = cr * bbi + ci * bbr;
    *zr = pr0;
    *zi = pi0;
}

// e^(l z) in float: the phase l Im z is formed and reduced modulo 2 pi in double (it
// reaches 1e5 rad at long L), then sine, cosine and the magnitude e^(l Re z) in float
__device__ __forceinline__ float2 pow_z(double zr, double zi, double l) {
    const double inv_two_pi = 0.15915494309189535, two_pi = 6.283185307179586;
    const double x = l * zi;
    const float ph = static_cast<float>(x - two_pi * floor(x * inv_two_pi));
    float sn, cs;
    sincosf(ph, &sn, &cs);
    const float mag = expf(static_cast<float>(l * zr));
    return make_float2(mag * cs, mag * sn);
}

// Khat[d] = FFT(K[d] zero-padded to N) / N, K computed here (see the file comment): each
// state's w and z once (double), then the power tables of kGroup states at a time in a
// small region T; each thread keeps the sums of its steps l = tid + threads k in registers.
__global__ void __launch_bounds__(kMaxThreads) s4d_kspec(ssm_s4d_params a, float2* Khat, int m) {
    extern __shared__ float2 sm[];
    __shared__ double s_w[64][4];  // per state: Re w, Im w, Re z, Im z
    const int N = 1 << m, L = a.seqlen, Ns = a.dstate, nt = blockDim.x;
    float2* X = sm;
    float2* W = sm + padded_len(N);
    float2* T = W + N / 2;  // [kGroup][nq + kPowChunk]: w z^(64 q) / N, then z^i
    const int d = blockIdx.x;
    const int nq = (L + kPowChunk - 1) / kPowChunk;
    const int row = nq + kPowChunk;
    const float inv_n = 1.0f / static_cast<float>(N);  // a power of two: exact
    for (int n = threadIdx.x; n < Ns; n += nt) s4d_wz(a, d, n, &s_w[n][0], &s_w[n][1], &s_w[n][2], &s_w[n][3]);
    __syncthreads();
    float acc[kMaxSteps];
#pragma unroll
    for (int k = 0; k < kMaxSteps; ++k) acc[k] = 0.f;
    for (int n0 = 0; n0 < Ns; n0 += kGroup) {
        const int ng = min(kGroup, Ns - n0);
        for (int e = threadIdx.x; e < ng * row; e += nt) {
            const int g = e / row, r = e % row;
            const double* wz = s_w[n0 + g];
            if (r < nq) {
                const float2 p = pow_z(wz[2], wz[3], static_cast<double>(r) * kPowChunk);
                const float wr = static_cast<float>(wz[0]) * inv_n, wi = static_cast<float>(wz[1]) * inv_n;
                T[e] = make_float2(wr * p.x - wi * p.y, wr * p.y + wi * p.x);
            } else {
                T[e] = pow_z(wz[2], wz[3], static_cast<double>(r - nq));
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
#pragma unroll
    for (int k = 0; k < 2 * kMaxSteps; ++k) {
        const int l = threadIdx.x + k * nt;
        if (l < N) X[pad(l)] = make_float2(k < kMaxSteps && l < L ? acc[k < kMaxSteps ? k : 0] : 0.f, 0.f);
    }
    make_twiddles(W, m);
    __syncthreads();
    fft_stockham(X, W, m);
    for (int k = threadIdx.x; k < N; k += nt) Khat[static_cast<size_t>(d) * N + k] = X[pad(k)];
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kMaxThreads) s4d_conv(ssm_s4d_params a, const float2* Khat, int m) {
    extern __shared__ float2 sm[];
    const int N = 1 << m;
    float2* X = sm;
    float2* W = sm + padded_len(N);
    const int d = blockIdx.y;
    const int b0 = 2 * blockIdx.x, b1 = b0 + 1;
    const bool has_b1 = b1 < a.batch;
    const int L = a.seqlen;
    const Tin* u = static_cast<const Tin*>(a.u);
    const size_t r0 = (static_cast<size_t>(b0) * a.dim + d) * L;
    const size_t r1 = (static_cast<size_t>(b1) * a.dim + d) * L;
    make_twiddles(W, m);
    for (int t = threadIdx.x; t < N; t += blockDim.x) {
        float re = 0.f, im = 0.f;
        if (t < L) {
            re = to_f32(u[r0 + t]);
            if (has_b1) im = to_f32(u[r1 + t]);
        }
        X[pad(t)] = make_float2(re, im);
    }
    __syncthreads();
    fft_stockham(X, W, m);
    // Y = X Khat (Khat holds 1/N); the inverse is conj(FFT(conj(Y)))
    const float2* kh = Khat + static_cast<size_t>(d) * N;
    for (int k = threadIdx.x; k < N; k += blockDim.x) {
        const float2 y = cmul(X[pad(k)], kh[k]);
        X[pad(k)] = make_float2(y.x, -y.y);
    }
    __syncthreads();
    fft_stockham(X, W, m);
    const float Dd = a.D_skip ? a.D_skip[d] : 0.f;
    Tout* y = static_cast<Tout*>(a.y);
    for (int t = threadIdx.x; t < L; t += blockDim.x) {
        const float2 v = X[pad(t)];  // conj of the inverse: y_b0 = v.x, y_b1 = -v.y
        io<Tout>::store(y, r0 + t, v.x + Dd * to_f32(u[r0 + t]));
        if (has_b1) io<Tout>::store(y, r1 + t, -v.y + Dd * to_f32(u[r1 + t]));
    }
}

int log2_fft(int L) {
    int m = 1;
    while ((1 << m) < 2 * L) ++m;
    return m;
}

size_t smem_bytes(int m) {
    return static_cast<size_t>(padded_len(1 << m) + (1 << (m - 1))) * sizeof(float2);
}
size_t kspec_smem_bytes(int m) { return smem_bytes(m) + kTableFloat2 * sizeof(float2); }

template <typename Tin, typename Tout>
cudaError_t launch_conv(const ssm_s4d_params& a, const float2* Khat, int m, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(s4d_conv<Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes(m)));
    if (e != cudaSuccess) return e;
    const dim3 grid((a.batch + 1) / 2, a.dim);
    s4d_conv<Tin, Tout><<<grid, fft_threads(m), smem_bytes(m), s>>>(a, Khat, m);
    return cudaGetLastError();
}

}  // namespace

bool s4d_conv_supported(const ssm_s4d_params& a) {
    return s4d_supported(a.dstate) && a.seqlen >= 1 && log2_fft(a.seqlen) <= kMaxLog2N;
}

size_t s4d_conv_workspace_size(const ssm_s4d_params& a) {
    if (!s4d_conv_supported(a)) return 0;
    return static_cast<size_t>(a.dim) * (static_cast<size_t>(1) << log2_fft(a.seqlen)) * sizeof(float2);
}

cudaError_t s4d_conv_launch(const ssm_s4d_params& a, void* workspace, cudaStream_t s) {
    const int m = log2_fft(a.seqlen);
    float2* Khat = static_cast<float2*>(workspace);
    cudaError_t e = cudaFuncSetAttribute(s4d_kspec, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kspec_smem_bytes(m)));
    if (e != cudaSuccess) return e;
    s4d_kspec<<<a.dim, fft_threads(m), kspec_smem_bytes(m), s>>>(a, Khat, m);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const bool ib = a.in_dtype == SSM_BF16, ob = a.out_dtype == SSM_BF16;
    if (ib && ob) return launch_conv<bf16_t, bf16_t>(a, Khat, m, s);
    if (ib) return launch_conv<bf16_t, float>(a, Khat, m, s);
    if (ob) return launch_conv<float, bf16_t>(a, Khat, m, s);
    return launch_conv<float, float>(a, Khat, m, s);
}

}  // namespace ssm
