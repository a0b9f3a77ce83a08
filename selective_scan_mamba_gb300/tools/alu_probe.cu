// alu_probe.cu -- per-SM throughput of the two arithmetic units a selective-scan update
// needs: MUFU.EX2 (ex2.approx.ftz.f32) and the FP32 FMA pipe (FFMA, and the f32x2 form),
// plus their mix at the update's ratio (one exponential, four FP32 operations).
//
// Each thread runs 8 independent dependency chains for kIter iterations (all values stay
// finite) and writes one float.  The grid is one wave: SMs x the resident CTAs of 512
// threads per SM the occupancy API reports.  Rates per second are from CUDA events around
// the last of three launches; rates per SM clock divide each SM's work by the longest
// clock64 span of a CTA (all of an SM's CTAs run concurrently).
#include <cstdio>
#include <cuda_runtime.h>

namespace {
constexpr int kIter = 4096;
constexpr int kThreads = 512;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads) probe(float* out, long long* cycles) {
    float v[8];
    float2 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = -0.01f * static_cast<float>(threadIdx.x % 7 + i);
        w[i] = make_float2(0.01f * i, 0.02f);
    }
    const float2 a = make_float2(0.999f, 0.998f), b = make_float2(0.001f, 0.002f);
    const long long t0 = clock64();
    for (int it = 0; it < kIter; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (KIND == 0) v[i] = ex2(-v[i]);
            if (KIND == 1) v[i] = fmaf(a.x, v[i], b.x);
            if (KIND == 2) w[i] = __ffma2_rn(a, w[i], b);
            if (KIND == 3) {
                v[i] = ex2(-v[i]);
                w[i] = __ffma2_rn(a, w[i], b);
                w[i] = __ffma2_rn(w[i], a, b);
            }
        }
    }
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i] + w[i].x + w[i].y;
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}
}  // namespace

int main() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, probe<3>, kThreads, 0);
    for (auto k : {probe<0>, probe<1>, probe<2>}) {
        int p = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p, k, kThreads, 0);
        per_sm = p < per_sm ? p : per_sm;
    }
    if (per_sm < 1) per_sm = 1;
    const int blocks = sms * per_sm;
    float* out = nullptr;
    long long* cyc = nullptr;
    if (cudaMalloc(&out, sizeof(float) * blocks * kThreads) != cudaSuccess ||
        cudaMalloc(&cyc, sizeof(long long) * blocks) != cudaSuccess) {
        fprintf(stderr, "allocation failed\n");
        return 1;
    }
    long long* hc = new long long[blocks];
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    struct Case { const char* name; void (*k)(float*, long long*); double ops_per_chain_step; };
    const Case cases[4] = {
        {"ex2 (MUFU.EX2, per op)", probe<0>, 1.0},
        {"ffma (FP32 FMA, per op)", probe<1>, 1.0},
        {"ffma2 (f32x2 FMA, per FP32 op)", probe<2>, 2.0},
        {"mix 1 ex2 + 4 FP32 ops (per ex2)", probe<3>, 1.0},
    };
    printf("{\"sms\": %d, \"ctas_per_sm\": %d, \"cases\": [", sms, per_sm);
    for (int c = 0; c < 4; ++c) {
        float ms = 0.f;
        for (int rep = 0; rep < 3; ++rep) {
            cudaEventRecord(e0);
            cases[c].k<<<blocks, kThreads>>>(out, cyc);
            cudaEventRecord(e1);
            cudaEventSynchronize(e1);
        }
        cudaEventElapsedTime(&ms, e0, e1);
        cudaMemcpy(hc, cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost);
        double span = 0.0;
        for (int i = 0; i < blocks; ++i) span = hc[i] > span ? static_cast<double>(hc[i]) : span;
        const double ops = static_cast<double>(blocks) * kThreads * 8 * kIter * cases[c].ops_per_chain_step;
        const double per_sm_clk = ops / sms / span;
        printf("%s{\"case\": \"%s\", \"ms\": %.4f, \"ops_per_s\": %.4e, \"ops_per_clk_per_sm\": %.2f}",
               c ? ", " : "", cases[c].name, ms, ops / (ms * 1e-3), per_sm_clk);
    }
    const cudaError_t e = cudaDeviceSynchronize();
    printf("], \"status\": \"%s\"}\n", cudaGetErrorString(e));
    delete[] hc;
    return e != cudaSuccess;
}
