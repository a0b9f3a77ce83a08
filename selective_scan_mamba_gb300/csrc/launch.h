// launch.h -- internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "ssmscan.h"

namespace ssm {

constexpr int kM1MaxThreads = 384;  // block-size cap of the tiled Mamba-1 kernel
constexpr int kM1MaxPairs = 2;      // (batch, group) B/C rows one CTA may span

// Mamba-1 scan arguments (device pointers, dims) as the kernels see them.
struct M1Args {
    int batch, dim, dstate, seqlen, ngroups;
    ssm_dtype in_dtype, out_dtype;
    const void* x;
    const void* delta;
    const float* delta_bias;
    int delta_softplus;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* h0;
    void* y;
    float* h_final;
    ssm_disc disc;
    int cpb_max;  // channels per CTA (tiled path)
    // choices of ssm_scan_opts (0 = automatic)
    int kernel;               // ssm_scan_kernel
    int tpc;                  // threads per channel
    int max_segments;         // time segments
    unsigned int wait_limit;  // polls before a device-side wait gives up (0 = default)
    int fault_test;           // testing: skip one tile's input copy (see ssmscan.h)
};

// backward of the Mamba-1 scan (scan_m1_bwd.cu)
using M1BwdArgs = ssm_scan_bwd_params;
bool m1_bwd_supported(const M1BwdArgs& a);
size_t m1_bwd_workspace_size(const M1BwdArgs& a);
cudaError_t m1_bwd_launch(const M1BwdArgs& a, void* workspace, cudaStream_t s);
bool ssd_bwd_supported(const ssd_bwd_params& a);
size_t ssd_bwd_workspace_size(const ssd_bwd_params& a);
cudaError_t ssd_bwd_launch(const ssd_bwd_params& a, void* workspace, cudaStream_t s);
// the same derivative in chunked form (ssd_bwd.cu), for the shapes it covers
bool ssd_chunked_bwd_supported(const ssd_bwd_params& a);
size_t ssd_chunked_bwd_workspace_size(const ssd_bwd_params& a);
cudaError_t ssd_chunked_bwd_launch(const ssd_bwd_params& a, void* workspace, cudaStream_t s);

// Mamba-3 complex scan (scan_m3.cu)
bool m3_supported(int dstate);
size_t m3_workspace_size(const ssm_mamba3_params& a);
cudaError_t m3_launch(const ssm_mamba3_params& a, void* workspace, cudaStream_t s);

// S4D (s4d.cu)
bool s4d_supported(int dstate);
size_t s4d_workspace_size(const ssm_s4d_params& a);
cudaError_t s4d_launch(const ssm_s4d_params& a, void* workspace, cudaStream_t s);
cudaError_t s4d_kernel_launch(const ssm_s4d_params& a, float* K, int L, cudaStream_t s);
// S4D convolution form by FFT (s4d_conv.cu)
bool s4d_conv_supported(const ssm_s4d_params& a);
size_t s4d_conv_workspace_size(const ssm_s4d_params& a);
cudaError_t s4d_conv_launch(const ssm_s4d_params& a, void* workspace, cudaStream_t s);

struct M1Plan {
    enum Kind { kGeneric = 0, kTiled = 1, kTma = 2, kTmem = 3 } kind;
    int tpc;      // threads per channel (tiled path)
    int grid;     // CTAs (tiled path)
    int cpb_max;  // channels per CTA (tiled path)
    size_t smem;  // dynamic shared memory per CTA (tiled path)
    int cps = 0;  // CTAs per (batch, group) (TMEM-broadcast path)
    int segs = 1;         // time segments (TMEM-broadcast path)
    int tps = 0;          // tiles per segment
    int cps_st = 0;       // CTAs per (batch, group) of the segment pass
    int cpb_st = 0;       // channels per CTA of the segment pass
    size_t smem_st = 0;   // dynamic shared memory per CTA of the segment pass
    size_t ws_state = 0;  // workspace offset of the segment sums of Delta
    size_t ws_bytes = 0;  // workspace bytes
};

size_t m1_tiled_smem_bytes(int cpb, int N, int T, size_t elem_size);
int m1_tile_steps(ssm_dtype in_dtype);
cudaError_t m1_plan(const M1Args& a, M1Plan* plan);
cudaError_t m1_launch(const M1Args& a, const M1Plan& plan, cudaStream_t s);

// bf16 fast path staged by TMA (scan_m1_tma.cu)
size_t m1_tma_smem_bytes(int cpb);
cudaError_t m1_tma_plan(const M1Args& a, M1Plan* plan);
cudaError_t m1_tma_launch(const M1Args& a, const M1Plan& plan, cudaStream_t s);
cudaError_t m1_tma_take_wait_timeouts(unsigned int* count);  // reads and clears

// bf16 fast path with B/C broadcast through tensor memory (scan_m1_tmem.cu)
cudaError_t m1_tmem_plan(const M1Args& a, M1Plan* plan);
cudaError_t m1_tmem_launch(const M1Args& a, const M1Plan& plan, void* workspace, cudaStream_t s);
cudaError_t m1_tmem_take_wait_timeouts(unsigned int* count);  // reads and clears

// TMA tensor map of a row-major [rows][inner] tensor (tmap.cu)
cudaError_t encode_tmap_2d(struct CUtensorMap_st* map, const void* base, int elem_bytes,
                           unsigned long long inner, unsigned long long rows, unsigned box_inner,
                           unsigned box_rows, bool swizzle128);
cudaError_t encode_tmap_nd(struct CUtensorMap_st* map, const void* base, int elem_bytes, int rank,
                           const unsigned long long* dims, const unsigned* box, bool swizzle128);
// raises the kernel's MaxDynamicSharedMemorySize on the current device to at least bytes
// (a driver call only when the limit set so far is smaller)
cudaError_t set_smem_attr(const void* kernel, int bytes);

// Launches `kernel` so that it may start before the kernel ahead of it in stream `s` has
// finished (programmatic stream serialisation); the kernel must call grid_dep_wait()
// before it touches memory the earlier kernel uses.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Decode-step arguments.
struct StepArgs {
    int batch, nheads, headdim, dstate, ngroups, a_per_state;
    ssm_dtype in_dtype, out_dtype;
    float* state;
    const void* x;
    const void* dt;
    const float* dt_bias;
    int dt_softplus;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    void* y;
    ssm_disc disc;
    int ntok = 1;  // consecutive tokens (token-major x, dt, B, C, z, y)
};
cudaError_t step_launch(const StepArgs& a, cudaStream_t s);

// SSD arguments.
struct SsdArgs {
    int batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
    ssm_dtype in_dtype, out_dtype;
    const void* x;
    const void* dt;
    const float* dt_bias;
    int dt_softplus;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* h0;
    void* y;
    float* h_final;
    ssm_disc disc;
    float* ws_states;  // [batch, nheads, nchunks, headdim, dstate] chunk states, then h_in
    float* ws_decay;   // [batch, nheads, nchunks] exp(sum of Delta*A over the chunk)
};
size_t ssd_workspace_bytes(const SsdArgs& a);
cudaError_t ssd_launch(const SsdArgs& a, cudaStream_t s);

// tensor-core SSD path (ssd_tc.cu)
bool ssd_tc_supported(const SsdArgs& a);
size_t ssd_tc_workspace_bytes(const SsdArgs& a);
cudaError_t ssd_tc_launch(const SsdArgs& a, void* workspace, cudaStream_t s);
cudaError_t ssd_tc_take_wait_timeouts(unsigned int* count);  // reads and clears

// Records `msg` as this thread's ssm_last_error() text and returns `st`.
ssm_status set_error(ssm_status st, const char* msg);

}  // namespace ssm
