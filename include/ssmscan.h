/*
 * ssmscan.h -- C ABI of libssmscan, a single-GPU (GB300, sm_103a) library of the
 * selective state-space scan used by Mamba-1 and Mamba-2.
 *
 * The operation, as the pages describe it ("From S4 to Mamba-3", ssmbench case
 * study, section 03/System):
 *   - mamba_minimal.py: Mamba-1 makes Delta, B and C input-dependent (selective)
 *     and runs the scan as an explicit time loop; an incremental step() serves
 *     decoding and must equal the full forward pass (09/Validation).
 *   - mamba2_minimal.py: with a scalar A per head the recurrence becomes SSD,
 *     computed as chunked decayed-attention matmuls with a carried (N, P) state;
 *     it must equal the sequential scan for aligned and misaligned chunk sizes
 *     (04/Approach "Chunked SSD with a sequential reference").
 *   - s4_minimal.py and Likely questions Q01: exact ZOH for a diagonal A gives
 *     B-bar = Delta*B*(e^z - 1)/z, z = Delta*a (optional here, SSM_DISC_ZOH).
 *   - mamba3_minimal.py / 04/Approach: the exponential-Euler rule A-bar =
 *     exp(Delta*A), B-bar = Delta*B that Mamba-3 reduces to at lambda = 1,
 *     theta = 0 (the default here, SSM_DISC_EXP_EULER).
 *
 * In formulas, per channel (Mamba-1) or per head (Mamba-2), for t = 0..L-1:
 *   Delta_t = softplus(delta_t + bias)      (or delta_t + bias without softplus)
 *   h_t     = exp(Delta_t A) (.) h_{t-1} + w_t B_t x_t,
 *             w_t = Delta_t (exp-Euler) or Delta_t (e^z - 1)/z, z = Delta_t A (ZOH)
 *   y_t     = (C_t . h_t + D x_t) * SiLU(z_t)     (gate only when z is given)
 * with h_{-1} = h0 (zeros when h0 is NULL) and h_final = h_{L-1}.
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every buffer.  The library allocates nothing
 *     and keeps no state except a per-thread error message.
 *   - Pointers: every tensor pointer is a DEVICE pointer of the current CUDA
 *     device; tensors are dense, row-major (last index fastest), and 16-byte
 *     aligned.  Optional tensors (marked "nullable") may be NULL.
 *   - Streams: `stream` is a cudaStream_t of the current device passed as void*
 *     (NULL = the legacy default stream).  Every call is asynchronous on that
 *     stream; results are ready when the stream reaches that point.
 *   - Errors: arguments are validated before anything is launched.  Bad
 *     arguments return SSM_ERR_INVALID_ARG, shapes outside what the kernels
 *     support return SSM_ERR_UNSUPPORTED, and a failed launch returns
 *     SSM_ERR_CUDA; in each case ssm_last_error() describes the problem and
 *     nothing has been written.  There is no CPU fallback.
 *   - Device-side waits: kernels that wait for their own asynchronous copies and
 *     tensor-core operations bound every wait.  A wait that runs out makes its
 *     block stop issuing work and finish; the call's outputs are then not valid.
 *     Calls are asynchronous, so this is reported afterwards: ssm_device_status()
 *     returns SSM_ERR_TIMEOUT until the event has been read.
 *   - Aliasing: outputs (and the workspace) must not overlap inputs or each
 *     other, except the decode state, which is updated in place by design.
 *     Overlaps are checked from the shapes and refused with SSM_ERR_INVALID_ARG.
 *   - Precision: inputs are bfloat16 or float32; A, D, biases and all states are
 *     float32; every accumulation is float32.
 */
#ifndef SSMSCAN_H
#define SSMSCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_ABI_VERSION 2

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,  /* null required pointer, bad size, misaligned pointer */
    SSM_ERR_UNSUPPORTED = 2,  /* valid, but outside the shapes the kernels implement */
    SSM_ERR_CUDA = 3,         /* a CUDA call or launch failed */
    SSM_ERR_TIMEOUT = 4       /* a bounded device-side wait gave up (ssm_device_status) */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

typedef enum {
    SSM_DISC_EXP_EULER = 0,   /* A-bar = exp(Delta A), B-bar = Delta B                 */
    SSM_DISC_ZOH = 1          /* A-bar = exp(Delta A), B-bar = Delta B (e^z - 1)/z     */
} ssm_disc;

/* ---------------------------------------------------------------------------
 * Mamba-1 selective scan (diagonal A per channel)
 *   ("From S4 to Mamba-3", 03/System, mamba_minimal.py)
 *
 * Shapes, Bt = batch, D = dim (d_inner), N = dstate, L = seqlen, G = ngroups:
 *   x, delta, z : [Bt, D, L]   in_dtype        (z nullable: no gate)
 *   y           : [Bt, D, L]   out_dtype
 *   B, C        : [Bt, G, N, L] in_dtype       (channel d uses group d / (D / G))
 *   A           : [D, N]       float32
 *   D_skip      : [D]          float32         (nullable: no skip term)
 *   delta_bias  : [D]          float32         (nullable: zero)
 *   h0, h_final : [Bt, D, N]   float32         (nullable: zero start / not written)
 * Limits: 1 <= N <= 256, G divides D, L >= 0 (L = 0 only copies h0 to h_final).
 * ------------------------------------------------------------------------- */
typedef struct {
    int batch, dim, dstate, seqlen, ngroups;
    ssm_dtype in_dtype, out_dtype;
    const void* x;
    const void* delta;
    const float* delta_bias;
    int delta_softplus;        /* nonzero: Delta = softplus(delta + bias) */
    const float* A;
    const void* B;
    const void* C;
    const float* D_skip;
    const void* z;
    const float* h0;
    void* y;
    float* h_final;
    ssm_disc disc;
} ssm_scan_params;

/* Runs the scan.  Needs no scratch memory: every problem runs in one pass over
 * the sequence (see ssm_scan_fwd_ex for the time-split plan of long sequences
 * with few channels, which carries segment states through a workspace). */
ssm_status ssm_scan_fwd(const ssm_scan_params* p, void* stream);

/* Kernel choice for ssm_scan_fwd_ex.  AUTO takes the fastest kernel that supports
 * the problem; naming one that does not returns SSM_ERR_UNSUPPORTED. */
typedef enum {
    SSM_SCAN_KERNEL_AUTO = 0,
    SSM_SCAN_KERNEL_TMEM = 1,     /* bf16 in, dstate 16, exp-Euler, L*2 and L*out a
                                     multiple of 16 bytes: TMA tiles, B/C broadcast
                                     through tensor memory, optional time split */
    SSM_SCAN_KERNEL_TMA = 2,      /* same inputs: TMA tiles, B/C read from shared memory */
    SSM_SCAN_KERNEL_TILED = 3,    /* dstate 16, exp-Euler, bf16 or fp32 in, 16-byte rows:
                                     cp.async-staged tiles */
    SSM_SCAN_KERNEL_GENERIC = 4   /* any supported shape, either discretisation */
} ssm_scan_kernel;

/* Options of ssm_scan_fwd_ex; a zero-filled struct (or NULL) means automatic. */
typedef struct {
    ssm_scan_kernel kernel;
    int threads_per_channel;  /* 0 = the kernel's own; TMEM: 4; TMA: 2 or 4;
                                 TILED: 1 (bf16 in only), 2 or 4 */
    int max_segments;         /* time segments of the TMEM kernel's split for long
                                 sequences with few channels: 0 = automatic,
                                 1 = never split, n = at most n */
    unsigned int wait_limit;  /* polls before a device-side wait gives up, in whole
                                 blocks of 1024; 0 = the default (2^24, seconds) */
    int fault_test;           /* testing only, 0 = off.  1: the TMEM kernel never copies
                                 the inputs of its second 64-step tile, so every wait
                                 for them runs out after wait_limit polls and the call
                                 is reported by ssm_device_status() as SSM_ERR_TIMEOUT.
                                 Needs a problem of at least two tiles. */
} ssm_scan_opts;

/* Device scratch ssm_scan_fwd_ex needs for this problem and these options (NULL =
 * automatic), in bytes; 0 for most shapes and whenever max_segments is 1. */
size_t ssm_scan_workspace_size(const ssm_scan_params* p, const ssm_scan_opts* opts);

/* ssm_scan_fwd with explicit options.  `workspace` is a device buffer of at least
 * ssm_scan_workspace_size(p, opts) bytes, 16-byte aligned (may be NULL when that
 * is 0); its contents on entry do not matter. */
ssm_status ssm_scan_fwd_ex(const ssm_scan_params* p, const ssm_scan_opts* opts,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Mamba-1 selective scan, backward: the reverse-mode derivative of ssm_scan_fwd
 *   (the pages train every model through the scan: "From S4 to Mamba-3", 03/System,
 *    the shared trainer; 05/Evaluation, per-model training-step latency)
 *
 * Given dy and dh_final, computes the gradients of
 *     sum_t dy_t * y_t + sum_n dh_final[n] * h_final[n]
 * with respect to every input of ssm_scan_fwd for the same `fwd` parameters (its y and
 * h_final pointers are ignored).  Walking the recurrence backwards in time with
 * g = dL/dh_t carried from later steps, E_t = exp(Delta_t A):
 *   G_t = g + do_t C_t,  do_t = dy_t SiLU(z_t),  dz_t = dy_t o_t SiLU'(z_t)
 *   dC_t += do_t h_t,  dB_t += G_t Delta_t x_t,  dx_t = sum_n G_t Delta_t B_t + do_t D
 *   dDelta_t = sum_n G_t (B_t x_t + h_{t-1} E_t A),  dA += G_t h_{t-1} E_t Delta_t,
 *   g <- G_t E_t,  d(delta)_t = dDelta_t sigmoid(delta_t + bias) under softplus,
 * where o_t is the pre-gate output; dh0 = g after step 0.
 *
 * Shapes as ssm_scan_fwd; every gradient is float32 and is written (not accumulated):
 *   dy          : [Bt, D, L]    fwd.out_dtype
 *   dh_final    : [Bt, D, N]    float32 (nullable: zero)
 *   dx, ddelta  : [Bt, D, L]
 *   dz          : [Bt, D, L]    (required exactly when fwd.z is given)
 *   dA          : [D, N]        (summed over the batch)
 *   dB, dC      : [Bt, G, N, L] (summed over the channels of the group)
 *   dD_skip     : [D]           (required exactly when fwd.D_skip is given)
 *   ddelta_bias : [D]           (required exactly when fwd.delta_bias is given)
 *   dh0         : [Bt, D, N]    (nullable: not written)
 * Limits: exponential-Euler only and dstate in {16, 32, 64, 128} (else SSM_ERR_UNSUPPORTED).
 * dA, dD_skip and ddelta_bias are summed in a fixed order and do not depend on launch
 * order.  dB and dC are sums over the channels of the group that the kernel adds up
 * with float32 atomic adds, so their last bits can differ between runs (each is within
 * rounding of the exact sum either way).
 * ------------------------------------------------------------------------- */
typedef struct {
    ssm_scan_params fwd;
    const void* dy;
    const float* dh_final;
    float* dx;
    float* ddelta;
    float* dz;
    float* dA;
    float* dB;
    float* dC;
    float* dD_skip;
    float* ddelta_bias;
    float* dh0;
} ssm_scan_bwd_params;

/* Device scratch for ssm_scan_bwd, in bytes (0 when the problem is invalid or
 * unsupported): state checkpoints at two levels, about 2 sqrt(L / 16) states per
 * channel, and per-(batch, channel) partial sums of dA, dD_skip, ddelta_bias. */
size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p);

/* Runs the backward pass.  `workspace`: at least ssm_scan_bwd_workspace_size(p) bytes,
 * 16-byte aligned; its contents on entry do not matter. */
ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * Mamba-3 scan: complex diagonal transition, exponential-trapezoidal rule
 *   ("From S4 to Mamba-3", 03/System, mamba3_minimal.py; 04/Approach, "Complex
 *    transitions for state tracking")
 *
 * Per channel d and state n, with A = A_re + i A_im (A_re = -exp(a) < 0, A_im = theta):
 *   Abar_t = exp(Delta_t A)                                           (complex)
 *   h_t    = Abar_t (h_{t-1} + (1 - lambda_t) Delta_t B_{t-1} x_{t-1})
 *            + lambda_t Delta_t B_t x_t                               (no t-1 term at t = 0)
 *   y_t    = (Re sum_n C_t[n] h_t[n] + D x_t) * SiLU(z_t)
 * At lambda = 1 and A_im = 0 this is ssm_scan_fwd with SSM_DISC_EXP_EULER (the pages'
 * reduction test).  The pages name the rule and that reduction only; this trapezoid
 * (left end decayed by the step's transition) is the reading taken.
 *
 * Shapes as ssm_scan_fwd, plus:
 *   A_re, A_im  : [D, N]        float32
 *   lam         : [Bt, D, L]    in_dtype (the trapezoid weight, after the caller's sigmoid)
 *   h0, h_final : [Bt, D, N, 2] float32 complex (re, im) pairs (nullable)
 * Limits: dstate in {4, 8, 16, 32, 64} (else SSM_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------- */
typedef struct {
    int batch, dim, dstate, seqlen, ngroups;
    ssm_dtype in_dtype, out_dtype;
    const void* x;
    const void* delta;
    const float* delta_bias;
    int delta_softplus;
    const float* A_re;
    const float* A_im;
    const void* lam;
    const void* B;
    const void* C;
    const float* D_skip;
    const void* z;
    const float* h0;
    void* y;
    float* h_final;
} ssm_mamba3_params;

/* Device scratch ssm_mamba3_scan_fwd needs, in bytes: 0 unless the sequence is split
 * into time segments (few channels, long L), then the segments' end states and sums of
 * Delta. */
size_t ssm_mamba3_scan_workspace_size(const ssm_mamba3_params* p);

/* `workspace`: at least ssm_mamba3_scan_workspace_size(p) bytes (may be NULL when 0). */
ssm_status ssm_mamba3_scan_fwd(const ssm_mamba3_params* p, void* workspace,
                               size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * S4D: linear time-invariant SSM, complex diagonal A, exact ZOH
 *   ("From S4 to Mamba-3", 03/System, s4_minimal.py; Likely questions Q01)
 *
 * Per channel d and state n, Delta = exp(log_dt[d]) and z = Delta A[d,n]:
 *   Abar = e^z,  Bbar = Delta B (e^z - 1)/z  (1 + z/2 + z^2/6 for |z| < 1e-4)
 *   recurrent form:    h_t = Abar h_{t-1} + Bbar u_t,  y_t = Re sum_n C h_t + D u_t
 *   convolution form:  K_l = Re sum_n C Bbar Abar^l,   y = K * u + D u
 * The two are equal from a zero state (the pages' equivalence test).
 *
 * Shapes (Bt = batch, D = dim, N = dstate complex states, L = seqlen):
 *   u, y          : [Bt, D, L]     in_dtype / out_dtype
 *   log_dt        : [D]            float32
 *   A, B, C       : [D, N, 2]      float32 complex (re, im)
 *   D_skip        : [D]            float32 (nullable)
 *   h0, h_final   : [Bt, D, N, 2]  float32 complex (nullable)
 * Limits: dstate in {4, 8, 16, 32, 64} (else SSM_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------- */
typedef struct {
    int batch, dim, dstate, seqlen;
    ssm_dtype in_dtype, out_dtype;
    const void* u;
    const float* log_dt;
    const float* A;
    const float* B;
    const float* C;
    const float* D_skip;
    const float* h0;
    void* y;
    float* h_final;
} ssm_s4d_params;

/* Device scratch ssm_s4d_scan_fwd needs, in bytes: 0 unless the sequence is split into
 * segments (few channels, long L), then the segments' end states. */
size_t ssm_s4d_scan_workspace_size(const ssm_s4d_params* p);

/* The recurrent form over the whole sequence (batch, u, y, h0, h_final are used).
 * `workspace`: at least ssm_s4d_scan_workspace_size(p) bytes (may be NULL when 0). */
ssm_status ssm_s4d_scan_fwd(const ssm_s4d_params* p, void* workspace, size_t workspace_bytes,
                            void* stream);

/* The convolution kernel K [dim, kernel_len] float32 (device pointer), from dim, dstate,
 * log_dt, A, B and C of `p` (the other fields are ignored). */
ssm_status ssm_s4d_kernel(const ssm_s4d_params* p, float* K, int kernel_len, void* stream);

/* The convolution form on the GPU: y = K * u + D u, K_l as above for l < L, from a zero
 * state ("From S4 to Mamba-3", 03/System: S4D trains as one FFT convolution).  The causal
 * convolution is the first L points of the cyclic one of length N = 2^ceil(log2 2L):
 * y = IFFT(FFT(K) . FFT(u)), computed in float32 (FFT error ~1e-6 of max|y|).  Uses batch,
 * dim, dstate, seqlen, dtypes, u, log_dt, A, B, C, D_skip and y of `p`; h0 and h_final
 * must be NULL (use ssm_s4d_scan_fwd for a carried state).
 * `workspace`: ssm_s4d_conv_workspace_size(p) bytes, 16-byte aligned, contents on entry
 * irrelevant (the spectrum of K, [dim, N] complex, and the transform's twiddle tables).
 * Limits: 1 <= L <= 8192 for the workspace query (N <= 16384 fits in shared memory; L = 0
 * is accepted by the call and does nothing), dim <= 65535, dstate as ssm_s4d_scan_fwd. */
size_t ssm_s4d_conv_workspace_size(const ssm_s4d_params* p);
ssm_status ssm_s4d_conv_fwd(const ssm_s4d_params* p, void* workspace, size_t workspace_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------
 * Mamba-2 chunked SSD scan (scalar A per head)
 *   ("From S4 to Mamba-3", 03/System, mamba2_minimal.py; 04/Approach)
 *
 * Shapes, Bt = batch, L = seqlen, H = nheads, P = headdim, N = dstate,
 * G = ngroups, Q = chunk_size:
 *   x, z, y     : [Bt, L, H, P]   in_dtype / out_dtype for y  (z nullable)
 *   dt          : [Bt, L, H]      in_dtype
 *   dt_bias     : [H]             float32 (nullable)
 *   A, D_skip   : [H]             float32 (D_skip nullable)
 *   B, C        : [Bt, L, G, N]   in_dtype (head h uses group h / (H / G))
 *   h0, h_final : [Bt, H, P, N]   float32 (nullable)
 * The sequence is processed in chunks of Q steps; the last chunk may be short.
 * Inside a chunk the output is a decayed-attention product and chunk states are
 * passed between chunks, so the result equals the sequential scan up to
 * rounding.  Limits: Q in {64, 128, 256}; P in {32, 64, 128}; N in {64, 128};
 * G divides H.  With bf16 inputs, P = 64 and N = 128 the tensor-core kernels
 * run every Q on 64-step tiles: for Q = 128 or 256 the decayed-attention block
 * of two different tiles of one chunk is applied through the state carried
 * between them, which is the same product regrouped (exact in real arithmetic),
 * so the result does not depend on Q there.
 * ------------------------------------------------------------------------- */
typedef struct {
    int batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
    ssm_dtype in_dtype, out_dtype;
    const void* x;
    const void* dt;
    const float* dt_bias;
    int dt_softplus;           /* nonzero: Delta = softplus(dt + dt_bias) */
    const float* A;
    const void* B;
    const void* C;
    const float* D_skip;
    const void* z;
    const float* h0;
    void* y;
    float* h_final;
    ssm_disc disc;
} ssd_params;

/* Device scratch needed by ssd_chunk_scan_fwd, in bytes (float32 chunk or
 * range states, decays and per-chunk step sums).  Only the sizes in `p` are
 * read; returns 0 when they are invalid or unsupported. */
size_t ssd_chunk_scan_workspace_size(const ssd_params* p);

/* Runs the chunked scan; `workspace` is a device buffer of at least
 * ssd_chunk_scan_workspace_size(p) bytes, contents on entry irrelevant. */
ssm_status ssd_chunk_scan_fwd(const ssd_params* p, void* workspace, size_t workspace_bytes,
                              void* stream);

/* ---------------------------------------------------------------------------
 * SSD scan without caller-provided scratch.
 * (This entry point has no counterpart in the paper; it exists for callers of
 * the library.)
 *
 * ssd_chunk_scan_fwd needs a device workspace from the caller.  Some callers
 * cannot allocate device memory: a plugin whose host framework reserves all
 * device memory in its own pool, or a serving loop that forbids allocation
 * once it is running.  This variant takes the same parameters and keeps its
 * scratch in one fixed device array inside the library, of
 * SSM_NOALLOC_SCRATCH_BYTES (32 MiB), which every GPU that loads the library
 * holds until the process exits.  It allocates nothing.
 *   - Problems whose scratch (ssd_chunk_scan_workspace_size) exceeds the array
 *     are rejected with SSM_ERR_INVALID_ARG and a message saying so.
 *   - The first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (that device must be current) and caches it; make
 *     that first call before any stream capture.  The address is valid in the
 *     CUDA context it was looked up in; a call under another context (after
 *     cudaDeviceReset, say) looks it up again.
 *   - `stream` must belong to the current device (the scratch size depends on
 *     that device); a stream of another device is refused.
 *   - All calls share the array: calls whose GPU work may overlap (other
 *     streams, other host threads) race on it; the caller must order them.
 *     The array keeps the last call's contents, and no part of it needs to
 *     start at zero.
 * ------------------------------------------------------------------------- */
#define SSM_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

ssm_status ssd_chunk_scan_fwd_noalloc(const ssd_params* p, void* stream);

/* Size in bytes of the library's fixed scratch array (SSM_NOALLOC_SCRATCH_BYTES). */
size_t ssd_noalloc_scratch_capacity(void);

/* ---------------------------------------------------------------------------
 * Single-step decode update, in place on the state
 *   ("From S4 to Mamba-3", 03/System: the incremental step() for decoding)
 *
 * Shapes, Bt = batch, H = nheads, P = headdim, N = dstate, G = ngroups:
 *   state  : [Bt, H, P, N]  float32, read and overwritten with the new state
 *   x, z, y: [Bt, H, P]     in_dtype / out_dtype for y  (z nullable)
 *   dt     : [Bt, H]        in_dtype;  dt_bias [H] float32 (nullable)
 *   A      : [H] float32 (a_per_state = 0, Mamba-2 form) or
 *            [H, N] float32 (a_per_state = 1, Mamba-1 form: H = channels, P = 1)
 *   B, C   : [Bt, G, N]     in_dtype (head h uses group h / (H / G))
 *   D_skip : [H] float32 (nullable)
 * Limits: N a multiple of 4 up to 256 for the vectorised path (other N are
 * served by a scalar path); G divides H.
 * ------------------------------------------------------------------------- */
typedef struct {
    int batch, nheads, headdim, dstate, ngroups;
    int a_per_state;
    ssm_dtype in_dtype, out_dtype;
    float* state;
    const void* x;
    const void* dt;
    const float* dt_bias;
    int dt_softplus;
    const float* A;
    const void* B;
    const void* C;
    const float* D_skip;
    const void* z;
    void* y;
    ssm_disc disc;
} ssm_step_params;

ssm_status ssm_state_update(const ssm_step_params* p, void* stream);

/* ---------------------------------------------------------------------------
 * Multi-token decode: `ntokens` consecutive steps of ssm_state_update in one call
 *   (the pages' incremental step() applied T times; 03/System)
 *
 * The state is read once, advanced through the T tokens in registers and written
 * once, so the HBM traffic per token falls from the whole state to the token data.
 * Token-major layouts, each token's slice laid out as in ssm_state_update:
 *   x, z, y : [T, Bt, H, P];   dt : [T, Bt, H];   B, C : [T, Bt, G, N]
 *   state, A, D_skip, dt_bias: as in ssm_state_update.
 * y[t] is the output after token t.  Limits: 1 <= ntokens <= 256, otherwise as
 * ssm_state_update.  ntokens = 1 equals ssm_state_update.
 * ------------------------------------------------------------------------- */
ssm_status ssm_state_update_tokens(const ssm_step_params* p, int ntokens, void* stream);

/* ---------------------------------------------------------------------------
 * Mamba-2 SSD backward: the reverse-mode derivative of the SSD scan
 *   (same passages as ssm_scan_bwd; mamba2_minimal.py for the scalar-A form)
 *
 * With a scalar A per head the SSD recurrence is the Mamba-1 scan over the H*P channels
 * of the heads, A tied across a head's channels and states and Delta, D and dt_bias
 * shared by its P channels; the gradients are those of ssm_scan_bwd on that view, the
 * tied ones summed (dA over the batch, the head's channels and the states; ddt over the
 * head's channels).  The derivative is of the recurrence, so it does not depend on the
 * chunk size of the forward call (fwd.chunk_size, y and h_final are ignored).
 *
 * For (dstate, headdim) in {(128, 64), (64, 64), (128, 32), (64, 32)} with in_dtype ==
 * out_dtype the library computes it in chunked form (64-step chunks, the pages' chunked
 * SSD differentiated product by product, float32 arithmetic); other shapes run the
 * tied recurrence.  Both give the same gradients to float32 rounding.
 *
 * Shapes as ssd_chunk_scan_fwd; every gradient is float32 and is written:
 *   dy          : [Bt, L, H, P]  fwd.out_dtype
 *   dh_final    : [Bt, H, P, N]  (nullable: zero)
 *   dx          : [Bt, L, H, P]
 *   ddt         : [Bt, L, H]
 *   dz          : [Bt, L, H, P]  (required exactly when fwd.z is given)
 *   dA          : [H]
 *   dB, dC      : [Bt, L, G, N]
 *   dD_skip     : [H]            (required exactly when fwd.D_skip is given)
 *   ddt_bias    : [H]            (required exactly when fwd.dt_bias is given)
 *   dh0         : [Bt, H, P, N]  (nullable: not written)
 * Limits: exponential-Euler only, dstate in {16, 32, 64, 128}.
 * ------------------------------------------------------------------------- */
typedef struct {
    ssd_params fwd;
    const void* dy;
    const float* dh_final;
    float* dx;
    float* ddt;
    float* dz;
    float* dA;
    float* dB;
    float* dC;
    float* dD_skip;
    float* ddt_bias;
    float* dh0;
} ssd_bwd_params;

/* Device scratch for ssd_scan_bwd in bytes (0 when invalid or unsupported).  Chunked
 * form: the chunk states and adjoints of a slice of (batch, head) sequences, the slice
 * no larger than x and dy together, plus a few floats per chunk; dB and dC are sums over
 * a group's heads added up with float32 atomic adds, ddt is written once.  Tied
 * recurrence: as for ssm_scan_bwd, and ddt, like dB and dC, is a sum over channels (the
 * head's P) added up with atomic adds.  dA, dD_skip, ddt_bias are summed in a fixed
 * order in both. */
size_t ssd_scan_bwd_workspace_size(const ssd_bwd_params* p);

ssm_status ssd_scan_bwd(const ssd_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* ssm_last_error(void);

/* Status of the work launched on the current device: waits for the device
 * (cudaDeviceSynchronize, so not inside a stream capture), then returns
 * SSM_ERR_TIMEOUT if a bounded device-side wait gave up since the previous call
 * (ssm_last_error() names the kernels; the outputs of the calls in between are
 * not valid), SSM_ERR_CUDA if the device reports an error, else SSM_OK.  Reading
 * clears the record. */
ssm_status ssm_device_status(void);

/* The same record as a count: how many bounded device-side waits gave up since
 * the previous read (0 in correct operation, and 0 after a CUDA error).  Waits
 * for the device and clears the record. */
unsigned int ssm_wait_timeouts(void);

/* SSM_ABI_VERSION of the loaded library. */
int ssm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSMSCAN_H */
