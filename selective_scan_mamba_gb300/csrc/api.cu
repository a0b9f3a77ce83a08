// api.cu -- the C ABI of libssmscan: argument checks, launch planning, status codes.
// Every check runs on the host before anything is launched; a rejected call touches
// neither the GPU nor any buffer.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "launch.h"
#include "ssmscan.h"

namespace {

thread_local char g_err[512] = "";

ssm_status fail(ssm_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

ssm_status cuda_fail(cudaError_t e, const char* where) {
    return fail(SSM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dtype_ok(ssm_dtype d) { return d == SSM_F32 || d == SSM_BF16; }

// Host-side fault hook for tests of the error paths: SSM_FAULT_INJECT=launch makes the
// next launch report a CUDA error without touching the GPU.
bool injected_launch_fault() {
    const char* v = getenv("SSM_FAULT_INJECT");
    return v && strcmp(v, "launch") == 0;
}

#define REQUIRE(cond, ...)                                    \
    do {                                                      \
        if (!(cond)) return fail(SSM_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

#define REQUIRE_PTR(p, name)                                                       \
    do {                                                                           \
        if ((p) == nullptr) return fail(SSM_ERR_INVALID_ARG, "%s is NULL", name);  \
        if (!aligned16(p)) return fail(SSM_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

#define OPTIONAL_PTR(p, name)                                                      \
    do {                                                                           \
        if ((p) != nullptr && !aligned16(p))                                       \
            return fail(SSM_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);   \
    } while (0)

// sizes, dtypes and modes only (what the workspace query reads)
ssm_status check_scan_sizes(const ssm_scan_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->batch >= 1 && p->dim >= 1 && p->dstate >= 1 && p->seqlen >= 0 && p->ngroups >= 1,
            "bad sizes: batch=%d dim=%d dstate=%d seqlen=%d ngroups=%d", p->batch, p->dim,
            p->dstate, p->seqlen, p->ngroups);
    REQUIRE(p->dim % p->ngroups == 0, "ngroups=%d does not divide dim=%d", p->ngroups, p->dim);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(p->disc == SSM_DISC_EXP_EULER || p->disc == SSM_DISC_ZOH, "unknown discretisation");
    REQUIRE(static_cast<long long>(p->batch) * p->dim * (p->seqlen > 0 ? p->seqlen : 1) < (1LL << 40),
            "tensor too large");
    if (p->dstate > 256) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 256", p->dstate);
    if (static_cast<long long>(p->batch) * p->dim > (1LL << 31) - 1)
        return fail(SSM_ERR_UNSUPPORTED, "batch*dim too large");
    return SSM_OK;
}

ssm_status check_scan(const ssm_scan_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->batch >= 1 && p->dim >= 1 && p->dstate >= 1 && p->seqlen >= 0 && p->ngroups >= 1,
            "bad sizes: batch=%d dim=%d dstate=%d seqlen=%d ngroups=%d", p->batch, p->dim,
            p->dstate, p->seqlen, p->ngroups);
    REQUIRE(p->dim % p->ngroups == 0, "ngroups=%d does not divide dim=%d", p->ngroups, p->dim);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(p->disc == SSM_DISC_EXP_EULER || p->disc == SSM_DISC_ZOH, "unknown discretisation");
    REQUIRE(static_cast<long long>(p->batch) * p->dim * (p->seqlen > 0 ? p->seqlen : 1) < (1LL << 40),
            "tensor too large");
    if (p->dstate > 256) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 256", p->dstate);
    if (static_cast<long long>(p->batch) * p->dim > (1LL << 31) - 1)
        return fail(SSM_ERR_UNSUPPORTED, "batch*dim too large");
    REQUIRE_PTR(p->A, "A");
    OPTIONAL_PTR(p->delta_bias, "delta_bias");
    OPTIONAL_PTR(p->D_skip, "D_skip");
    OPTIONAL_PTR(p->h0, "h0");
    OPTIONAL_PTR(p->h_final, "h_final");
    if (p->seqlen > 0) {
        REQUIRE_PTR(p->x, "x");
        REQUIRE_PTR(p->delta, "delta");
        REQUIRE_PTR(p->B, "B");
        REQUIRE_PTR(p->C, "C");
        REQUIRE_PTR(p->y, "y");
        OPTIONAL_PTR(p->z, "z");
    }
    return SSM_OK;
}

// sizes, modes and support of the backward (what its workspace query reads)
ssm_status check_scan_bwd_sizes(const ssm_scan_bwd_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    ssm_status st = check_scan_sizes(&p->fwd);
    if (st != SSM_OK) return st;
    if (p->fwd.disc != SSM_DISC_EXP_EULER)
        return fail(SSM_ERR_UNSUPPORTED, "backward: exponential-Euler only");
    if (!ssm::m1_bwd_supported(*p))
        return fail(SSM_ERR_UNSUPPORTED, "backward: dstate=%d (16, 32, 64 or 128 supported)", p->fwd.dstate);
    return SSM_OK;
}

ssm_status check_scan_bwd(const ssm_scan_bwd_params* p) {
    ssm_status st = check_scan_bwd_sizes(p);
    if (st != SSM_OK) return st;
    const ssm_scan_params* f = &p->fwd;
    REQUIRE_PTR(f->A, "A");
    REQUIRE_PTR(p->dA, "dA");
    OPTIONAL_PTR(f->h0, "h0");
    OPTIONAL_PTR(p->dh_final, "dh_final");
    OPTIONAL_PTR(p->dh0, "dh0");
    REQUIRE((f->D_skip == nullptr) == (p->dD_skip == nullptr), "dD_skip must be given exactly when D_skip is");
    REQUIRE((f->delta_bias == nullptr) == (p->ddelta_bias == nullptr),
            "ddelta_bias must be given exactly when delta_bias is");
    REQUIRE((f->z == nullptr) == (p->dz == nullptr), "dz must be given exactly when z is");
    OPTIONAL_PTR(f->D_skip, "D_skip");
    OPTIONAL_PTR(f->delta_bias, "delta_bias");
    OPTIONAL_PTR(p->dD_skip, "dD_skip");
    OPTIONAL_PTR(p->ddelta_bias, "ddelta_bias");
    if (f->seqlen > 0) {
        REQUIRE_PTR(f->x, "x");
        REQUIRE_PTR(f->delta, "delta");
        REQUIRE_PTR(f->B, "B");
        REQUIRE_PTR(f->C, "C");
        REQUIRE_PTR(p->dy, "dy");
        REQUIRE_PTR(p->dx, "dx");
        REQUIRE_PTR(p->ddelta, "ddelta");
        REQUIRE_PTR(p->dB, "dB");
        REQUIRE_PTR(p->dC, "dC");
        OPTIONAL_PTR(f->z, "z");
        OPTIONAL_PTR(p->dz, "dz");
    }
    return SSM_OK;
}

ssm_status check_s4d_params(const ssm_s4d_params* p, bool scan) {
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->dim >= 1 && p->dstate >= 1, "bad sizes: dim=%d dstate=%d", p->dim, p->dstate);
    if (!ssm::s4d_supported(p->dstate))
        return fail(SSM_ERR_UNSUPPORTED, "s4d: dstate=%d (4, 8, 16, 32 or 64 supported)", p->dstate);
    REQUIRE_PTR(p->log_dt, "log_dt");
    REQUIRE_PTR(p->A, "A");
    REQUIRE_PTR(p->B, "B");
    REQUIRE_PTR(p->C, "C");
    if (!scan) return SSM_OK;
    REQUIRE(p->batch >= 1 && p->seqlen >= 0, "bad sizes: batch=%d seqlen=%d", p->batch, p->seqlen);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(static_cast<long long>(p->batch) * p->dim * (p->seqlen > 0 ? p->seqlen : 1) < (1LL << 40),
            "tensor too large");
    OPTIONAL_PTR(p->D_skip, "D_skip");
    OPTIONAL_PTR(p->h0, "h0");
    OPTIONAL_PTR(p->h_final, "h_final");
    if (p->seqlen > 0) {
        REQUIRE_PTR(p->u, "u");
        REQUIRE_PTR(p->y, "y");
    }
    return SSM_OK;
}

ssm_status check_ssd_bwd_sizes(const ssd_bwd_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    const ssd_params* f = &p->fwd;
    REQUIRE(f->batch >= 1 && f->seqlen >= 0 && f->nheads >= 1 && f->headdim >= 1 && f->dstate >= 1 &&
                f->ngroups >= 1,
            "bad sizes: batch=%d seqlen=%d nheads=%d headdim=%d dstate=%d ngroups=%d", f->batch,
            f->seqlen, f->nheads, f->headdim, f->dstate, f->ngroups);
    REQUIRE(f->nheads % f->ngroups == 0, "ngroups=%d does not divide nheads=%d", f->ngroups, f->nheads);
    REQUIRE(dtype_ok(f->in_dtype) && dtype_ok(f->out_dtype), "unknown dtype");
    REQUIRE(static_cast<long long>(f->batch) * f->seqlen * f->nheads * f->headdim < (1LL << 40),
            "tensor too large");
    if (static_cast<long long>(f->nheads) * f->headdim > (1 << 24))
        return fail(SSM_ERR_UNSUPPORTED, "nheads*headdim too large");
    if (f->disc != SSM_DISC_EXP_EULER) return fail(SSM_ERR_UNSUPPORTED, "backward: exponential-Euler only");
    if (!ssm::ssd_bwd_supported(*p))
        return fail(SSM_ERR_UNSUPPORTED, "backward: dstate=%d (16, 32, 64 or 128 supported)", f->dstate);
    return SSM_OK;
}

ssm_status check_ssd_bwd(const ssd_bwd_params* p) {
    ssm_status st = check_ssd_bwd_sizes(p);
    if (st != SSM_OK) return st;
    const ssd_params* f = &p->fwd;
    REQUIRE_PTR(f->A, "A");
    REQUIRE_PTR(p->dA, "dA");
    OPTIONAL_PTR(f->h0, "h0");
    OPTIONAL_PTR(p->dh_final, "dh_final");
    OPTIONAL_PTR(p->dh0, "dh0");
    REQUIRE((f->D_skip == nullptr) == (p->dD_skip == nullptr), "dD_skip must be given exactly when D_skip is");
    REQUIRE((f->dt_bias == nullptr) == (p->ddt_bias == nullptr), "ddt_bias must be given exactly when dt_bias is");
    REQUIRE((f->z == nullptr) == (p->dz == nullptr), "dz must be given exactly when z is");
    OPTIONAL_PTR(f->D_skip, "D_skip");
    OPTIONAL_PTR(f->dt_bias, "dt_bias");
    OPTIONAL_PTR(p->dD_skip, "dD_skip");
    OPTIONAL_PTR(p->ddt_bias, "ddt_bias");
    if (f->seqlen > 0) {
        REQUIRE_PTR(f->x, "x");
        REQUIRE_PTR(f->dt, "dt");
        REQUIRE_PTR(f->B, "B");
        REQUIRE_PTR(f->C, "C");
        REQUIRE_PTR(p->dy, "dy");
        REQUIRE_PTR(p->dx, "dx");
        REQUIRE_PTR(p->ddt, "ddt");
        REQUIRE_PTR(p->dB, "dB");
        REQUIRE_PTR(p->dC, "dC");
        OPTIONAL_PTR(f->z, "z");
        OPTIONAL_PTR(p->dz, "dz");
    }
    return SSM_OK;
}

ssm::M1Args scan_args(const ssm_scan_params* p) {
    ssm::M1Args a;
    a.batch = p->batch;
    a.dim = p->dim;
    a.dstate = p->dstate;
    a.seqlen = p->seqlen;
    a.ngroups = p->ngroups;
    a.in_dtype = p->in_dtype;
    a.out_dtype = p->out_dtype;
    a.x = p->x;
    a.delta = p->delta;
    a.delta_bias = p->delta_bias;
    a.delta_softplus = p->delta_softplus;
    a.A = p->A;
    a.B = p->B;
    a.C = p->C;
    a.D = p->D_skip;
    a.z = p->z;
    a.h0 = p->h0;
    a.y = p->y;
    a.h_final = p->h_final;
    a.disc = p->disc;
    a.cpb_max = 0;
    return a;
}

ssm_status check_ssd_sizes(const ssd_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->batch >= 1 && p->seqlen >= 0 && p->nheads >= 1 && p->headdim >= 1 &&
                p->dstate >= 1 && p->ngroups >= 1 && p->chunk_size >= 1,
            "bad sizes: batch=%d seqlen=%d nheads=%d headdim=%d dstate=%d ngroups=%d chunk=%d",
            p->batch, p->seqlen, p->nheads, p->headdim, p->dstate, p->ngroups, p->chunk_size);
    REQUIRE(p->nheads % p->ngroups == 0, "ngroups=%d does not divide nheads=%d", p->ngroups,
            p->nheads);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(p->disc == SSM_DISC_EXP_EULER || p->disc == SSM_DISC_ZOH, "unknown discretisation");
    if (p->chunk_size != 64 && p->chunk_size != 128 && p->chunk_size != 256)
        return fail(SSM_ERR_UNSUPPORTED, "chunk_size=%d (supported: 64, 128, 256)", p->chunk_size);
    if (p->headdim != 32 && p->headdim != 64 && p->headdim != 128)
        return fail(SSM_ERR_UNSUPPORTED, "headdim=%d (supported: 32, 64, 128)", p->headdim);
    if (p->dstate != 64 && p->dstate != 128)
        return fail(SSM_ERR_UNSUPPORTED, "dstate=%d (supported: 64, 128)", p->dstate);
    if (p->headdim * p->dstate > 8192)
        return fail(SSM_ERR_UNSUPPORTED, "headdim*dstate=%d > 8192", p->headdim * p->dstate);
    REQUIRE(static_cast<long long>(p->batch) * (p->seqlen > 0 ? p->seqlen : 1) * p->nheads * p->headdim <
                (1LL << 40),
            "tensor too large");
    return SSM_OK;
}

ssm_status check_ssd(const ssd_params* p) {
    ssm_status st = check_ssd_sizes(p);
    if (st != SSM_OK) return st;
    REQUIRE_PTR(p->A, "A");
    OPTIONAL_PTR(p->dt_bias, "dt_bias");
    OPTIONAL_PTR(p->D_skip, "D_skip");
    OPTIONAL_PTR(p->h0, "h0");
    OPTIONAL_PTR(p->h_final, "h_final");
    if (p->seqlen > 0) {
        REQUIRE_PTR(p->x, "x");
        REQUIRE_PTR(p->dt, "dt");
        REQUIRE_PTR(p->B, "B");
        REQUIRE_PTR(p->C, "C");
        REQUIRE_PTR(p->y, "y");
        OPTIONAL_PTR(p->z, "z");
    }
    return SSM_OK;
}

ssm_status check_step(const ssm_step_params* p) {
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->batch >= 1 && p->nheads >= 1 && p->headdim >= 1 && p->dstate >= 1 &&
                p->ngroups >= 1,
            "bad sizes: batch=%d nheads=%d headdim=%d dstate=%d ngroups=%d", p->batch, p->nheads,
            p->headdim, p->dstate, p->ngroups);
    REQUIRE(p->nheads % p->ngroups == 0, "ngroups=%d does not divide nheads=%d", p->ngroups,
            p->nheads);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(p->disc == SSM_DISC_EXP_EULER || p->disc == SSM_DISC_ZOH, "unknown discretisation");
    REQUIRE(p->a_per_state == 0 || p->a_per_state == 1, "a_per_state must be 0 or 1");
    if (p->dstate > 4096) return fail(SSM_ERR_UNSUPPORTED, "dstate=%d > 4096", p->dstate);
    REQUIRE(static_cast<long long>(p->batch) * p->nheads * p->headdim * p->dstate < (1LL << 40),
            "state too large");
    // the kernels keep (batch, head) indices and B/C row offsets in 32 bits
    if (static_cast<long long>(p->batch) * p->nheads > (1LL << 31) - 1 ||
        static_cast<long long>(p->batch) * p->ngroups * p->dstate > (1LL << 31) - 1)
        return fail(SSM_ERR_UNSUPPORTED, "batch*nheads or batch*ngroups*dstate too large");
    REQUIRE_PTR(p->state, "state");
    REQUIRE_PTR(p->x, "x");
    REQUIRE_PTR(p->dt, "dt");
    REQUIRE_PTR(p->A, "A");
    REQUIRE_PTR(p->B, "B");
    REQUIRE_PTR(p->C, "C");
    REQUIRE_PTR(p->y, "y");
    OPTIONAL_PTR(p->dt_bias, "dt_bias");
    OPTIONAL_PTR(p->D_skip, "D_skip");
    OPTIONAL_PTR(p->z, "z");
    return SSM_OK;
}

}  // namespace

namespace ssm {
ssm_status set_error(ssm_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace ssm

extern "C" {

int ssm_abi_version(void) { return SSM_ABI_VERSION; }

const char* ssm_last_error(void) { return g_err; }

unsigned int ssm_wait_timeouts(void) {
    return ssm::m1_tma_wait_timeouts() + ssm::m1_tmem_wait_timeouts() + ssm::ssd_tc_wait_timeouts();
}

size_t ssm_scan_workspace_size(const ssm_scan_params* p) {
    if (check_scan_sizes(p) != SSM_OK || p->seqlen == 0) return 0;
    ssm::M1Plan plan;
    if (ssm::m1_tmem_plan(scan_args(p), &plan) != cudaSuccess) return 0;
    return plan.kind == ssm::M1Plan::kTmem ? plan.ws_bytes : 0;
}

size_t ssm_mamba3_scan_workspace_size(const ssm_mamba3_params* p) {
    if (p == nullptr || p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->ngroups < 1 ||
        p->dim % p->ngroups != 0 || !ssm::m3_supported(p->dstate))
        return 0;
    return ssm::m3_workspace_size(*p);
}

ssm_status ssm_mamba3_scan_fwd(const ssm_mamba3_params* p, void* workspace, size_t workspace_bytes,
                               void* stream) {
    g_err[0] = '\0';
    REQUIRE(p != nullptr, "params is NULL");
    REQUIRE(p->batch >= 1 && p->dim >= 1 && p->dstate >= 1 && p->seqlen >= 0 && p->ngroups >= 1,
            "bad sizes: batch=%d dim=%d dstate=%d seqlen=%d ngroups=%d", p->batch, p->dim,
            p->dstate, p->seqlen, p->ngroups);
    REQUIRE(p->dim % p->ngroups == 0, "ngroups=%d does not divide dim=%d", p->ngroups, p->dim);
    REQUIRE(dtype_ok(p->in_dtype) && dtype_ok(p->out_dtype), "unknown dtype");
    REQUIRE(static_cast<long long>(p->batch) * p->dim * (p->seqlen > 0 ? p->seqlen : 1) < (1LL << 40),
            "tensor too large");
    if (!ssm::m3_supported(p->dstate))
        return fail(SSM_ERR_UNSUPPORTED, "mamba3: dstate=%d (4, 8, 16, 32 or 64 supported)", p->dstate);
    REQUIRE_PTR(p->A_re, "A_re");
    REQUIRE_PTR(p->A_im, "A_im");
    OPTIONAL_PTR(p->delta_bias, "delta_bias");
    OPTIONAL_PTR(p->D_skip, "D_skip");
    OPTIONAL_PTR(p->h0, "h0");
    OPTIONAL_PTR(p->h_final, "h_final");
    if (p->seqlen > 0) {
        REQUIRE_PTR(p->x, "x");
        REQUIRE_PTR(p->delta, "delta");
        REQUIRE_PTR(p->lam, "lam");
        REQUIRE_PTR(p->B, "B");
        REQUIRE_PTR(p->C, "C");
        REQUIRE_PTR(p->y, "y");
        OPTIONAL_PTR(p->z, "z");
    }
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->seqlen == 0) {
        if (p->h_final) {
            const size_t bytes = static_cast<size_t>(p->batch) * p->dim * p->dstate * 2 * sizeof(float);
            cudaError_t e = p->h0 ? cudaMemcpyAsync(p->h_final, p->h0, bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(p->h_final, 0, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e, "ssm_mamba3_scan_fwd (empty sequence)");
        }
        return SSM_OK;
    }
    const size_t need = ssm::m3_workspace_size(*p);
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    cudaError_t e = ssm::m3_launch(*p, workspace, s);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_mamba3_scan_fwd launch");
    return SSM_OK;
}


size_t ssm_s4d_scan_workspace_size(const ssm_s4d_params* p) {
    if (p == nullptr || p->batch < 1 || p->dim < 1 || p->seqlen < 0 || !ssm::s4d_supported(p->dstate))
        return 0;
    return ssm::s4d_workspace_size(*p);
}

ssm_status ssm_s4d_scan_fwd(const ssm_s4d_params* p, void* workspace, size_t workspace_bytes,
                            void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_s4d_params(p, true);
    if (st != SSM_OK) return st;
    const size_t need = ssm::s4d_workspace_size(*p);
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->seqlen == 0) {
        if (p->h_final) {
            const size_t bytes = static_cast<size_t>(p->batch) * p->dim * p->dstate * 2 * sizeof(float);
            cudaError_t e = p->h0 ? cudaMemcpyAsync(p->h_final, p->h0, bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(p->h_final, 0, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_scan_fwd (empty sequence)");
        }
        return SSM_OK;
    }
    cudaError_t e = ssm::s4d_launch(*p, workspace, s);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_scan_fwd launch");
    return SSM_OK;
}

ssm_status ssm_s4d_kernel(const ssm_s4d_params* p, float* K, int kernel_len, void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_s4d_params(p, false);
    if (st != SSM_OK) return st;
    REQUIRE(kernel_len >= 0, "kernel_len=%d", kernel_len);
    if (p->dim > 65535) return fail(SSM_ERR_UNSUPPORTED, "s4d kernel: dim=%d > 65535", p->dim);
    if (kernel_len > 0) REQUIRE_PTR(K, "K");
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::s4d_kernel_launch(*p, K, kernel_len, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_kernel launch");
    return SSM_OK;
}

size_t ssd_scan_bwd_workspace_size(const ssd_bwd_params* p) {
    if (check_ssd_bwd_sizes(p) != SSM_OK) return 0;
    return ssm::ssd_bwd_workspace_size(*p);
}

ssm_status ssd_scan_bwd(const ssd_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_ssd_bwd(p);
    if (st != SSM_OK) return st;
    const size_t need = ssm::ssd_bwd_workspace_size(*p);
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::ssd_bwd_launch(*p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_bwd launch");
    return SSM_OK;
}

size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p) {
    if (check_scan_bwd_sizes(p) != SSM_OK) return 0;
    return ssm::m1_bwd_workspace_size(*p);
}

ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_scan_bwd(p);
    if (st != SSM_OK) return st;
    const size_t need = ssm::m1_bwd_workspace_size(*p);
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::m1_bwd_launch(*p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_bwd launch");
    return SSM_OK;
}

ssm_status ssm_scan_fwd(const ssm_scan_params* p, void* workspace, size_t workspace_bytes,
                        void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_scan(p);
    if (st != SSM_OK) return st;
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->seqlen == 0) {
        if (p->h_final) {
            const size_t bytes = static_cast<size_t>(p->batch) * p->dim * p->dstate * sizeof(float);
            cudaError_t e = p->h0 ? cudaMemcpyAsync(p->h_final, p->h0, bytes, cudaMemcpyDeviceToDevice, s)
                                  : cudaMemsetAsync(p->h_final, 0, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd (empty sequence)");
        }
        return SSM_OK;
    }
    ssm::M1Args a = scan_args(p);
    ssm::M1Plan plan;
    cudaError_t e = ssm::m1_tmem_plan(a, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd plan");
    if (plan.kind == ssm::M1Plan::kTmem) {
        if (workspace_bytes < plan.ws_bytes)
            return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                        plan.ws_bytes);
        if (plan.ws_bytes > 0 && (workspace == nullptr || !aligned16(workspace)))
            return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
        e = ssm::m1_tmem_launch(a, plan, workspace, s);
        if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
        return SSM_OK;
    }
    e = ssm::m1_tma_plan(a, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd plan");
    if (plan.kind == ssm::M1Plan::kTma) {
        e = ssm::m1_tma_launch(a, plan, s);
        if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
        return SSM_OK;
    }
    e = ssm::m1_plan(a, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd plan");
    e = ssm::m1_launch(a, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
    return SSM_OK;
}

static ssm::SsdArgs ssd_args(const ssd_params* p, void* workspace) {
    ssm::SsdArgs a;
    a.batch = p->batch;
    a.seqlen = p->seqlen;
    a.nheads = p->nheads;
    a.headdim = p->headdim;
    a.dstate = p->dstate;
    a.ngroups = p->ngroups;
    a.chunk = p->chunk_size;
    a.in_dtype = p->in_dtype;
    a.out_dtype = p->out_dtype;
    a.x = p->x;
    a.dt = p->dt;
    a.dt_bias = p->dt_bias;
    a.dt_softplus = p->dt_softplus;
    a.A = p->A;
    a.B = p->B;
    a.C = p->C;
    a.D = p->D_skip;
    a.z = p->z;
    a.h0 = p->h0;
    a.y = p->y;
    a.h_final = p->h_final;
    a.disc = p->disc;
    a.ws_states = static_cast<float*>(workspace);
    a.ws_decay = nullptr;
    return a;
}

size_t ssd_chunk_scan_workspace_size(const ssd_params* p) {
    if (check_ssd_sizes(p) != SSM_OK) return 0;
    return ssm::ssd_workspace_bytes(ssd_args(p, nullptr));
}

ssm_status ssd_chunk_scan_fwd(const ssd_params* p, void* workspace, size_t workspace_bytes,
                              void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_ssd(p);
    if (st != SSM_OK) return st;
    ssm::SsdArgs a = ssd_args(p, workspace);
    const size_t need = ssm::ssd_workspace_bytes(a);
    if (workspace_bytes < need)
        return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (workspace == nullptr || !aligned16(workspace)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    if (!ssm::ssd_tc_supported(a)) {
        // CUDA-core path: chunk states, then per-chunk decay sums, in the workspace
        const size_t nch = (static_cast<size_t>(p->seqlen) + p->chunk_size - 1) / p->chunk_size;
        const size_t states = static_cast<size_t>(p->batch) * p->nheads * nch * p->headdim *
                              p->dstate * sizeof(float);
        a.ws_decay = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              ((states + 255) / 256) * 256);
    }
    cudaError_t e = ssm::ssd_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssd_chunk_scan_fwd launch");
    return SSM_OK;
}

static ssm_status state_update(const ssm_step_params* p, int ntokens, void* stream) {
    g_err[0] = '\0';
    ssm_status st = check_step(p);
    if (st != SSM_OK) return st;
    REQUIRE(ntokens >= 1 && ntokens <= 256, "ntokens=%d (1..256)", ntokens);
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    ssm::StepArgs a;
    a.batch = p->batch;
    a.nheads = p->nheads;
    a.headdim = p->headdim;
    a.dstate = p->dstate;
    a.ngroups = p->ngroups;
    a.a_per_state = p->a_per_state;
    a.in_dtype = p->in_dtype;
    a.out_dtype = p->out_dtype;
    a.state = p->state;
    a.x = p->x;
    a.dt = p->dt;
    a.dt_bias = p->dt_bias;
    a.dt_softplus = p->dt_softplus;
    a.A = p->A;
    a.B = p->B;
    a.C = p->C;
    a.D = p->D_skip;
    a.z = p->z;
    a.y = p->y;
    a.disc = p->disc;
    a.ntok = ntokens;
    cudaError_t e = ssm::step_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_state_update launch");
    return SSM_OK;
}

ssm_status ssm_state_update(const ssm_step_params* p, void* stream) {
    return state_update(p, 1, stream);
}

ssm_status ssm_state_update_tokens(const ssm_step_params* p, int ntokens, void* stream) {
    return state_update(p, ntokens, stream);
}

}  // extern "C"
