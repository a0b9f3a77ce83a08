// api.cu -- the C ABI of libssmscan: argument checks, launch planning, status codes.
// Every check runs on the host before anything is launched; a rejected call touches
// neither the GPU nor any buffer.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <initializer_list>

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

size_t esize(ssm_dtype d) { return d == SSM_BF16 ? 2 : 4; }

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

#define RETURN_IF_FAILED(expr)           \
    do {                                 \
        const ssm_status st_ = (expr);   \
        if (st_ != SSM_OK) return st_;   \
    } while (0)

// ---------------------------------------------------------------------------------------
// overlap checks: byte ranges of the tensors a call writes against those it reads
// ---------------------------------------------------------------------------------------
struct Span {
    const void* p;
    size_t bytes;
    const char* name;
};

bool overlap(const Span& a, const Span& b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every output against every input and against the other outputs.
ssm_status check_disjoint(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        for (const Span& i : ins)
            if (overlap(*o, i))
                return fail(SSM_ERR_INVALID_ARG, "%s overlaps the input %s", o->name, i.name);
        for (auto q = outs.begin(); q != o; ++q)
            if (overlap(*o, *q))
                return fail(SSM_ERR_INVALID_ARG, "%s overlaps the output %s", o->name, q->name);
    }
    return SSM_OK;
}

ssm_status check_workspace(const void* ws, size_t have, size_t need) {
    if (have < need) return fail(SSM_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", have, need);
    if (need > 0 && (ws == nullptr || !aligned16(ws)))
        return fail(SSM_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
    return SSM_OK;
}

// ---------------------------------------------------------------------------------------
// per entry point: sizes, dtypes and modes (all the workspace queries read), then, when
// `ptrs`, the pointers and their overlaps
// ---------------------------------------------------------------------------------------
ssm_status check_scan(const ssm_scan_params* p, bool ptrs) {
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
    if (!ptrs) return SSM_OK;
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

// byte sizes of the scan's tensors
struct ScanSizes {
    size_t row, y, bc, a, d, h;
    explicit ScanSizes(const ssm_scan_params& p) {
        const size_t bdl = static_cast<size_t>(p.batch) * p.dim * p.seqlen;
        row = bdl * esize(p.in_dtype);
        y = bdl * esize(p.out_dtype);
        bc = static_cast<size_t>(p.batch) * p.ngroups * p.dstate * p.seqlen * esize(p.in_dtype);
        a = static_cast<size_t>(p.dim) * p.dstate * 4;
        d = static_cast<size_t>(p.dim) * 4;
        h = static_cast<size_t>(p.batch) * p.dim * p.dstate * 4;
    }
};

ssm_status check_scan_overlap(const ssm_scan_params* p, const void* ws, size_t ws_bytes) {
    const ScanSizes s(*p);
    return check_disjoint({{p->y, s.y, "y"}, {p->h_final, s.h, "h_final"}, {ws, ws_bytes, "workspace"}},
                          {{p->x, s.row, "x"}, {p->delta, s.row, "delta"}, {p->z, s.row, "z"},
                           {p->B, s.bc, "B"}, {p->C, s.bc, "C"}, {p->A, s.a, "A"},
                           {p->D_skip, s.d, "D_skip"}, {p->delta_bias, s.d, "delta_bias"},
                           {p->h0, s.h, "h0"}});
}

ssm_status check_scan_opts(const ssm_scan_opts* o) {
    if (o == nullptr) return SSM_OK;
    REQUIRE(o->kernel >= SSM_SCAN_KERNEL_AUTO && o->kernel <= SSM_SCAN_KERNEL_GENERIC,
            "unknown kernel %d", static_cast<int>(o->kernel));
    REQUIRE(o->threads_per_channel == 0 || o->threads_per_channel == 1 ||
                o->threads_per_channel == 2 || o->threads_per_channel == 4,
            "threads_per_channel=%d (0, 1, 2 or 4)", o->threads_per_channel);
    REQUIRE(o->max_segments >= 0, "max_segments=%d", o->max_segments);
    REQUIRE(o->fault_test == 0 || o->fault_test == 1, "fault_test=%d", o->fault_test);
    return SSM_OK;
}

ssm_status check_scan_bwd(const ssm_scan_bwd_params* p, bool ptrs) {
    REQUIRE(p != nullptr, "params is NULL");
    RETURN_IF_FAILED(check_scan(&p->fwd, false));
    if (p->fwd.disc != SSM_DISC_EXP_EULER)
        return fail(SSM_ERR_UNSUPPORTED, "backward: exponential-Euler only");
    if (!ssm::m1_bwd_supported(*p))
        return fail(SSM_ERR_UNSUPPORTED, "backward: dstate=%d (16, 32, 64 or 128 supported)", p->fwd.dstate);
    if (!ptrs) return SSM_OK;
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

ssm_status check_scan_bwd_overlap(const ssm_scan_bwd_params* p, const void* ws, size_t ws_bytes) {
    const ssm_scan_params* f = &p->fwd;
    const ScanSizes s(*f);
    const size_t g32 = static_cast<size_t>(f->batch) * f->dim * f->seqlen * 4;  // float32 [Bt, D, L]
    const size_t bc32 = static_cast<size_t>(f->batch) * f->ngroups * f->dstate * f->seqlen * 4;
    return check_disjoint(
        {{p->dx, g32, "dx"}, {p->ddelta, g32, "ddelta"}, {p->dz, g32, "dz"}, {p->dA, s.a, "dA"},
         {p->dB, bc32, "dB"}, {p->dC, bc32, "dC"}, {p->dD_skip, s.d, "dD_skip"},
         {p->ddelta_bias, s.d, "ddelta_bias"}, {p->dh0, s.h, "dh0"}, {ws, ws_bytes, "workspace"}},
        {{f->x, s.row, "x"}, {f->delta, s.row, "delta"}, {f->z, s.row, "z"}, {f->B, s.bc, "B"},
         {f->C, s.bc, "C"}, {f->A, s.a, "A"}, {f->D_skip, s.d, "D_skip"},
         {f->delta_bias, s.d, "delta_bias"}, {f->h0, s.h, "h0"}, {p->dy, s.y, "dy"},
         {p->dh_final, s.h, "dh_final"}});
}

ssm_status check_mamba3(const ssm_mamba3_params* p, bool ptrs) {
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
    if (!ptrs) return SSM_OK;
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
    const size_t bdl = static_cast<size_t>(p->batch) * p->dim * p->seqlen;
    const size_t row = bdl * esize(p->in_dtype), yb = bdl * esize(p->out_dtype);
    const size_t bc = static_cast<size_t>(p->batch) * p->ngroups * p->dstate * p->seqlen * esize(p->in_dtype);
    const size_t a = static_cast<size_t>(p->dim) * p->dstate * 4, d = static_cast<size_t>(p->dim) * 4;
    const size_t h = static_cast<size_t>(p->batch) * p->dim * p->dstate * 2 * 4;
    return check_disjoint({{p->y, yb, "y"}, {p->h_final, h, "h_final"}},
                          {{p->x, row, "x"}, {p->delta, row, "delta"}, {p->lam, row, "lam"},
                           {p->z, row, "z"}, {p->B, bc, "B"}, {p->C, bc, "C"}, {p->A_re, a, "A_re"},
                           {p->A_im, a, "A_im"}, {p->D_skip, d, "D_skip"},
                           {p->delta_bias, d, "delta_bias"}, {p->h0, h, "h0"}});
}

// scan: the recurrent form (batch, u, y, h0, h_final used); otherwise the kernel K
ssm_status check_s4d(const ssm_s4d_params* p, bool scan) {
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

struct S4dSizes {
    size_t u, y, dt, abc, h;
    explicit S4dSizes(const ssm_s4d_params& p) {
        const size_t bdl = static_cast<size_t>(p.batch) * p.dim * p.seqlen;
        u = bdl * esize(p.in_dtype);
        y = bdl * esize(p.out_dtype);
        dt = static_cast<size_t>(p.dim) * 4;
        abc = static_cast<size_t>(p.dim) * p.dstate * 2 * 4;
        h = static_cast<size_t>(p.batch) * p.dim * p.dstate * 2 * 4;
    }
};

ssm_status check_ssd(const ssd_params* p, bool ptrs) {
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
    if (!ptrs) return SSM_OK;
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

struct SsdSizes {
    size_t row, y, dt, bc, hd, h;
    explicit SsdSizes(const ssd_params& p) {
        const size_t blhp = static_cast<size_t>(p.batch) * p.seqlen * p.nheads * p.headdim;
        row = blhp * esize(p.in_dtype);
        y = blhp * esize(p.out_dtype);
        dt = static_cast<size_t>(p.batch) * p.seqlen * p.nheads * esize(p.in_dtype);
        bc = static_cast<size_t>(p.batch) * p.seqlen * p.ngroups * p.dstate * esize(p.in_dtype);
        hd = static_cast<size_t>(p.nheads) * 4;
        h = static_cast<size_t>(p.batch) * p.nheads * p.headdim * p.dstate * 4;
    }
};

ssm_status check_ssd_overlap(const ssd_params* p, const void* ws, size_t ws_bytes) {
    const SsdSizes s(*p);
    return check_disjoint({{p->y, s.y, "y"}, {p->h_final, s.h, "h_final"}, {ws, ws_bytes, "workspace"}},
                          {{p->x, s.row, "x"}, {p->z, s.row, "z"}, {p->dt, s.dt, "dt"},
                           {p->B, s.bc, "B"}, {p->C, s.bc, "C"}, {p->A, s.hd, "A"},
                           {p->D_skip, s.hd, "D_skip"}, {p->dt_bias, s.hd, "dt_bias"},
                           {p->h0, s.h, "h0"}});
}

ssm_status check_ssd_bwd(const ssd_bwd_params* p, bool ptrs) {
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
    if (!ptrs) return SSM_OK;
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

ssm_status check_ssd_bwd_overlap(const ssd_bwd_params* p, const void* ws, size_t ws_bytes) {
    const ssd_params* f = &p->fwd;
    const SsdSizes s(*f);
    const size_t blhp = static_cast<size_t>(f->batch) * f->seqlen * f->nheads * f->headdim;
    const size_t g32 = blhp * 4;
    const size_t dt32 = static_cast<size_t>(f->batch) * f->seqlen * f->nheads * 4;
    const size_t bc32 = static_cast<size_t>(f->batch) * f->seqlen * f->ngroups * f->dstate * 4;
    return check_disjoint(
        {{p->dx, g32, "dx"}, {p->ddt, dt32, "ddt"}, {p->dz, g32, "dz"}, {p->dA, s.hd, "dA"},
         {p->dB, bc32, "dB"}, {p->dC, bc32, "dC"}, {p->dD_skip, s.hd, "dD_skip"},
         {p->ddt_bias, s.hd, "ddt_bias"}, {p->dh0, s.h, "dh0"}, {ws, ws_bytes, "workspace"}},
        {{f->x, s.row, "x"}, {f->z, s.row, "z"}, {f->dt, s.dt, "dt"}, {f->B, s.bc, "B"},
         {f->C, s.bc, "C"}, {f->A, s.hd, "A"}, {f->D_skip, s.hd, "D_skip"},
         {f->dt_bias, s.hd, "dt_bias"}, {f->h0, s.h, "h0"},
         {p->dy, blhp * esize(f->out_dtype), "dy"}, {p->dh_final, s.h, "dh_final"}});
}

ssm_status check_step(const ssm_step_params* p, int ntokens) {
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
    REQUIRE(ntokens >= 1 && ntokens <= 256, "ntokens=%d (1..256)", ntokens);
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
    const size_t T = static_cast<size_t>(ntokens);
    const size_t bhp = static_cast<size_t>(p->batch) * p->nheads * p->headdim;
    const size_t row = T * bhp * esize(p->in_dtype), yb = T * bhp * esize(p->out_dtype);
    const size_t dt = T * p->batch * p->nheads * esize(p->in_dtype);
    const size_t bc = T * p->batch * p->ngroups * p->dstate * esize(p->in_dtype);
    const size_t a = static_cast<size_t>(p->nheads) * (p->a_per_state ? p->dstate : 1) * 4;
    const size_t hd = static_cast<size_t>(p->nheads) * 4;
    const size_t st = bhp * p->dstate * 4;
    // the state is read and written in place: it must only stay clear of the inputs and y
    return check_disjoint({{p->y, yb, "y"}, {p->state, st, "state"}},
                          {{p->x, row, "x"}, {p->z, row, "z"}, {p->dt, dt, "dt"}, {p->B, bc, "B"},
                           {p->C, bc, "C"}, {p->A, a, "A"}, {p->D_skip, hd, "D_skip"},
                           {p->dt_bias, hd, "dt_bias"}});
}

ssm::M1Args scan_args(const ssm_scan_params* p, const ssm_scan_opts* o) {
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
    a.kernel = o ? o->kernel : SSM_SCAN_KERNEL_AUTO;
    a.tpc = o ? o->threads_per_channel : 0;
    a.max_segments = o ? o->max_segments : 0;
    a.wait_limit = o ? o->wait_limit : 0;
    a.fault_test = o ? o->fault_test : 0;
    return a;
}

const char* kernel_name(int k) {
    switch (k) {
        case SSM_SCAN_KERNEL_TMEM: return "TMEM";
        case SSM_SCAN_KERNEL_TMA: return "TMA";
        case SSM_SCAN_KERNEL_TILED: return "TILED";
        case SSM_SCAN_KERNEL_GENERIC: return "GENERIC";
        default: return "AUTO";
    }
}

// The plan of the scan: the first of the TMEM, TMA, tiled and generic kernels that takes
// the problem and the options.
ssm_status plan_scan(const ssm::M1Args& a, ssm::M1Plan* plan) {
    cudaError_t e = ssm::m1_tmem_plan(a, plan);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd plan");
    if (plan->kind != ssm::M1Plan::kTmem) {
        if ((e = ssm::m1_tma_plan(a, plan)) != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd plan");
        if (plan->kind != ssm::M1Plan::kTma) {
            if (a.kernel == SSM_SCAN_KERNEL_GENERIC) {
                plan->kind = ssm::M1Plan::kGeneric;
            } else if ((e = ssm::m1_plan(a, plan)) != cudaSuccess) {
                return cuda_fail(e, "ssm_scan_fwd plan");
            }
        }
    }
    static const int kind_of[] = {SSM_SCAN_KERNEL_GENERIC, SSM_SCAN_KERNEL_TILED, SSM_SCAN_KERNEL_TMA,
                                  SSM_SCAN_KERNEL_TMEM};
    const int got = kind_of[plan->kind];
    if (a.kernel != SSM_SCAN_KERNEL_AUTO && a.kernel != got)
        return fail(SSM_ERR_UNSUPPORTED, "the %s kernel cannot run this problem with these options",
                    kernel_name(a.kernel));
    if (a.tpc != 0 && got == SSM_SCAN_KERNEL_GENERIC)
        return fail(SSM_ERR_UNSUPPORTED, "threads_per_channel=%d: no kernel that takes it runs this problem",
                    a.tpc);
    if (a.fault_test && (got != SSM_SCAN_KERNEL_TMEM || a.seqlen <= 64))
        return fail(SSM_ERR_UNSUPPORTED, "fault_test needs the TMEM kernel and at least two tiles");
    return SSM_OK;
}

size_t scan_workspace_bytes(const ssm::M1Plan& plan) {
    return plan.kind == ssm::M1Plan::kTmem ? plan.ws_bytes : 0;
}

ssm_status empty_sequence(float* h_final, const float* h0, size_t bytes, cudaStream_t s, const char* who) {
    if (h_final == nullptr) return SSM_OK;
    cudaError_t e = h0 ? cudaMemcpyAsync(h_final, h0, bytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h_final, 0, bytes, s);
    return e == cudaSuccess ? SSM_OK : cuda_fail(e, who);
}

ssm_status run_scan(const ssm_scan_params* p, const ssm_scan_opts* opts, void* workspace,
                    size_t workspace_bytes, void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_scan(p, true));
    RETURN_IF_FAILED(check_scan_opts(opts));
    RETURN_IF_FAILED(check_scan_overlap(p, nullptr, 0));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->seqlen == 0)
        return empty_sequence(p->h_final, p->h0, ScanSizes(*p).h, s, "ssm_scan_fwd (empty sequence)");
    ssm::M1Args a = scan_args(p, opts);
    ssm::M1Plan plan;
    RETURN_IF_FAILED(plan_scan(a, &plan));
    const size_t need = scan_workspace_bytes(plan);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    if (need > 0) RETURN_IF_FAILED(check_scan_overlap(p, workspace, need));
    cudaError_t e;
    switch (plan.kind) {
        case ssm::M1Plan::kTmem: e = ssm::m1_tmem_launch(a, plan, workspace, s); break;
        case ssm::M1Plan::kTma: e = ssm::m1_tma_launch(a, plan, s); break;
        default: e = ssm::m1_launch(a, plan, s); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
    return SSM_OK;
}

ssm::SsdArgs ssd_args(const ssd_params* p, void* workspace) {
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

ssm_status state_update(const ssm_step_params* p, int ntokens, void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_step(p, ntokens));
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

}  // namespace

namespace ssm {
ssm_status set_error(ssm_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace ssm

extern "C" {

int ssm_abi_version(void) { return SSM_ABI_VERSION; }

const char* ssm_last_error(void) { return g_err; }

ssm_status ssm_device_status(void) {
    g_err[0] = '\0';
    unsigned int n[3] = {0, 0, 0};
    cudaError_t e = ssm::m1_tma_take_wait_timeouts(&n[0]);
    if (e == cudaSuccess) e = ssm::m1_tmem_take_wait_timeouts(&n[1]);
    if (e == cudaSuccess) e = ssm::ssd_tc_take_wait_timeouts(&n[2]);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_device_status");
    if (n[0] + n[1] + n[2] == 0) return SSM_OK;
    return fail(SSM_ERR_TIMEOUT,
                "bounded device-side waits gave up since the last check (Mamba-1 TMA kernel: %u, "
                "Mamba-1 TMEM kernel: %u, SSD tensor-core kernels: %u); the outputs of the calls "
                "launched in between are not valid",
                n[0], n[1], n[2]);
}

unsigned int ssm_wait_timeouts(void) {
    unsigned int n[3] = {0, 0, 0};
    if (ssm::m1_tma_take_wait_timeouts(&n[0]) != cudaSuccess) return 0;
    if (ssm::m1_tmem_take_wait_timeouts(&n[1]) != cudaSuccess) return 0;
    if (ssm::ssd_tc_take_wait_timeouts(&n[2]) != cudaSuccess) return 0;
    return n[0] + n[1] + n[2];
}

ssm_status ssm_scan_fwd(const ssm_scan_params* p, void* stream) {
    ssm_scan_opts o;
    memset(&o, 0, sizeof(o));
    o.max_segments = 1;  // no time split: no scratch
    return run_scan(p, &o, nullptr, 0, stream);
}

ssm_status ssm_scan_fwd_ex(const ssm_scan_params* p, const ssm_scan_opts* opts, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return run_scan(p, opts, workspace, workspace_bytes, stream);
}

size_t ssm_scan_workspace_size(const ssm_scan_params* p, const ssm_scan_opts* opts) {
    if (check_scan(p, false) != SSM_OK || check_scan_opts(opts) != SSM_OK || p->seqlen == 0) return 0;
    ssm::M1Plan plan;
    if (plan_scan(scan_args(p, opts), &plan) != SSM_OK) return 0;
    return scan_workspace_bytes(plan);
}

size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p) {
    if (check_scan_bwd(p, false) != SSM_OK) return 0;
    return ssm::m1_bwd_workspace_size(*p);
}

ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_scan_bwd(p, true));
    const size_t need = ssm::m1_bwd_workspace_size(*p);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    RETURN_IF_FAILED(check_scan_bwd_overlap(p, workspace, need));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::m1_bwd_launch(*p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_bwd launch");
    return SSM_OK;
}

size_t ssm_mamba3_scan_workspace_size(const ssm_mamba3_params* p) {
    if (check_mamba3(p, false) != SSM_OK) return 0;
    return ssm::m3_workspace_size(*p);
}

ssm_status ssm_mamba3_scan_fwd(const ssm_mamba3_params* p, void* workspace, size_t workspace_bytes,
                               void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_mamba3(p, true));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t need = p->seqlen == 0 ? 0 : ssm::m3_workspace_size(*p);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    if (need > 0) {
        const size_t bdl = static_cast<size_t>(p->batch) * p->dim * p->seqlen;
        RETURN_IF_FAILED(check_disjoint(
            {{workspace, need, "workspace"}},
            {{p->x, bdl * esize(p->in_dtype), "x"}, {p->delta, bdl * esize(p->in_dtype), "delta"},
             {p->lam, bdl * esize(p->in_dtype), "lam"}, {p->y, bdl * esize(p->out_dtype), "y"}}));
    }
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    if (p->seqlen == 0)
        return empty_sequence(p->h_final, p->h0, static_cast<size_t>(p->batch) * p->dim * p->dstate * 2 * 4,
                              s, "ssm_mamba3_scan_fwd (empty sequence)");
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
    RETURN_IF_FAILED(check_s4d(p, true));
    const size_t need = ssm::s4d_workspace_size(*p);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    const S4dSizes s(*p);
    RETURN_IF_FAILED(check_disjoint({{p->y, s.y, "y"}, {p->h_final, s.h, "h_final"}, {workspace, need, "workspace"}},
                                    {{p->u, s.u, "u"}, {p->log_dt, s.dt, "log_dt"}, {p->A, s.abc, "A"},
                                     {p->B, s.abc, "B"}, {p->C, s.abc, "C"}, {p->D_skip, s.dt, "D_skip"},
                                     {p->h0, s.h, "h0"}}));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p->seqlen == 0) return empty_sequence(p->h_final, p->h0, s.h, st, "ssm_s4d_scan_fwd (empty sequence)");
    cudaError_t e = ssm::s4d_launch(*p, workspace, st);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_scan_fwd launch");
    return SSM_OK;
}

ssm_status ssm_s4d_kernel(const ssm_s4d_params* p, float* K, int kernel_len, void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_s4d(p, false));
    REQUIRE(kernel_len >= 0, "kernel_len=%d", kernel_len);
    if (p->dim > 65535) return fail(SSM_ERR_UNSUPPORTED, "s4d kernel: dim=%d > 65535", p->dim);
    if (kernel_len > 0) REQUIRE_PTR(K, "K");
    const size_t abc = static_cast<size_t>(p->dim) * p->dstate * 2 * 4;
    RETURN_IF_FAILED(check_disjoint({{K, static_cast<size_t>(p->dim) * kernel_len * 4, "K"}},
                                    {{p->log_dt, static_cast<size_t>(p->dim) * 4, "log_dt"},
                                     {p->A, abc, "A"}, {p->B, abc, "B"}, {p->C, abc, "C"}}));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::s4d_kernel_launch(*p, K, kernel_len, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_kernel launch");
    return SSM_OK;
}

size_t ssm_s4d_conv_workspace_size(const ssm_s4d_params* p) {
    if (p == nullptr || p->batch < 1 || p->dim < 1 || p->dim > 65535 || p->seqlen < 1) return 0;
    return ssm::s4d_conv_workspace_size(*p);
}

ssm_status ssm_s4d_conv_fwd(const ssm_s4d_params* p, void* workspace, size_t workspace_bytes,
                            void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_s4d(p, true));
    REQUIRE(p->h0 == nullptr && p->h_final == nullptr,
            "the convolution form starts from a zero state and gives no final state: h0 and "
            "h_final must be NULL (use ssm_s4d_scan_fwd for either)");
    if (p->dim > 65535) return fail(SSM_ERR_UNSUPPORTED, "s4d convolution: dim=%d > 65535", p->dim);
    if (p->seqlen > 0 && !ssm::s4d_conv_supported(*p))
        return fail(SSM_ERR_UNSUPPORTED, "s4d convolution: seqlen=%d > 8192 (the FFT of length "
                    "2^ceil(log2 2L) must fit in shared memory; use ssm_s4d_scan_fwd)", p->seqlen);
    const size_t need = p->seqlen > 0 ? ssm::s4d_conv_workspace_size(*p) : 0;
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    const S4dSizes s(*p);
    RETURN_IF_FAILED(check_disjoint({{p->y, s.y, "y"}, {workspace, need, "workspace"}},
                                    {{p->u, s.u, "u"}, {p->log_dt, s.dt, "log_dt"}, {p->A, s.abc, "A"},
                                     {p->B, s.abc, "B"}, {p->C, s.abc, "C"}, {p->D_skip, s.dt, "D_skip"}}));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    if (p->seqlen == 0) return SSM_OK;
    cudaError_t e = ssm::s4d_conv_launch(*p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_s4d_conv_fwd launch");
    return SSM_OK;
}

size_t ssd_chunk_scan_workspace_size(const ssd_params* p) {
    if (check_ssd(p, false) != SSM_OK) return 0;
    return ssm::ssd_workspace_bytes(ssd_args(p, nullptr));
}

ssm_status ssd_chunk_scan_fwd(const ssd_params* p, void* workspace, size_t workspace_bytes,
                              void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_ssd(p, true));
    ssm::SsdArgs a = ssd_args(p, workspace);
    const size_t need = ssm::ssd_workspace_bytes(a);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    RETURN_IF_FAILED(check_ssd_overlap(p, workspace, need));
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

size_t ssd_scan_bwd_workspace_size(const ssd_bwd_params* p) {
    if (check_ssd_bwd(p, false) != SSM_OK) return 0;
    return ssm::ssd_bwd_workspace_size(*p);
}

ssm_status ssd_scan_bwd(const ssd_bwd_params* p, void* workspace, size_t workspace_bytes,
                        void* stream) {
    g_err[0] = '\0';
    RETURN_IF_FAILED(check_ssd_bwd(p, true));
    const size_t need = ssm::ssd_bwd_workspace_size(*p);
    RETURN_IF_FAILED(check_workspace(workspace, workspace_bytes, need));
    RETURN_IF_FAILED(check_ssd_bwd_overlap(p, workspace, need));
    if (injected_launch_fault()) return fail(SSM_ERR_CUDA, "injected launch fault");
    cudaError_t e = ssm::ssd_bwd_launch(*p, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_bwd launch");
    return SSM_OK;
}

ssm_status ssm_state_update(const ssm_step_params* p, void* stream) {
    return state_update(p, 1, stream);
}

ssm_status ssm_state_update_tokens(const ssm_step_params* p, int ntokens, void* stream) {
    return state_update(p, ntokens, stream);
}

}  // extern "C"
