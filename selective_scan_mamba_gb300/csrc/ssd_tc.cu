// ssd_tc.cu -- Mamba-2 chunked SSD scan on the 5th-generation tensor cores (sm_103a).
//
// ("From S4 to Mamba-3", 03/System, mamba2_minimal.py: with a scalar A per head the
// recurrence is computed as chunked decayed-attention matmuls with a carried (N, P)
// state; 04/Approach: it equals the sequential scan.)  For a chunk of Q = 64 steps and
// s_t = running sum of Delta*A_h inside the chunk:
//   Y_diag[t,p] = sum_{s<=t} (C_t . B_s) exp(s_t - s_s) w_s x_s[p]          (decayed attention)
//   Y_off[t,p]  = exp(s_t) sum_n C_t[n] h_in[p,n]                           (carried state)
//   S[n,p]      = sum_s B_s[n] exp(s_end - s_s) w_s x_s[p]                  (chunk state)
//   h_out       = exp(s_end) h_in + S^T,   y = Y_diag + Y_off + D x, gated.
//
// Three launches.
//  1. prep: per (batch, head, chunk) the running sums s_t (in log2 units) and the input
//     weights w_t (Delta, or Delta*phi1 for ZOH) from the raw time steps, into the
//     workspace (512 bytes per chunk, copied next to the chunk's tiles later).
//  2. cuts: the (batch, head, chunk) units, taken head-major, are cut into one contiguous,
//     equal range per SM.  For every range that stops inside a sequence, the local end
//     state (from zero) over its chunks of that sequence, B^T (f o X) with
//     f_s = exp(s_range_end - s_s) w_s accumulated in TMEM, and its total decay; these
//     cut chunks are dealt out to the CTAs in equal shares (pieces), two chunks a step.
//  3. main: each CTA walks its range in order with the state in fp32 registers; where the
//     range starts inside a sequence the state there is h0 folded through the pieces of
//     the cuts before it.  Per chunk, TMA brings x, B, C (bf16, 128-byte swizzle, 3-stage ring)
//     and the step quantities; one warp issues tcgen05.mma (kind::f16, bf16 in, fp32
//     accumulators in TMEM):
//   MMA1  CB = C . B^T                        M=64  N=64 K=128  C, B K-major (exact bf16)
//   MMA2  Yd = M_hi . X + M_lo . X            M=64  N=64 K=64   M = CB o decay o w split
//                                                               into two bf16 parts; X
//                                                               MN-major
//   MMA3  Yo = C . H^T                        M=64  N=64 K=128  state rounded to bf16, held
//                                                               as [n][p] (MN-major); the
//                                                               exp(s_t) row scale is
//                                                               applied in fp32 afterwards
//   MMA4  S  = B^T . [F_hi | F_lo]            M=128 N=128 K=64  B MN-major; F = f o X,
//                                                               f_s = exp(s_end - s_s) w_s,
//                                                               split into two bf16 parts
//                                                               side by side along N
// Warp roles (18 warps): 16 compute warps build M and F of chunk c and then finish the
// outputs and the state update of chunk c-1.  Once chunk c is built, one warp issues
// MMA2 of chunk c and then MMA1 two chunks ahead, another issues MMA3 and MMA4 of chunk
// c and the TMA copies, so that the two issue streams run on different SM sub-partitions.
// Hand-offs go through mbarriers; the MMAs of chunk c run while the compute warps build
// chunk c+1.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kQ = 64, kP = 64, kNs = 128;
constexpr int kCompute = 16;                   // warps that build operands and finish outputs
constexpr int kMmaWarp = kCompute;             // issues the tensor-core MMAs
constexpr int kLoadWarp = kCompute + 1;        // issues the TMA copies
constexpr int kThreads = (kCompute + 2) * 32;

// main launch TMEM columns: two CB slots, Y_diag, Y_off, S (high then low part)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColCB = 0, kColYd = 128, kColYo = 192, kColS = 256;

// descriptor advanced by `bytes` along its start address (the address field holds
// address >> 4 in its low 14 bits; shared-memory addresses stay below 2^18)
__device__ __forceinline__ uint64_t dadv(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

struct SsdMaps {
    CUtensorMap x, b, c;
};

// per-chunk step quantities, written by the prep launch
struct ChunkArr {
    float cum2[kQ];  // running sum of Delta*A inside the chunk, log2 units (flat past the end)
    float w[kQ];     // input weight: Delta, or Delta*phi1(Delta*A) for ZOH (0 past the end)
};
constexpr int kArrBytes = static_cast<int>(sizeof(ChunkArr));  // 512

// main launch shared memory (bytes); tiles 1024-byte aligned, rows of 128 bytes
constexpr int kStages = 3;
constexpr int kStX = 0, kStB = 8192, kStC = 24576, kStArr = 40960;  // x [s][p], B, C [s][n]
constexpr int kStBytes = 41984;
constexpr int kOffM = kStages * kStBytes;  // 2 x [64 t][64 s] bf16 masked decayed CB, hi then lo
constexpr int kOffF = kOffM + 2 * 16384;   // 2 x [64 s][64 p] f_s x_s, hi then lo
constexpr int kOffHm = kOffF + 2 * 16384;  // [128 n][64 p] bf16 carried state
constexpr int kOffBar = kOffHm + 16384;
constexpr int kSmemBytes = kOffBar + 128;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // + alignment slack
constexpr uint32_t kTxMain = 40960 + kArrBytes;

// cuts launch: each step takes two chunks (128 steps of x and B, two chunks' step
// quantities); a ring of kCStages such stages and kCF F buffers (the F builders run up to
// kCF steps ahead of the MMAs)
constexpr int kCStages = 3;
constexpr int kCF = 2;
constexpr int kCRows = 2 * kQ;  // s rows per step
constexpr int kCStX = 0, kCStB = 16384, kCStArr = 49152, kCStBytes = 50176;  // x [s][p], B [s][n]
constexpr int kCFBytes = 32768;  // F_hi then F_lo, [128 s][64 p] each
constexpr int kCOffF = kCStages * kCStBytes;
constexpr int kCOffBar = kCOffF + kCF * kCFBytes;
constexpr int kCSmemBytes = kCOffBar + 192;
constexpr int kCSmemAlloc = kCSmemBytes + 1024;
constexpr uint32_t kTxCutTiles = 16384 + 32768;  // x and B of two chunks

// 16-byte chunk `cq` (8 bf16) of row `r` in a 128-byte-row swizzled tile
__device__ __forceinline__ int chunk_off(int r, int cq) { return r * 128 + (((cq ^ (r & 7))) << 4); }

// v = hi + lo with hi, lo bf16 (8 values -> two packed 16-byte chunks)
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        h[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        l[j] = pack_bf16x2(v[2 * j] - lo_bf16(h[j]), v[2 * j + 1] - hi_bf16(h[j]));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void unpack8(uint4 w, float* v) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = lo_bf16(a[j]);
        v[2 * j + 1] = hi_bf16(a[j]);
    }
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}
// contiguous bulk copy (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// first unit of range i when `total` units are cut into `nct` equal ranges
__host__ __device__ __forceinline__ long long range_begin(long long total, int nct, int i) {
    return total * i / nct;
}

// ---------------------------------------------------------------------------------------
// prep launch: one warp per (batch, head, chunk), two steps per lane
// ---------------------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(256) ssd_tc_prep(SsdArgs a, ChunkArr* out) {
    grid_dep_launch();  // the next launch may set itself up meanwhile
    const int L = a.seqlen, H = a.nheads;
    const int nch = (L + kQ - 1) / kQ;
    const long long units = static_cast<long long>(a.batch) * H * nch;
    const long long u = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (u >= units) return;
    const int lane = threadIdx.x & 31;
    const int c = static_cast<int>(u % nch);
    const int hd = static_cast<int>((u / nch) % H), b = static_cast<int>(u / (static_cast<long long>(nch) * H));
    const float Ah = a.A[hd];
    const float bias = a.dt_bias ? a.dt_bias[hd] : 0.f;
    const Tin* DT = static_cast<const Tin*>(a.dt);
    const int t0 = c * kQ, qv = min(kQ, L - t0);
    float d2[2], w2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int s = 2 * lane + j;
        float dt = 0.f;
        if (s < qv) {
            const float v = to_f32(DT[(static_cast<size_t>(b) * L + t0 + s) * H + hd]) + bias;
            dt = a.dt_softplus ? softplus_accurate(v) : v;
        }
        d2[j] = dt * Ah;
        w2[j] = a.disc == SSM_DISC_ZOH ? dt * phi1f(dt * Ah) : dt;
    }
    const float p1 = d2[0] + d2[1];
    float run = p1;  // inclusive prefix of the lane pairs
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, run, off);
        if (lane >= off) run += o;
    }
    const float excl = run - p1;
    ChunkArr& A = out[u];
    *reinterpret_cast<float2*>(&A.cum2[2 * lane]) =
        make_float2((excl + d2[0]) * SSM_LOG2E, (excl + p1) * SSM_LOG2E);
    *reinterpret_cast<float2*>(&A.w[2 * lane]) = make_float2(w2[0], w2[1]);
}

// ---------------------------------------------------------------------------------------
// Cuts.  Range i's cut is its chunks in its last sequence when that sequence goes on past
// the range end: the local end state (from zero) and the total decay of those chunks are
// what the next range of the sequence starts from.  The cut chunks of all ranges, cut
// after cut, are dealt out in equal contiguous shares to the cuts launch's CTAs (cuts are
// 0 to ~40 chunks long, so one CTA per cut would leave most SMs waiting for the longest).
// The share of one CTA inside one cut is a piece; folding a cut's pieces in time order,
// h = decay * h + S, gives the same state as the whole cut.
// ---------------------------------------------------------------------------------------
constexpr int kMaxRanges = 160;  // ranges (CTAs of the main launch) at most

// One piece: chunks [ca, ce) of sequence wk (= batch * nheads + head).  Its state and
// decay go to slot = its index in `piece`.
struct CutPiece {
    int wk, ca, ce;
};
// Built on the host (a few microseconds) and passed by value: no device set-up work.
struct CutPlan {
    int ncta;                          // CTAs of the cuts launch
    int cta_first[kMaxRanges + 1];     // pieces of CTA q: [cta_first[q], cta_first[q + 1])
    int cut_first[kMaxRanges + 1];     // pieces of range i's cut: [cut_first[i], cut_first[i + 1])
    CutPiece piece[2 * kMaxRanges];    // in time order within each cut, cut after cut
};
// the piece slots of the ranges, for the main launch
struct CutSlots {
    int cut_first[kMaxRanges + 1];
};

// Range i's cut: units [beg, beg + len), len = 0 when the range ends with its sequence.
void range_cut(long long total, int nct, int nch, int i, long long* beg, long long* len) {
    const long long u0 = range_begin(total, nct, i), u1 = range_begin(total, nct, i + 1);
    const long long ws = ((u1 - 1) / nch) * nch;
    *beg = u0 > ws ? u0 : ws;
    *len = (u1 <= u0 || u1 - ws == nch) ? 0 : u1 - *beg;
}

// The cut chunks of all ranges, cut after cut, form one list of T chunks; CTA q of the
// cuts launch takes [q T / n, (q + 1) T / n) of it, n = min(nct, T), so no share is empty.
// Returns the number of pieces (0: no cuts).
int build_cut_plan(long long total, int nct, int nch, CutPlan* P) {
    long long T = 0, beg, len;
    for (int i = 0; i < nct; ++i) {
        range_cut(total, nct, nch, i, &beg, &len);
        T += len;
    }
    const int n = static_cast<int>(T < nct ? T : nct);
    P->ncta = n;
    int np = 0, next_q = 0;
    long long F = 0;  // flat position of the cut's first chunk
    for (int i = 0; i < nct; ++i) {
        P->cut_first[i] = np;
        range_cut(total, nct, nch, i, &beg, &len);
        if (len == 0) continue;
        const long long wk = beg / nch, off = beg - wk * nch;
        // CTA of flat position f: the q with floor(q T / n) <= f < floor((q + 1) T / n)
        const int qa = static_cast<int>(((F + 1) * n - 1) / T), qb = static_cast<int>(((F + len) * n - 1) / T);
        for (int q = qa; q <= qb; ++q) {
            const long long fa = static_cast<long long>(q) * T / n, fb = static_cast<long long>(q + 1) * T / n;
            const long long lo = (fa > F ? fa : F) - F, hi = (fb < F + len ? fb : F + len) - F;
            while (next_q <= q) P->cta_first[next_q++] = np;
            P->piece[np++] = CutPiece{static_cast<int>(wk), static_cast<int>(off + lo), static_cast<int>(off + hi)};
        }
        F += len;
    }
    P->cut_first[nct] = np;
    while (next_q <= n) P->cta_first[next_q++] = np;
    return np;
}

// cuts launch: each CTA walks its pieces, each piece last chunk to first, two chunks per
// step (hi = the later, lo = the one before it; a piece of odd length ends with a step
// whose lo half lies outside the piece and is built as zeros), accumulating B^T (f x) in
// TMEM with K = 128 per step.  Warps 0-15 build F and read each piece's state out, warp
// 16 issues the MMAs, warp 17 the copies.  Steps run on over the pieces, so the copy ring
// and the F buffers stay full across piece boundaries.
struct CutSteps {  // the step sequence of one CTA: piece p, its local step j
    const CutPiece* pieces;
    int p = 0, j = 0;
    __device__ int steps_of(int q) const { return (pieces[q].ce - pieces[q].ca + 1) >> 1; }
    __device__ void next() {
        if (++j == steps_of(p)) {
            ++p;
            j = 0;
        }
    }
    __device__ int hi() const { return pieces[p].ce - 1 - 2 * j; }  // chunk of the later half
    __device__ bool lo_ok() const { return hi() - 1 >= pieces[p].ca; }
};

__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_cuts(const __grid_constant__ SsdMaps maps, SsdArgs a, const __grid_constant__ CutPlan plan,
                const ChunkArr* arrs, float* cut_state, float* cut_decay) {
    const int L = a.seqlen, H = a.nheads;
    const int nch = (L + kQ - 1) / kQ;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + kCOffBar);  // [kCStages]
    uint64_t* mma_bar = tma_bar + kCStages;  // [kCF] MMA of step k done (k % kCF)
    uint64_t* done_bar = mma_bar + kCF;      // [4] F of step k built (k % 4): builders stay
                                             // within 3 steps of each other
    uint64_t* free_bar = done_bar + 4;       // [kCStages] the stage's MMA done (its reuse)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(free_bar + kCStages);
    uint64_t* drain_bar = free_bar + kCStages + 1;  // after an abort: the issued MMAs are done

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    grid_dep_launch();
    if (warp == 0) tc::tmem_alloc(tslot, 128);
    if (tid == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.b);
        for (int s = 0; s < kCStages; ++s) mbar_init(&tma_bar[s], 1);
        for (int j = 0; j < kCF; ++j) mbar_init(&mma_bar[j], 1);
        for (int j = 0; j < 4; ++j) mbar_init(&done_bar[j], kCompute);
        for (int j = 0; j < kCStages; ++j) mbar_init(&free_bar[j], 1);
        mbar_init(drain_bar, 1);
        mbar_fence_init();
        wait_setup(0);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    grid_dep_wait();  // the step quantities written by the launch before
    const uint32_t tmem = *tslot;
    // this CTA's pieces [p0, p1), walked one after another: nsteps steps in all
    const int p0 = plan.cta_first[blockIdx.x], p1 = plan.cta_first[blockIdx.x + 1];
    CutSteps walk{plan.piece, p0, 0};
    int nsteps = 0;
    for (int p = p0; p < p1; ++p) nsteps += walk.steps_of(p);

    int last_issued = -1;  // load warp, lane 0: the last step whose copy went out
    bool live = true;      // MMA warp: no wait has failed yet
    if (warp == kLoadWarp) {
        if (lane == 0) {
            for (int k = 0; k < nsteps; ++k, walk.next()) {
                // step k reuses the stage of step k - kCStages once that step's MMA is done
                if (k >= kCStages && !mbar_wait_lane(&free_bar[k % kCStages], ((k - kCStages) / kCStages) & 1))
                    break;
                last_issued = k;
                const int wk = plan.piece[walk.p].wk, hi = walk.hi();
                const bool lo_ok = walk.lo_ok();
                const int b = wk / H, hd = wk % H, g = hd / (H / a.ngroups);
                unsigned char* st = sm + (k % kCStages) * kCStBytes;
                uint64_t* bar = &tma_bar[k % kCStages];
                mbar_arrive_expect_tx(bar, kTxCutTiles + (lo_ok ? 2 : 1) * kArrBytes);
                // rows (hi - 1) * 64 .. hi * 64 + 63; before the sequence start (hi = 0)
                // the copy reads zeros
                tma_load_4d(st + kCStX, &maps.x, 0, hd, (hi - 1) * kQ, b, bar);
                tma_load_4d(st + kCStB, &maps.b, 0, g, (hi - 1) * kQ, b, bar);
                tma_load_4d(st + kCStB + 16384, &maps.b, 64, g, (hi - 1) * kQ, b, bar);
                const ChunkArr* ar = arrs + static_cast<size_t>(wk) * nch;
                if (lo_ok) bulk_load(st + kCStArr, ar + hi - 1, kArrBytes, bar);
                bulk_load(st + kCStArr + kArrBytes, ar + hi, kArrBytes, bar);
            }
        }
    } else if (warp == kMmaWarp) {
        for (int k = 0; k < nsteps; ++k, walk.next()) {
            const bool built = mbar_wait_warp_ok(&done_bar[k & 3], (k >> 2) & 1);
            const bool landed = mbar_wait_warp_ok(&tma_bar[k % kCStages], (k / kCStages) & 1);
            tc::fence_after();
            live = built && landed && live;
            if (!live) continue;  // the CTA has aborted: issue nothing more
            const unsigned char* st = sm + (k % kCStages) * kCStBytes;
            const uint32_t sbm = smem_u32(st + kCStB);
            const uint32_t sf = smem_u32(sm + kCOffF + (k % kCF) * kCFBytes);
            // S[n][p_hi | p_lo] += B^T [F_hi | F_lo]: N = 128 over the two adjacent parts,
            // K = 128 over the two chunks; a piece's first step starts the accumulator afresh
            const uint32_t id4 = tc::idesc_bf16_mn(128, 128, true, true);
            const uint64_t dB = tc::desc_sw128_mn(sbm, 16384), dF = tc::desc_sw128_mn(sf, 16384);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_warp(tmem, dadv(dB, kk * 2048), dadv(dF, kk * 2048), id4,
                                  (walk.j > 0 || kk > 0) ? 1u : 0u);
            tc::mma_commit_warp(&mma_bar[k % kCF]);
            tc::mma_commit_warp(&free_bar[k % kCStages]);
            __syncwarp();
        }
    } else {
        const int fs = tid >> 2, fp = (tid & 3) * 16;  // F elements (s, p..p+15), s over both chunks
        const bool in_hi = fs >= kQ;                   // row of the later chunk
        const int s_in = fs & (kQ - 1);
        const int q4 = warp & 3, cg = warp >> 2;
        const int hn = 32 * q4 + lane, hp = 16 * cg;
        float tailf = 1.f;  // decay of the piece's chunks already walked (later in time)
        for (int k = 0; k < nsteps; ++k) {
            if (k >= kCF) {  // MMA of step k-kCF done: its F buffer is free
                mbar_wait_warp(&mma_bar[k % kCF], (k / kCF - 1) & 1);
                tc::fence_after();
            }
            mbar_wait_warp(&tma_bar[k % kCStages], (k / kCStages) & 1);
            const unsigned char* st = sm + (k % kCStages) * kCStBytes;
            const ChunkArr& Ah = *reinterpret_cast<const ChunkArr*>(st + kCStArr + kArrBytes);
            const ChunkArr& Al = *reinterpret_cast<const ChunkArr*>(st + kCStArr);
            const bool lo_ok = walk.lo_ok();
            const float dec_hi = ex2_approx(Ah.cum2[kQ - 1]);
            // f_s = exp(s_end - s_s) w_s relative to the end of the piece's later chunks
            float f;
            if (in_hi) {
                f = tailf * ex2_approx(Ah.cum2[kQ - 1] - Ah.cum2[s_in]) * Ah.w[s_in];
            } else {
                f = lo_ok ? tailf * dec_hi * ex2_approx(Al.cum2[kQ - 1] - Al.cum2[s_in]) * Al.w[s_in] : 0.f;
            }
            tailf *= lo_ok ? dec_hi * ex2_approx(Al.cum2[kQ - 1]) : dec_hi;
            unsigned char* F = sm + kCOffF + (k % kCF) * kCFBytes;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
                if (in_hi || lo_ok) {  // outside the piece: zeros, whatever x holds there
                    float v[8];
                    unpack8(*reinterpret_cast<const uint4*>(st + kCStX + chunk_off(fs, (fp >> 3) + q)), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] *= f;
                    split8(v, hi, lo);
                }
                *reinterpret_cast<uint4*>(F + chunk_off(fs, (fp >> 3) + q)) = hi;
                *reinterpret_cast<uint4*>(F + 16384 + chunk_off(fs, (fp >> 3) + q)) = lo;
            }
            tc::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&done_bar[k & 3]);
            if (walk.j + 1 == walk.steps_of(walk.p)) {
                // the piece's last step: once its MMA is done, read the state out (the next
                // piece's first MMA waits for F built after this read)
                mbar_wait_warp(&mma_bar[k % kCF], (k / kCF) & 1);
                tc::fence_after();
                uint32_t r[16], r2[16];
                tc::tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + hp, r);
                tc::tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 + hp, r2);
                tc::tmem_wait();
                tc::fence_before();
                const int slot = walk.p;
                float* dst = cut_state + static_cast<size_t>(slot) * kP * kNs;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    dst[static_cast<size_t>(hp + j) * kNs + hn] = __uint_as_float(r[j]) + __uint_as_float(r2[j]);
                if (tid == 0) cut_decay[slot] = tailf;
                tailf = 1.f;
            }
            walk.next();
        }
    }
    // a CTA whose waits gave up lets its copies and MMAs in flight finish before the
    // shared and tensor memory they write is released
    if (warp == kLoadWarp && lane == 0 && wait_aborted()) drain_ring(tma_bar, kCStages, last_issued);
    if (warp == kMmaWarp && wait_aborted_warp()) {
        tc::mma_commit_warp(drain_bar);  // the issuing lane's MMAs
        if (lane == 0) mbar_drain(drain_bar, 0);
        __syncwarp();
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------------------
// main launch
// ---------------------------------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_main(const __grid_constant__ SsdMaps maps, SsdArgs a, int nct, const __grid_constant__ CutSlots slots,
                const ChunkArr* arrs, const float* cut_state, const float* cut_decay) {
    const int L = a.seqlen, H = a.nheads;
    const int nch = (L + kQ - 1) / kQ;
    const long long total = static_cast<long long>(a.batch) * H * nch;
    const int ci = blockIdx.x;
    const long long u0 = range_begin(total, nct, ci), u1 = range_begin(total, nct, ci + 1);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + kOffBar);  // [kStages]
    uint64_t* bar_a = tma_bar + kStages;  // [2] MMA1 (C B^T) of a chunk done, by chunk parity
    uint64_t* bar_b = bar_a + 2;          // MMA2-4 of a chunk done
    uint64_t* done_bar = bar_b + 1;       // [2] the compute warps finished a step
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done_bar + 2);
    uint64_t* drain_bar = done_bar + 3;   // [2] after an abort: each issuing warp's MMAs done

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (tid == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.b);
        prefetch_tmap(&maps.c);
        for (int s = 0; s < kStages; ++s) mbar_init(&tma_bar[s], 1);
        for (int j = 0; j < 2; ++j) {
            mbar_init(&bar_a[j], 1);
            mbar_init(&done_bar[j], kCompute);
        }
        mbar_init(bar_b, 2);  // one commit from each of the two issuing warps
        mbar_init(&drain_bar[0], 1);
        mbar_init(&drain_bar[1], 1);
        mbar_fence_init();
        wait_setup(0);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    grid_dep_wait();  // the step quantities and cut states of the launches before
    const uint32_t tmem = *tslot;
    const Tin* Z = static_cast<const Tin*>(a.z);
    const size_t PN = static_cast<size_t>(kP) * kNs;

    // Running chunk number G over the CTA's ranges: stage G % 3, CB slot and M/F buffers
    // G & 1, bar_a[G & 1] with parity (G >> 1) & 1.  Steps (n + 1 per range) alternate
    // between the two done barriers, so that no waiter can fall two phases behind.
    uint32_t gseq = 0, dstep = 0, b_seq = 0;
    long long last_g = -1;  // load warp, lane 0: running number of the last chunk copied
    bool live = true;       // issuing warps: no wait has failed yet

    for (long long u = u0; u < u1;) {
        const int wk = static_cast<int>(u / nch);
        const int c0 = static_cast<int>(u % nch);
        const int n = static_cast<int>(min(static_cast<long long>(nch - c0), u1 - u));
        const int b = wk / H, hd = wk % H, g = hd / (H / a.ngroups);
        const size_t bh = static_cast<size_t>(b) * H + hd;
        const uint32_t G0 = gseq;
        auto stage_of = [&](int k) { return sm + ((G0 + k) % kStages) * kStBytes; };
        auto tma_bar_of = [&](int k) { return &tma_bar[(G0 + k) % kStages]; };
        auto tma_par = [&](int k) { return ((G0 + k) / kStages) & 1; };

        if (warp == kLoadWarp) {
            auto issue = [&](int k) {  // chunk c0 + k
                last_g = static_cast<long long>(G0) + k;
                const int c = c0 + k;
                unsigned char* st = stage_of(k);
                uint64_t* bar = tma_bar_of(k);
                mbar_arrive_expect_tx(bar, kTxMain);
                tma_load_4d(st + kStX, &maps.x, 0, hd, c * kQ, b, bar);
                tma_load_4d(st + kStB, &maps.b, 0, g, c * kQ, b, bar);
                tma_load_4d(st + kStB + 8192, &maps.b, 64, g, c * kQ, b, bar);
                tma_load_4d(st + kStC, &maps.c, 0, g, c * kQ, b, bar);
                tma_load_4d(st + kStC + 8192, &maps.c, 64, g, c * kQ, b, bar);
                bulk_load(st + kStArr, arrs + static_cast<size_t>(wk) * nch + c, kArrBytes, bar);
            };
            if (lane == 0)
                for (int k = 0; k < kStages && k < n; ++k) issue(k);
            const uint32_t id3 = tc::idesc_bf16_mn(64, 64, false, true);
            const uint32_t id4 = tc::idesc_bf16_mn(128, 128, true, true);
            const uint64_t dH = tc::desc_sw128_mn(smem_u32(sm + kOffHm), 16384);
            for (int k = 0; k <= n; ++k) {
                // once a wait has failed (the CTA aborted) this warp issues nothing more
                live = mbar_wait_warp_ok(&done_bar[dstep & 1], (dstep >> 1) & 1) && live;
                ++dstep;
                tc::fence_after();
                if (k < n && live) {  // MMA3 and MMA4 of chunk k (MMA2: the MMA warp)
                    const unsigned char* st = stage_of(k);
                    const uint64_t dC = tc::desc_sw128(smem_u32(st + kStC));
                    const uint64_t dB = tc::desc_sw128_mn(smem_u32(st + kStB), 8192);
                    const uint64_t dF = tc::desc_sw128_mn(smem_u32(sm + kOffF + ((G0 + k) & 1) * 16384), 8192);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // Yo = C H^T (K = 128 over n)
                        tc::mma_bf16_warp(tmem + kColYo, dadv(dC, (kk >> 2) * 8192 + (kk & 3) * 32),
                                          dadv(dH, kk * 2048), id3, kk > 0);
                        // S[n][p_hi | p_lo] = B^T [F_hi | F_lo] (N = 128, K = 64 over s)
                        if (kk < 4)
                            tc::mma_bf16_warp(tmem + kColS, dadv(dB, kk * 2048), dadv(dF, kk * 2048), id4, kk > 0);
                    }
                    tc::mma_commit_warp(bar_b);
                }
                __syncwarp();
                // the stage of chunk k-1 is free (its MMAs and outputs are done)
                if (lane == 0 && live && k >= 1 && k + 2 < n) issue(k + 2);
            }
        } else if (warp == kMmaWarp) {
            const uint32_t id1 = tc::idesc_bf16(64, 64), id2 = tc::idesc_bf16_mn(64, 64, false, true);
            auto mma1 = [&](int k) {  // CB of chunk k into its slot, then commit
                live = mbar_wait_warp_ok(tma_bar_of(k), tma_par(k)) && live;
                if (!live) return;
                const unsigned char* st = stage_of(k);
                const uint64_t dC = tc::desc_sw128(smem_u32(st + kStC)), dB = tc::desc_sw128(smem_u32(st + kStB));
                const uint32_t slot = tmem + kColCB + 64 * ((G0 + k) & 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    tc::mma_bf16_warp(slot, dadv(dC, off), dadv(dB, off), id1, kk > 0);
                }
                tc::mma_commit_warp(&bar_a[(G0 + k) & 1]);
            };
            mma1(0);
            if (n > 1) mma1(1);
            for (int k = 0; k <= n; ++k) {
                // the compute warps finished step k
                live = mbar_wait_warp_ok(&done_bar[dstep & 1], (dstep >> 1) & 1) && live;
                ++dstep;
                tc::fence_after();
                if (k < n && live) {  // MMA2 of chunk k: Yd = M_hi X + M_lo X
                    const unsigned char* st = stage_of(k);
                    const uint64_t dX = tc::desc_sw128_mn(smem_u32(st + kStX), 8192);
                    const uint64_t dM = tc::desc_sw128(smem_u32(sm + kOffM + ((G0 + k) & 1) * 16384));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_bf16_warp(tmem + kColYd, dadv(dM, (kk >> 2) * 8192 + (kk & 3) * 32),
                                          dadv(dX, (kk & 3) * 2048), id2, kk > 0);
                    tc::mma_commit_warp(bar_b);
                }
                __syncwarp();
                if (live && k + 2 < n) mma1(k + 2);  // its slot held CB of chunk k, read in step k
            }
        } else {
            const int q4 = warp & 3, cg = warp >> 2;
            const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q4) << 16);
            const int tr = 16 * q4 + (lane & 15);        // row t (M build, outputs)
            const int pc = 8 * cg + 32 * (lane >> 4);    // first of 8 columns (s in M, p in outputs)
            const int hn = 32 * q4 + lane, hp = 16 * cg;  // state row n, first of 16 columns p
            const int fs = tid >> 3, fp = (tid & 7) * 8;  // F element (s, p..p+7)
            const float Dh = a.D ? a.D[hd] : 0.f;

            // state at the start of the range in this sequence: h0, then the cuts before it
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) h[j] = a.h0 ? a.h0[bh * PN + static_cast<size_t>(hp + j) * kNs + hn] : 0.f;
            if (c0 > 0) {
                const long long ws = static_cast<long long>(wk) * nch;
                int j0 = ci - 1;
                while (j0 > 0 && range_begin(total, nct, j0) > ws) --j0;
                // the pieces of the cuts of ranges j0 .. ci-1, in time order
                for (int j = slots.cut_first[j0]; j < slots.cut_first[ci]; ++j) {
                    const float dec = cut_decay[j];
                    const float* cs = cut_state + static_cast<size_t>(j) * PN;
#pragma unroll
                    for (int i = 0; i < 16; ++i) h[i] = dec * h[i] + cs[static_cast<size_t>(hp + i) * kNs + hn];
                }
            }
            auto write_hm = [&]() {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    *reinterpret_cast<uint4*>(sm + kOffHm + chunk_off(hn, 2 * cg + j)) =
                        make_uint4(pack_bf16x2(h[8 * j], h[8 * j + 1]), pack_bf16x2(h[8 * j + 2], h[8 * j + 3]),
                                   pack_bf16x2(h[8 * j + 4], h[8 * j + 5]), pack_bf16x2(h[8 * j + 6], h[8 * j + 7]));
            };
            write_hm();

            for (int k = 0; k <= n; ++k) {
                if (k < n) {
                    const uint32_t G = G0 + k;
                    mbar_wait_warp(&bar_a[G & 1], (G >> 1) & 1);  // CB of chunk k is in its slot
                    tc::fence_after();
                    uint32_t r[8];
                    tc::tmem_ld_16x32bx2_x8(tlane + kColCB + 64 * (G & 1) + 8 * cg, r);
                    mbar_wait_warp(tma_bar_of(k), tma_par(k));
                    const unsigned char* st = stage_of(k);
                    const ChunkArr& A = *reinterpret_cast<const ChunkArr*>(st + kStArr);
                    unsigned char* Mb = sm + kOffM + (G & 1) * 16384;
                    unsigned char* Fb = sm + kOffF + (G & 1) * 16384;
                    const float cend = A.cum2[kQ - 1];
                    // (2) F[s][p] = f_s x_s[p] as bf16 hi + lo, f_s = exp(s_end - s_s) w_s
                    {
                        const float f = ex2_approx(cend - A.cum2[fs]) * A.w[fs];
                        float v[8];
                        unpack8(*reinterpret_cast<const uint4*>(st + kStX + chunk_off(fs, fp >> 3)), v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] *= f;
                        uint4 hi, lo;
                        split8(v, hi, lo);
                        *reinterpret_cast<uint4*>(Fb + chunk_off(fs, fp >> 3)) = hi;
                        *reinterpret_cast<uint4*>(Fb + 8192 + chunk_off(fs, fp >> 3)) = lo;
                    }
                    // (1) M[t][s] = CB[t][s] exp(s_t - s_s) w_s for s <= t, as bf16 hi + lo
                    {
                        const float ct = A.cum2[tr];
                        float csa[8], wsa[8];
                        *reinterpret_cast<float4*>(csa) = *reinterpret_cast<const float4*>(&A.cum2[pc]);
                        *reinterpret_cast<float4*>(csa + 4) = *reinterpret_cast<const float4*>(&A.cum2[pc + 4]);
                        *reinterpret_cast<float4*>(wsa) = *reinterpret_cast<const float4*>(&A.w[pc]);
                        *reinterpret_cast<float4*>(wsa + 4) = *reinterpret_cast<const float4*>(&A.w[pc + 4]);
                        tc::tmem_wait();
                        float m[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float v = __uint_as_float(r[e]) * ex2_approx(ct - csa[e]) * wsa[e];
                            m[e] = (pc + e <= tr) ? v : 0.f;
                        }
                        uint4 hi, lo;
                        split8(m, hi, lo);
                        *reinterpret_cast<uint4*>(Mb + chunk_off(tr, pc >> 3)) = hi;
                        *reinterpret_cast<uint4*>(Mb + 8192 + chunk_off(tr, pc >> 3)) = lo;
                    }
                }
                if (k > 0) {
                    const int kp = k - 1;
                    mbar_wait_warp(bar_b, b_seq & 1);  // Y_diag, Y_off and S of chunk k-1
                    ++b_seq;
                    tc::fence_after();
                    uint32_t sv[16], sl[16];
                    tc::tmem_ld_32x32b_x16(tlane + kColS + hp, sv);
                    tc::tmem_ld_32x32b_x16(tlane + kColS + 64 + hp, sl);
                    const unsigned char* st = stage_of(kp);
                    const ChunkArr& A = *reinterpret_cast<const ChunkArr*>(st + kStArr);
                    const float dec = ex2_approx(A.cum2[kQ - 1]);
                    tc::tmem_wait();
                    uint32_t yd[8], yo[8];  // in flight during the state update
                    tc::tmem_ld_16x32bx2_x8(tlane + kColYd + 8 * cg, yd);
                    tc::tmem_ld_16x32bx2_x8(tlane + kColYo + 8 * cg, yo);
                    // (4) state after chunk kp: row n = hn, columns p = hp .. hp + 15
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        h[j] = dec * h[j] + (__uint_as_float(sv[j]) + __uint_as_float(sl[j]));
                    write_hm();
                    const int t0 = (c0 + kp) * kQ;
                    const bool live = tr < L - t0;
                    float xv[8];
                    unpack8(*reinterpret_cast<const uint4*>(st + kStX + chunk_off(tr, pc >> 3)), xv);
                    const float et = ex2_approx(A.cum2[tr]);
                    const size_t row = ((static_cast<size_t>(b) * L + t0 + tr) * H + hd) * kP + pc;
                    float zv[8];
                    if (Z && live) unpack8(*reinterpret_cast<const uint4*>(Z + row), zv);
                    tc::tmem_wait();
                    // (3) outputs of chunk kp: row t = tr, columns p = pc .. pc + 7
                    if (live) {
                        float out[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float v = __uint_as_float(yd[e]) + et * __uint_as_float(yo[e]) + Dh * xv[e];
                            if (Z) v *= silu_accurate(zv[e]);
                            out[e] = v;
                        }
                        Tout* yp = static_cast<Tout*>(a.y) + row;
                        if constexpr (sizeof(Tout) == 2) {
                            *reinterpret_cast<uint4*>(yp) =
                                make_uint4(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]),
                                           pack_bf16x2(out[4], out[5]), pack_bf16x2(out[6], out[7]));
                        } else {
                            reinterpret_cast<float4*>(yp)[0] = make_float4(out[0], out[1], out[2], out[3]);
                            reinterpret_cast<float4*>(yp)[1] = make_float4(out[4], out[5], out[6], out[7]);
                        }
                    }
                }
                tc::fence_async_smem();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&done_bar[dstep & 1]);
                ++dstep;
            }
            if (c0 + n == nch && a.h_final) {
#pragma unroll
                for (int j = 0; j < 16; ++j) a.h_final[bh * PN + static_cast<size_t>(hp + j) * kNs + hn] = h[j];
            }
        }
        gseq += n;
        u += n;
    }
    // a CTA whose waits gave up lets its copies and MMAs in flight finish before the
    // shared and tensor memory they write is released
    if (warp == kLoadWarp || warp == kMmaWarp) {
        if (wait_aborted_warp()) {
            if (warp == kLoadWarp && lane == 0) drain_ring(tma_bar, kStages, last_g);
            uint64_t* db = &drain_bar[warp == kLoadWarp ? 0 : 1];
            tc::mma_commit_warp(db);  // the issuing lane's MMAs
            if (lane == 0) mbar_drain(db, 0);
            __syncwarp();
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

cudaError_t encode_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t d3, unsigned rows = kQ);

long long tc_units(const SsdArgs& a) {
    return static_cast<long long>(a.batch) * a.nheads * ((a.seqlen + kQ - 1) / kQ);
}

// one range per SM (fewer when there are fewer units)
int tc_ctas(long long total) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms > kMaxRanges) sms = kMaxRanges;
    return static_cast<int>(total < sms ? total : sms);
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// workspace: piece states [pieces][P][N] fp32, piece decays [pieces], step quantities
// [units]; nct ranges give at most 2 nct - 1 pieces
struct TcWorkspace {
    size_t off_decay, off_arr, bytes;
    TcWorkspace(int nct, long long units) {
        const size_t np = 2 * static_cast<size_t>(nct);
        off_decay = round256(np * kP * kNs * sizeof(float));
        off_arr = off_decay + round256(np * sizeof(float));
        bytes = off_arr + round256(static_cast<size_t>(units) * kArrBytes);
    }
};

}  // namespace

// The tensor-core path covers the Mamba-2 130m/780m layer shapes: headdim 64, dstate 128,
// bf16 inputs, chunk 64, 128 or 256; other shapes use the CUDA-core kernels in ssd.cu.
// Every chunk size runs on 64-step tiles.  For a chunk of 128 or 256 steps the
// decayed-attention block between two different tiles i > j of the chunk,
//   sum_{s in j} (C_t . B_s) exp(s_t - s_s) w_s x_s  (t in tile i),
// equals exp(s_t - s_{end of j}) C_t . (sum_{s in j} B_s exp(s_{end of j} - s_s) w_s x_s)
// carried forward to tile i: the chunk-state product regrouped, exact in real arithmetic.
bool ssd_tc_supported(const SsdArgs& a) {
    return a.chunk % kQ == 0 && a.headdim == kP && a.dstate == kNs && a.in_dtype == SSM_BF16 &&
           a.seqlen > 0;
}

size_t ssd_tc_workspace_bytes(const SsdArgs& a) {
    const long long units = tc_units(a);
    return TcWorkspace(tc_ctas(units), units).bytes;
}

cudaError_t ssd_tc_launch(const SsdArgs& a, void* workspace, cudaStream_t s) {
    const long long total = tc_units(a);
    const int nct = tc_ctas(total);
    const TcWorkspace wl(nct, total);
    SsdMaps maps;
    cudaError_t e;
    const uint64_t H = a.nheads, G = a.ngroups, L = a.seqlen, Bt = a.batch;
    if ((e = encode_4d(&maps.x, a.x, kP, H, L, Bt)) != cudaSuccess) return e;
    if ((e = encode_4d(&maps.b, a.B, kNs, G, L, Bt)) != cudaSuccess) return e;
    if ((e = encode_4d(&maps.c, a.C, kNs, G, L, Bt)) != cudaSuccess) return e;
    char* ws = static_cast<char*>(workspace);
    float* cut_state = reinterpret_cast<float*>(ws);
    float* cut_decay = reinterpret_cast<float*>(ws + wl.off_decay);
    ChunkArr* arrs = reinterpret_cast<ChunkArr*>(ws + wl.off_arr);
    ssd_tc_prep<bf16_t><<<static_cast<unsigned>((total + 7) / 8), 256, 0, s>>>(a, arrs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // a cut exists where a range boundary falls inside a sequence
    const int nch = (a.seqlen + kQ - 1) / kQ;
    CutPlan plan;
    CutSlots slots;
    if (build_cut_plan(total, nct, nch, &plan) > 0) {
        SsdMaps cmaps;  // 128-row boxes: two chunks per copy
        if ((e = encode_4d(&cmaps.x, a.x, kP, H, L, Bt, kCRows)) != cudaSuccess) return e;
        if ((e = encode_4d(&cmaps.b, a.B, kNs, G, L, Bt, kCRows)) != cudaSuccess) return e;
        cmaps.c = maps.c;  // (not read by the cuts launch)
        if ((e = set_smem_attr(reinterpret_cast<const void*>(ssd_tc_cuts), kCSmemAlloc)) != cudaSuccess)
            return e;
        if ((e = launch_dependent(ssd_tc_cuts, plan.ncta, kThreads, kCSmemAlloc, s, cmaps, a, plan, arrs, cut_state,
                                  cut_decay)) != cudaSuccess)
            return e;
    }
    for (int i = 0; i <= nct; ++i) slots.cut_first[i] = plan.cut_first[i];
    if (a.out_dtype == SSM_BF16) {
        auto k = ssd_tc_main<bf16_t, bf16_t>;
        if ((e = set_smem_attr(reinterpret_cast<const void*>(k), kSmemAlloc)) !=
            cudaSuccess)
            return e;
        e = launch_dependent(k, nct, kThreads, kSmemAlloc, s, maps, a, nct, slots, arrs, cut_state, cut_decay);
    } else {
        auto k = ssd_tc_main<bf16_t, float>;
        if ((e = set_smem_attr(reinterpret_cast<const void*>(k), kSmemAlloc)) !=
            cudaSuccess)
            return e;
        e = launch_dependent(k, nct, kThreads, kSmemAlloc, s, maps, a, nct, slots, arrs, cut_state, cut_decay);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t ssd_tc_take_wait_timeouts(unsigned int* count) {
    return take_wait_timeouts(count);
}

namespace {
cudaError_t encode_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t d3, unsigned rows) {
    // [d3][d2][d1][d0] bf16, box {64, 1, rows, 1}, 128-byte swizzle
    const unsigned long long dims[4] = {d0, d1, d2, d3};
    const unsigned box[4] = {64, 1, rows, 1};
    return encode_tmap_nd(map, base, 2, 4, dims, box, true);
}
}  // namespace

}  // namespace ssm
