// Fused MaxSim forward for sm_103a: TMA -> tcgen05.mma -> TMEM -> fused
// running max / argmax / sum epilogue. The [query rows, document tokens]
// similarity tile exists only in tensor memory and registers.
//
// Work decomposition (one persistent CTA per SM):
//  * Query rows are flattened: row r = i * lq_pad + s. A "row block" holds up
//    to 4 M-tiles of 128 rows that stay resident in shared memory. A query
//    longer than a row block is split into chunks whose partial scores are
//    summed afterwards ("late-interaction-kernels" design notes, "Long-query
//    chunking": the sum of maxima decomposes over query tokens).
//  * Documents are packed token rows (dense D is the special case
//    cu[j] = j * Ld). A "doc range" is a run of whole documents holding about
//    total_d / n_dr tokens; a work unit is (row block, doc range).
//  * Each document is cut into tiles of up to 128 of its own tokens; the MMA N
//    of a tile is its token count rounded up to 16, so work follows the real
//    tokens ("Flash-MaxSim" Sec. 4.3.2) and a tile never spans two documents.
//  * Masking without per-element work in the epilogue: the prep warps
//    overwrite, in shared memory, the operand rows of masked tokens and of the
//    padding up to N with NaN. Every similarity in those columns is then NaN,
//    and max.f32 returns its non-NaN operand, so those columns can never win:
//    the same effect as setting them to -inf before the max ("Flash-MaxSim"
//    Sec. 4.1.1; design notes, "Mask handling"). A row whose every column is
//    masked keeps m = -inf.
//  * For every (tile, M-tile) one MMA chain S = Q_blk * D_tile^T (K = dim)
//    accumulates in a 128-column TMEM buffer; the epilogue warps read it
//    with tcgen05.ld while the tensor core fills the next buffer. For 16-bit
//    operands the load itself returns each 32-column chunk's maximum
//    (tcgen05.ld.red .max), so the running max costs one max per chunk. One
//    elected lane of an MMA warp issues each K = dim chain from a single asm
//    block; a single CTA has two MMA warps (M-tiles alternate between them)
//    so that one issues while the other waits on a barrier.
//  * Pair mode (a cluster of two CTAs on two SMs, query rows in shared
//    memory, four accumulator buffers): the MMA is
//    tcgen05.mma.cta_group::2 with M = 256, issued by the even CTA. Each CTA
//    keeps its own row block of query rows (the A half of the MMA) and loads
//    half of every document tile (the B half): one instruction drives both
//    tensor cores and each document tile is read once per pair. The prep and
//    epilogue warps of both CTAs report to the even CTA's barriers; the MMA
//    completion is multicast to both.
//  * INT8 mode ("Flash-MaxSim" Sec. 4.3.1): the tensor-core kind for 8-bit
//    integers is not available on sm_103a, so the prep warps convert the INT8
//    document tile to f16 in shared memory (exact: |v| <= 127), the MMA
//    accumulates in fp32 (exact: |dot| < 2^24 for dim <= 256), and the
//    epilogue applies the per-token scales: v = dot * d_scale[t] before the
//    max, q_scale[s] on the row maximum.
//
// Epilogue ("late-interaction-kernels" notes, "Forward"):
//  * running max per query row: m <- max(m, chunk max); the argmax moves only
//    on a strictly greater chunk max and, inside a 32-column chunk, takes the
//    lowest column: the overall lowest index wins among equal maxima;
//  * at a document's end: m <- 0 unless finite and the row is active, then the
//    rows of each query are summed (warp shuffles, then a fixed-order sum of
//    per-warp partials), so the scores are bitwise reproducible.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace maxsim {

constexpr int kBN = 128;          // document tokens per tile (largest MMA N)
constexpr int kBM = 128;          // query rows per M-tile (MMA M)
constexpr int kMaxMT = 4;         // M-tiles per row block
constexpr int kNAcc = 4;          // TMEM accumulator buffers (4 x 128 columns)
constexpr int kEpiGroups = 2;     // epilogue warpgroups; group g owns the M-tiles k with k % 2 == g
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kThreads = 128 + 32 * kEpiWarps;  // warp 0 TMA, warp 1 MMA, warps 2-3 prep, then the epilogue
constexpr int kEpiWarp0 = 4;

constexpr int kAtomBytes = 128 * 128;  // one 128-row x 128-byte swizzled block
// Registers per thread: the launch gives every thread kRegsLaunch; the
// producer / MMA / prep warpgroup then hands registers to the two epilogue
// warpgroups, which hold a whole accumulator buffer row (128 values).
constexpr int kRegsLaunch = 168;
constexpr int kRegsCtl = 80;
constexpr int kRegsEpi = 208;
static_assert(kRegsCtl * 128 + kRegsEpi * 256 <= kRegsLaunch * (128 + 32 * kEpiWarps), "register split");
constexpr int kMaxStages = 8;

// Device status codes (match maxsim_status).
constexpr int kStatusTimeout = 4;
constexpr int kStatusBadInput = 6;

struct FwdArgs {
    // query rows, padded layout: row r = i * lq_pad + s
    int32_t nq;
    int32_t lq_pad;       // rows per query (power of two <= 16, or a multiple of 32)
    int32_t lq_out;       // argmax columns per (i, j) row
    const uint8_t* q_active;  // [R] nonzero = row contributes (NULL = all)
    const uint8_t* q_real;    // [R] nonzero = a real token (NULL = all)
    const float* q_scale;     // [R] INT8 mode: per-row query scale
    int32_t rb_rows;      // rows per row block
    int32_t n_chunks;     // row blocks per query (> 1 only when lq_pad > rb_rows)
    int32_t n_rb;
    // documents (packed token rows)
    const int32_t* cu_d;  // [nd + 1] or NULL => cu[j] = j * ld
    int32_t nd;
    int32_t ld;
    int32_t total_d;
    const uint8_t* d_mask;   // [total_d] or NULL
    const float* d_scale;    // [total_d] INT8 mode: per-token document scale
    int32_t n_dr;         // document ranges
    int32_t n_units;      // n_rb * n_dr
    // pair-list mode (score_pairs_packed): a unit is one query and a run of
    // its (query, document) pairs; NULL pr_sorted = the [Nq, Nd] grid
    const int32_t* pr_pairs;   // [num_pairs, 2] (query index, document index)
    const int32_t* pr_sorted;  // [num_pairs] pair indices grouped by query
    const int32_t* pr_qptr;    // [nq + 1] first grouped position of each query's pairs
    const int32_t* pr_uptr;    // [nq + 1] first unit of each query; pr_uptr[nq] = number of units
    int32_t pr_chunk;          // pairs per unit
    // outputs
    float* scores;        // [nq, nd]
    float* partial;       // [n_chunks, nq, nd] when n_chunks > 1
    int32_t* argmax;      // [nq * nd, lq_out] or NULL
    // operand geometry
    int32_t k_steps;      // dim / 16 MMA instructions per tile
    int32_t k_atoms;      // 64-element (128-byte) blocks of a 16-bit operand row
    int32_t k8_atoms;     // 128-element blocks of an INT8 row (INT8 mode)
    int32_t dim;
    int32_t stages;       // operand ring depth
    int32_t stages8;      // INT8 staging ring depth (INT8 mode)
    int32_t q_slots;      // M-tiles of Q resident in shared memory
    int32_t n_pr;         // pair mode: row-block pairs (ceil(n_rb / 2))
    uint32_t idesc;       // tcgen05 instruction descriptor without N
    uint32_t nan_pair;    // two 16-bit NaNs of the operand type
    int* status;          // device status word
    uint64_t timeout_ns;  // bound on any single wait
    // Fault-handling test hook (0 = off): the epilogue warps first wait on a
    // barrier that nothing arrives at, giving up after this many ns; every
    // other wait and every drain keeps timeout_ns.
    uint64_t inject_wait_ns;
};

struct RowBlock {
    int32_t row0, row_end;  // global padded rows [row0, row_end)
    int32_t q0, nqb;        // first query, number of queries in the block
    int32_t chunk;          // chunk index within the query (0 if unchunked)
    int32_t mt;             // M-tiles to compute
};

__device__ __forceinline__ RowBlock row_block(const FwdArgs& a, int32_t rb) {
    RowBlock b;
    if (rb >= a.n_rb) {  // the odd CTA of a last, half-empty pair
        b.row0 = b.row_end = a.nq * a.lq_pad;
        b.q0 = a.nq;
        b.nqb = 0;
        b.chunk = 0;
        b.mt = 0;
        return b;
    }
    if (a.n_chunks == 1) {
        int32_t qpb = a.rb_rows / a.lq_pad;
        b.q0 = rb * qpb;
        int32_t q1 = min(b.q0 + qpb, a.nq);
        b.nqb = q1 - b.q0;
        b.row0 = b.q0 * a.lq_pad;
        b.row_end = q1 * a.lq_pad;
        b.chunk = 0;
    } else {
        int32_t i = rb / a.n_chunks;
        b.chunk = rb % a.n_chunks;
        b.q0 = i;
        b.nqb = 1;
        b.row0 = i * a.lq_pad + b.chunk * a.rb_rows;
        b.row_end = min(b.row0 + a.rb_rows, (i + 1) * a.lq_pad);
    }
    b.mt = (b.row_end - b.row0 + kBM - 1) / kBM;
    return b;
}

__device__ __forceinline__ int32_t doc_start(const FwdArgs& a, int32_t j) {
    // Clamped so that inconsistent offsets (reported separately) stay in bounds.
    return a.cu_d ? min(max(__ldg(a.cu_d + j), 0), a.total_d) : j * a.ld;
}

// First document of range dr: lower bound of the token target dr*total/n_dr.
__device__ __forceinline__ int32_t range_first_doc(const FwdArgs& a, int32_t dr) {
    if (dr <= 0) return 0;
    if (dr >= a.n_dr) return a.nd;
    int64_t target = (static_cast<int64_t>(a.total_d) * dr) / a.n_dr;
    if (!a.cu_d) {
        if (a.ld == 0) return static_cast<int32_t>((static_cast<int64_t>(a.nd) * dr) / a.n_dr);
        int64_t j = (target + a.ld - 1) / a.ld;
        return static_cast<int32_t>(j < a.nd ? j : a.nd);
    }
    int32_t lo = 0, hi = a.nd;  // first j with cu[j] >= target
    while (lo < hi) {
        int32_t mid = (lo + hi) >> 1;
        if (__ldg(a.cu_d + mid) < target) lo = mid + 1; else hi = mid;
    }
    return lo;
}

struct Unit {
    RowBlock rb;
    int32_t mt;          // M-tiles computed per tile (the pair's larger block in pair mode)
    int32_t j0, j1;      // documents [j0, j1)
    int32_t tok0;        // first token of document j0
};

template <bool kPair>
__device__ __forceinline__ Unit make_unit(const FwdArgs& a, int32_t u, uint32_t rank) {
    Unit w;
    int32_t dr;
    if constexpr (kPair) {
        const int32_t pr = u % a.n_pr;
        dr = u / a.n_pr;
        w.rb = row_block(a, 2 * pr + static_cast<int32_t>(rank));
        w.mt = max(w.rb.mt, row_block(a, 2 * pr + 1 - static_cast<int32_t>(rank)).mt);
    } else {
        if (a.pr_sorted) {
            // query i owns units pr_uptr[i] .. pr_uptr[i+1]-1: the last i with pr_uptr[i] <= u
            int32_t lo = 0, hi = a.nq - 1;
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (__ldg(a.pr_uptr + mid) <= u) lo = mid; else hi = mid - 1;
            }
            const int32_t i = lo;
            const int32_t k0 = __ldg(a.pr_qptr + i) + (u - __ldg(a.pr_uptr + i)) * a.pr_chunk;
            w.rb.q0 = i;
            w.rb.nqb = 1;
            w.rb.chunk = 0;
            w.rb.row0 = i * a.lq_pad;
            w.rb.row_end = w.rb.row0 + a.lq_pad;
            w.rb.mt = (a.lq_pad + kBM - 1) / kBM;
            w.mt = w.rb.mt;
            w.j0 = k0;
            w.j1 = min(k0 + a.pr_chunk, __ldg(a.pr_qptr + i + 1));
            w.tok0 = 0;
            return w;
        }
        w.rb = row_block(a, u % a.n_rb);
        w.mt = w.rb.mt;
        dr = u / a.n_rb;
    }
    w.j0 = range_first_doc(a, dr);
    w.j1 = range_first_doc(a, dr + 1);
    w.tok0 = doc_start(a, w.j0);
    return w;
}

// Output index of (query i, document position oj): the [Nq, Nd] grid, or in
// pair-list mode the pair index itself.
__device__ __forceinline__ int64_t out_index(const FwdArgs& a, int32_t i, int32_t oj) {
    return a.pr_sorted ? static_cast<int64_t>(oj) : static_cast<int64_t>(i) * a.nd + oj;
}

// Walks the tiles of a unit in order: documents j0..j1-1 (in pair-list mode
// the documents of grouped pairs j0..j1-1), each cut into tiles of up to kBN
// of its own tokens; empty documents have no tile. The bounds of the next
// document are loaded one document ahead and only clamped when they are
// used, so the loads' latency is not waited for at a document boundary.
struct TileWalk {
    int32_t j, j1, ds, de, t0;
    int32_t oj;                    // output column of document j (pair index in pair-list mode)
    int32_t nx_oj, nx_s, nx_e;     // raw bounds of the next document (nx_s unused on the grid)
    __device__ __forceinline__ static int32_t raw_start(const FwdArgs& a, int32_t j) {
        return a.cu_d ? __ldg(a.cu_d + j) : j * a.ld;
    }
    __device__ __forceinline__ static int32_t clamp_start(const FwdArgs& a, int32_t v) {
        // inconsistent offsets (reported separately) stay in bounds
        return min(max(v, 0), a.total_d);
    }
    // pair-list mode: pair, and raw token range of its document, at grouped position k
    __device__ __forceinline__ void load_pair(const FwdArgs& a, int32_t k, int32_t& p, int32_t& s0, int32_t& e0) const {
        p = __ldg(a.pr_sorted + k);
        const int32_t doc = __ldg(a.pr_pairs + 2 * p + 1);
        s0 = __ldg(a.cu_d + doc);
        e0 = __ldg(a.cu_d + doc + 1);
    }
    __device__ __forceinline__ void begin(const FwdArgs& a, const Unit& w) {
        j = w.j0;
        j1 = w.j1;
        t0 = 0;
        if (!a.pr_sorted) {
            ds = w.tok0;
            de = j < j1 ? doc_start(a, j + 1) : ds;
            oj = j;
            nx_e = raw_start(a, min(j + 2, a.nd));  // promoted only while j + 1 < j1
        } else if (j < j1) {
            int32_t s0, e0;
            load_pair(a, j, oj, s0, e0);
            ds = clamp_start(a, s0);
            de = max(ds, clamp_start(a, e0));
            load_pair(a, min(j + 1, j1 - 1), nx_oj, nx_s, nx_e);
        } else {
            ds = de = 0;
            oj = 0;
        }
        skip_empty(a);
    }
    __device__ __forceinline__ void next_doc(const FwdArgs& a) {
        ++j;
        t0 = 0;
        if (!a.pr_sorted) {
            ds = de;
            de = clamp_start(a, nx_e);
            oj = j;
            nx_e = raw_start(a, min(j + 2, a.nd));
        } else {
            oj = nx_oj;
            ds = clamp_start(a, nx_s);
            de = max(ds, clamp_start(a, nx_e));
            load_pair(a, min(j + 1, j1 - 1), nx_oj, nx_s, nx_e);
        }
    }
    __device__ __forceinline__ void skip_empty(const FwdArgs& a) {
        while (j < j1 && de <= ds) next_doc(a);
    }
    __device__ __forceinline__ bool valid() const { return j < j1; }
    __device__ __forceinline__ int32_t row() const { return ds + t0; }                 // first token row
    __device__ __forceinline__ int32_t ntok() const { return min(kBN, de - ds - t0); }  // real tokens
    __device__ __forceinline__ bool last_of_doc() const { return ds + t0 + kBN >= de; }
    __device__ __forceinline__ void advance(const FwdArgs& a) {
        if (last_of_doc()) {
            next_doc(a);
            skip_empty(a);
        } else {
            t0 += kBN;
        }
    }
};

__device__ __forceinline__ int32_t mma_n(int32_t ntok) { return (ntok + 15) & ~15; }

// Shared-memory control block (after the operand buffers).
struct alignas(16) SmemCtl {
    uint64_t q_full, q_empty;
    uint64_t d_full[kMaxStages], d_ready[kMaxStages], d_empty[kMaxStages];
    uint64_t d8_full[kMaxStages], d8_empty[kMaxStages];
    uint64_t q_ready;  // pair mode: both CTAs' query rows have landed
    uint64_t acc_full[kNAcc], acc_empty[kNAcc];
    uint64_t mma_done;
    uint64_t epi_bar;                // rendezvous of all epilogue warps
    uint64_t epi_bar_g[kEpiGroups];  // rendezvous of one epilogue warpgroup
    uint64_t never;    // never arrived at (the fault-handling test hook waits on it)
    uint32_t tmem_base;
    volatile int32_t abort;
    float wslot[2][kMaxMT * 4];  // per-warp partial sums of the document being closed (by parity)
};
// INT8 mode only: after the control block, a per-warp copy of the tile's
// document scales, float[kEpiWarps][kBN].
constexpr int kDScaleBytes = kEpiWarps * kBN * 4;

__device__ __forceinline__ void record_status(const FwdArgs& a, int code) {
    if (a.status) atomicCAS(a.status, 0, code);
}

// Bounded wait: gives up after limit_ns (records the status and raises the
// CTA abort flag) or when another role has already aborted. Inlined: the
// kernel's warpgroups run under different register budgets (setmaxnreg),
// which an out-of-line call shared between them cannot follow.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar_slow(const FwdArgs& a, SmemCtl* ctl, uint32_t bar, uint32_t parity,
                                              uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (ctl->abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                ctl->abort = 1;
                record_status(a, kStatusTimeout);
                return false;
            }
        }
    }
}

// kCluster: the barrier also receives arrivals from the other CTA of a pair
// (acquire at cluster scope).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(const FwdArgs& a, SmemCtl* ctl, uint32_t bar, uint32_t parity) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow<kCluster>(a, ctl, bar, parity, a.timeout_ns);
}

// wait_bar for a whole warp that runs warp-uniform code: every lane polls,
// and the warp continues together with one answer.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar_warp(const FwdArgs& a, SmemCtl* ctl, uint32_t bar, uint32_t parity) {
    const bool ok = wait_bar<kCluster>(a, ctl, bar, parity);
    return __all_sync(0xFFFFFFFFu, ok);
}

// Bounded rendezvous of the epilogue warps (an mbarrier phase per use),
// so that a warp that gave up on a wait can never strand the others.
__device__ __forceinline__ bool epi_sync(const FwdArgs& a, SmemCtl* ctl, uint64_t* bar, uint32_t& phase) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(bar));
    const bool ok = wait_bar(a, ctl, smem_u32(bar), phase);
    phase ^= 1u;
    return ok;
}

// ---------------------------------------------------------------- epilogue helpers

// max over 32 values and m; NaN entries are ignored by max.f32.
__device__ __forceinline__ float chunk_max(const float (&x)[32], float m) {
    float a0 = fmax3(x[0], x[1], x[2]), a1 = fmax3(x[3], x[4], x[5]), a2 = fmax3(x[6], x[7], x[8]);
    float a3 = fmax3(x[9], x[10], x[11]), a4 = fmax3(x[12], x[13], x[14]), a5 = fmax3(x[15], x[16], x[17]);
    float a6 = fmax3(x[18], x[19], x[20]), a7 = fmax3(x[21], x[22], x[23]), a8 = fmax3(x[24], x[25], x[26]);
    float a9 = fmax3(x[27], x[28], x[29]), a10 = fmax3(x[30], x[31], m);
    float b0 = fmax3(a0, a1, a2), b1 = fmax3(a3, a4, a5), b2 = fmax3(a6, a7, a8), b3 = fmax3(a9, a10, b0);
    return fmax3(b1, b2, b3);
}

// Lowest e with y[e] == cm, where cm is the largest non-NaN entry of y.
// set.ge turns each column into 1.0 (equal to the maximum) or 0.0 (below it,
// or NaN), and the flags are added as t_e * 2^-e: the sum lies in
// [2^-e0, 2^(1-e0)) for the lowest flagged e0 (rounded toward zero, so the
// lower flags never carry into the next power of two), and its exponent is
// -e0. One compare (integer pipe) and one FMA (floating-point pipe) per
// column, in place of a compare and a select on the integer pipe.
__device__ __forceinline__ int32_t first_equal32(const float (&y)[32], float cm) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        float t;
        asm("set.ge.f32.f32 %0, %1, %2;" : "=f"(t) : "f"(y[e]), "f"(cm));
        acc[e >> 3] = __fmaf_rz(t, __uint_as_float(static_cast<uint32_t>(127 - e) << 23), acc[e >> 3]);
    }
    const float s = __fadd_rz(__fadd_rz(acc[0], acc[1]), __fadd_rz(acc[2], acc[3]));
    return 127 - static_cast<int32_t>(__float_as_uint(s) >> 23);
}

// Fold one 32-column chunk into (m, am); col0 = index of column 0 relative to
// the document's first token.
template <bool kArg>
__device__ __forceinline__ void fold_chunk(const float (&y)[32], int32_t col0, float& m, int32_t& am) {
    if constexpr (!kArg) {
        m = chunk_max(y, m);
    } else {
        const float kNegInf = __int_as_float(0xff800000u);
        const float cm = chunk_max(y, kNegInf);
        const bool upd = cm > m;  // false for NaN
        if (__any_sync(0xFFFFFFFFu, upd)) {
            const int32_t idx = first_equal32(y, cm);
            if (upd) {
                am = col0 + idx;
                m = cm;
            }
        }
    }
}

// Fold one 32-column chunk whose maximum cm is already known (from the TMEM
// load): only a chunk that beats the running maximum is searched for its
// lowest column equal to cm.
__device__ __forceinline__ void fold_chunk_max(const float (&y)[32], float cm, int32_t col0, float& m, int32_t& am) {
    const bool upd = cm > m;  // false for NaN
    if (__any_sync(0xFFFFFFFFu, upd)) {
        const int32_t idx = first_equal32(y, cm);
        if (upd) {
            am = col0 + idx;
            m = cm;
        }
    }
}

// ---------------------------------------------------------------- the kernel

template <bool kArg, bool kInt8, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    maxsim_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_d,
                      const FwdArgs a) {
    constexpr int kG = kPair ? 2 : 1;              // tcgen05 CTA group
    // Single CTAs keep the query rows in tensor memory (the MMA's A operand
    // then costs no shared-memory bandwidth) next to two accumulator
    // buffers; CTA pairs keep them in shared memory next to four.
    constexpr int kAccBufs = kNAcc;
    // Two MMA warps (1 and 3) share the issue work: M-tiles k = i, i + 2, ...
    // go to warp i, so that one issues while the other waits or keeps books.
    // An INT8 CTA pair has one issuer and two prep warps (the widening).
    constexpr int kMmaWarps = (kPair && kInt8) ? 1 : 2;
    constexpr int kPrepWarps = 3 - kMmaWarps;
    constexpr int kDRows = kPair ? kBN / 2 : kBN;  // document rows per operand stage in this CTA
    constexpr int kDAtom = kDRows * 128;           // bytes of one 128-byte-wide K block of a stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t q_tile_bytes = a.k_atoms * kAtomBytes;  // one 128-row M-tile of Q
    const int32_t d_stage_bytes = a.k_atoms * kDAtom;     // this CTA's rows of one operand tile
    const int32_t d8_stage_bytes = a.k8_atoms * kDAtom;   // this CTA's rows of one INT8 tile
    uint8_t* sQ = smem;
    uint8_t* sD = smem + a.q_slots * q_tile_bytes;
    uint8_t* sD8 = sD + a.stages * d_stage_bytes;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(sD8 + (kInt8 ? a.stages8 * d8_stage_bytes : 0));
    float* dscale = reinterpret_cast<float*>(ctl + 1);  // [kEpiWarps][kBN], INT8 mode

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // shared::cluster address of a barrier of this CTA in the pair's even CTA
    auto at_leader = [&](const uint64_t* bar) -> uint32_t {
        return kPair ? map_shared_rank(smem_u32(bar), 0) : smem_u32(bar);
    };
    auto arrive_leader = [&](const uint64_t* bar) {
        if constexpr (kPair) mbar_arrive_cluster(at_leader(bar));
        else mbar_arrive(smem_u32(bar));
    };
    // accumulator buffer handed back: only tensor-memory reads precede it
    auto release_acc = [&](const uint64_t* bar) {
        if constexpr (kPair) mbar_arrive_remote(at_leader(bar));
        else mbar_arrive(smem_u32(bar));
    };

    // Ring depths index fixed-size barrier arrays: refuse a launch that breaks
    // them (both CTAs of a pair see the same arguments and return together).
    if (a.stages < 1 || a.stages > kMaxStages || (kInt8 && (a.stages8 < 1 || a.stages8 > kMaxStages)) ||
        a.q_slots < 1 || a.q_slots > kMaxMT) {
        if (threadIdx.x == 0) record_status(a, kStatusBadInput);
        return;
    }

    if (threadIdx.x == 0) {
        const uint32_t ctas = kPair ? 2u : 1u;
        mbar_init(smem_u32(&ctl->q_full), 1);
        mbar_init(smem_u32(&ctl->q_empty), kMmaWarps);
        mbar_init(smem_u32(&ctl->q_ready), ctas);
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(smem_u32(&ctl->d_full[s]), 1);
            mbar_init(smem_u32(&ctl->d_ready[s]), kPrepWarps * ctas);
            mbar_init(smem_u32(&ctl->d_empty[s]), kMmaWarps);
        }
        for (int s = 0; s < a.stages8; ++s) {
            mbar_init(smem_u32(&ctl->d8_full[s]), 1);
            mbar_init(smem_u32(&ctl->d8_empty[s]), kPrepWarps);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(smem_u32(&ctl->acc_full[b]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[b]), 4 * ctas);
        }
        mbar_init(smem_u32(&ctl->mma_done), kMmaWarps);
        mbar_init(smem_u32(&ctl->epi_bar), kEpiWarps);
        for (int gg = 0; gg < kEpiGroups; ++gg) mbar_init(smem_u32(&ctl->epi_bar_g[gg]), 4);
        mbar_init(smem_u32(&ctl->never), 1);
        ctl->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_d);
    }
    if (warp == 1) {
        tmem_alloc<kG>(smem_u32(&ctl->tmem_base), kNAcc * kBN);
        tmem_relinquish<kG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // barriers of both CTAs exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int32_t n_units = a.pr_sorted ? __ldg(a.pr_uptr + a.nq) : a.n_units;
    const int32_t u0 = kPair ? static_cast<int32_t>(blockIdx.x >> 1) : static_cast<int32_t>(blockIdx.x);
    const int32_t u_step = kPair ? static_cast<int32_t>(gridDim.x >> 1) : static_cast<int32_t>(gridDim.x);

    // Warpgroup 0 (producer, MMA, prep) gives registers to the epilogue
    // warpgroups; each branch below runs under its own register budget.
    if (warp < kEpiWarp0) {
    regs_release<kRegsCtl>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();
            // f16/bf16: tiles go straight into the operand ring; INT8: into the staging ring
            const int32_t ring = kInt8 ? a.stages8 : a.stages;
            const int32_t bytes = kInt8 ? d8_stage_bytes : d_stage_bytes;
            const int32_t boxes = kInt8 ? a.k8_atoms : a.k_atoms;
            const int32_t box_cols = kInt8 ? 128 : 64;
            uint8_t* base = kInt8 ? sD8 : sD;
            int32_t stage = 0;
            uint32_t phase = 0, q_phase = 0;
            bool first_unit = true;
            int64_t issued = 0, q_issued = 0;
            bool ok = true;
            for (int32_t u = u0; u < n_units && ok; u += u_step) {
                const Unit w = make_unit<kPair>(a, u, rank);
                if (!first_unit) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->q_empty), q_phase)) break;
                    q_phase ^= 1u;
                }
                first_unit = false;
                const uint32_t qbar = smem_u32(&ctl->q_full);
                mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(w.mt * q_tile_bytes));
                for (int32_t k = 0; k < w.mt; ++k)
                    for (int32_t ka = 0; ka < a.k_atoms; ++ka)
                        tma_load_2d(smem_u32(sQ + k * q_tile_bytes + ka * kAtomBytes), &tm_q, qbar, ka * 64,
                                    w.rb.row0 + k * kBM);
                ++q_issued;
                TileWalk tw;
                for (tw.begin(a, w); tw.valid(); tw.advance(a)) {
                    const uint32_t empty = smem_u32(kInt8 ? &ctl->d8_empty[stage] : &ctl->d_empty[stage]);
                    if (!wait_bar(a, ctl, empty, phase ^ 1u)) { ok = false; break; }
                    const uint32_t fullb = smem_u32(kInt8 ? &ctl->d8_full[stage] : &ctl->d_full[stage]);
                    mbar_arrive_expect_tx(fullb, static_cast<uint32_t>(bytes));
                    // this CTA's rows of the tile: all of them, or its half in pair mode
                    const int32_t y = tw.row() + (kPair ? static_cast<int32_t>(rank) * (mma_n(tw.ntok()) >> 1) : 0);
                    for (int32_t ka = 0; ka < boxes; ++ka)
                        tma_load_2d_hint(smem_u32(base + stage * bytes + ka * kDAtom), &tm_d, fullb, ka * box_cols, y,
                                         pol_stream);
                    ++issued;
                    if (++stage == ring) { stage = 0; phase ^= 1u; }
                }
            }
            if (ctl->abort) {
                // Let every copy still in flight land before the CTA exits: the
                // query rows of the current unit (the n-th load completes phase
                // n - 1 of q_full; an earlier one was consumed before the next
                // was issued) and the last ring stages.
                if (q_issued > 0) {
                    const uint64_t t0 = global_timer_ns();
                    const uint32_t qb = smem_u32(&ctl->q_full), qp = static_cast<uint32_t>((q_issued - 1) & 1);
                    while (!mbar_try_wait(qb, qp) && global_timer_ns() - t0 < a.timeout_ns) {}
                }
                const int64_t outstanding = issued < ring ? issued : ring;
                int32_t s = stage;
                uint32_t ph = phase;
                for (int64_t n = 0; n < outstanding; ++n) {
                    if (--s < 0) { s = ring - 1; ph ^= 1u; }
                    const uint32_t fullb = smem_u32(kInt8 ? &ctl->d8_full[s] : &ctl->d_full[s]);
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(fullb, ph) && global_timer_ns() - t0 < a.timeout_ns) {}
                }
            }
        }
    } else if (warp == 1 || (kMmaWarps == 2 && warp == 3)) {
        // ------------------------------------------------------------ MMA issuers (even CTA of a pair)
        // Each MMA warp runs this loop with warp-uniform values; one elected
        // lane issues the MMA chains and the commits.
        if (leader) {
            const int32_t mi = warp == 1 ? 0 : 1;
            int32_t stage = 0;
            int64_t buf = 0;  // global index of the tile's first accumulator buffer use
            uint32_t phase = 0, q_phase = 0;
            const uint64_t q_desc0 = sdesc_k_sw128(smem_u32(sQ));
            const uint32_t idesc_m = a.idesc | (static_cast<uint32_t>((kPair ? 2 * kBM : kBM) >> 4) << 24);
            constexpr uint32_t kA16 = kAtomBytes >> 4, kB16 = kDAtom >> 4;
            bool ok = true;
            for (int32_t u = u0; u < n_units && ok; u += u_step) {
                const Unit w = make_unit<kPair>(a, u, rank);
                TileWalk tw;
                tw.begin(a, w);
                if constexpr (kPair) {
                    if (!wait_bar_warp<true>(a, ctl, smem_u32(&ctl->q_ready), q_phase)) break;
                } else {
                    if (!wait_bar_warp(a, ctl, smem_u32(&ctl->q_full), q_phase)) break;
                }
                q_phase ^= 1u;
                tc_fence_after();
                for (; tw.valid() && ok; tw.advance(a)) {
                    if (!wait_bar_warp<kPair>(a, ctl, smem_u32(&ctl->d_ready[stage]), phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t idesc = idesc_m | (static_cast<uint32_t>(mma_n(tw.ntok()) >> 3) << 17);
                    const uint64_t b_desc0 = sdesc_k_sw128(smem_u32(sD + stage * d_stage_bytes));
                    for (int32_t k = mi; k < w.mt; k += kMmaWarps) {
                        const int64_t idx = buf + k;
                        const int32_t acc = static_cast<int32_t>(idx % kAccBufs);
                        const uint32_t acc_phase = static_cast<uint32_t>((idx / kAccBufs) & 1);
                        if (!wait_bar_warp<kPair>(a, ctl, smem_u32(&ctl->acc_empty[acc]), acc_phase ^ 1u)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                        if (a.k_steps == 8) {  // dim 128: one chain
                            const uint64_t a_desc0 = q_desc0 + static_cast<uint64_t>((k * q_tile_bytes) >> 4);
                            mma_chain8_ss<kG, kA16, kB16>(d_tmem, a_desc0, b_desc0, idesc, 0u);
                        } else {
                            const uint64_t a_desc0 = q_desc0 + static_cast<uint64_t>((k * q_tile_bytes) >> 4);
                            // 64-element atoms as 4-step chains, then single steps
                            int32_t ks = 0;
                            for (; ks + 4 <= a.k_steps; ks += 4)
                                mma_chain4_ss<kG>(d_tmem, a_desc0 + (ks >> 2) * kA16, b_desc0 + (ks >> 2) * kB16, idesc,
                                                  ks > 0 ? 1u : 0u);
                            for (; ks < a.k_steps; ++ks)
                                mma_step_ss<kG>(d_tmem, a_desc0 + (ks >> 2) * kA16 + (ks & 3) * 2,
                                                b_desc0 + (ks >> 2) * kB16 + (ks & 3) * 2, idesc, ks > 0 ? 1u : 0u);
                        }
                        mma_commit_elect<kG>(smem_u32(&ctl->acc_full[acc]));
                    }
                    if (!ok) break;
                    buf += w.mt;
                    mma_commit_elect<kG>(smem_u32(&ctl->d_empty[stage]));
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_elect<kG>(smem_u32(&ctl->q_empty));
            }
            // Drain: wait until every MMA issued above has completed.
            mma_commit_elect<kG>(smem_u32(&ctl->mma_done), 1);
            if (lane == 0) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_u32(&ctl->mma_done), 0) && global_timer_ns() - t0 < a.timeout_ns) {}
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ operand prep
        // f16/bf16: NaN-fill masked / padding rows in place. INT8: convert the
        // staged INT8 tile to f16 rows (NaN for masked / padding rows). In pair
        // mode each CTA handles its half of the tile's rows.
        const int pt = threadIdx.x - 64;  // 0 .. 32 * kPrepWarps - 1
        constexpr int kPrepThreads = 32 * kPrepWarps;
        // INT8 widening: when the chunks of a row (dim / 16) divide the prep
        // threads, each thread keeps one chunk column for the whole kernel
        const int32_t prep_chunks = a.dim >> 4;
        const bool prep_fixed_chunk = prep_chunks > 0 && kPrepThreads % prep_chunks == 0;
        const int32_t prep_c = prep_fixed_chunk ? pt % prep_chunks : 0;
        const int32_t prep_r0 = prep_fixed_chunk ? pt / prep_chunks : 0;
        const int32_t prep_rstep = prep_fixed_chunk ? kPrepThreads / prep_chunks : 1;
        int32_t stage = 0, stage8 = 0;
        uint32_t phase = 0, phase8 = 0, q_phase = 0;
        bool ok = true;
        for (int32_t u = u0; u < n_units && ok; u += u_step) {
            const Unit w = make_unit<kPair>(a, u, rank);
            if constexpr (kPair) {
                // report this CTA's query rows to the MMA issuer
                if (pt == 0) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->q_full), q_phase)) { ok = false; break; }
                    arrive_leader(&ctl->q_ready);
                }
                q_phase ^= 1u;
            }
            TileWalk tw;
            for (tw.begin(a, w); tw.valid(); tw.advance(a)) {
                const int32_t n = tw.ntok(), N = mma_n(n);
                const int32_t rows = kPair ? (N >> 1) : N;                      // this CTA's rows
                const int32_t tr0 = kPair ? static_cast<int32_t>(rank) * rows : 0;  // their first tile row
                const int32_t row0 = tw.row() + tr0;
                uint8_t* dst = sD + stage * d_stage_bytes;
                if constexpr (kInt8) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->d8_full[stage8]), phase8)) { ok = false; break; }
                    if (!wait_bar(a, ctl, smem_u32(&ctl->d_empty[stage]), phase ^ 1u)) { ok = false; break; }
                    const uint8_t* src = sD8 + stage8 * d8_stage_bytes;
                    // one 16-byte INT8 chunk (c) of row r: 16 f16 values = two 16-byte
                    // chunks of a 64-element swizzled atom
                    auto widen = [&](int32_t r, int32_t c) {
                        const bool nan_row = tr0 + r >= n || (a.d_mask != nullptr && a.d_mask[row0 + r] == 0);
                        uint4 lo, hi;
                        if (nan_row) {
                            lo = make_uint4(a.nan_pair, a.nan_pair, a.nan_pair, a.nan_pair);
                            hi = lo;
                        } else {
                            // INT8 rows: 128-byte swizzled rows of 128 elements per staging block
                            const int32_t blk = c >> 3, cc = c & 7;
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                src + blk * kDAtom + r * 128 + ((cc ^ (r & 7)) << 4));
                            lo = i8x8_to_f16x8(v.x, v.y);
                            hi = i8x8_to_f16x8(v.z, v.w);
                        }
                        const int32_t atom = c >> 2, c16 = (c & 3) * 2;
                        uint8_t* rowp = dst + atom * kDAtom + r * 128;
                        *reinterpret_cast<uint4*>(rowp + (((c16 + 0) ^ (r & 7)) << 4)) = lo;
                        *reinterpret_cast<uint4*>(rowp + (((c16 + 1) ^ (r & 7)) << 4)) = hi;
                    };
                    if (prep_fixed_chunk) {
                        // every thread keeps one chunk column; rows step by the threads
                        // per chunk column (no division in the loop)
#pragma unroll 4
                        for (int32_t r = prep_r0; r < rows; r += prep_rstep) widen(r, prep_c);
                    } else {
                        const int32_t chunks = a.dim >> 4;  // 16-byte INT8 chunks per row
                        for (int32_t x = pt; x < rows * chunks; x += kPrepThreads) {
                            const int32_t r = x / chunks;
                            widen(r, x - r * chunks);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        arrive_leader(&ctl->d_ready[stage]);
                        mbar_arrive(smem_u32(&ctl->d8_empty[stage8]));
                    }
                    if (++stage8 == a.stages8) { stage8 = 0; phase8 ^= 1u; }
                } else {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->d_full[stage]), phase)) { ok = false; break; }
                    if (a.d_mask != nullptr || tr0 + rows > n) {
                        const uint4 nan4 = make_uint4(a.nan_pair, a.nan_pair, a.nan_pair, a.nan_pair);
                        for (int32_t r = pt; r < rows; r += kPrepThreads) {
                            if (tr0 + r < n && (a.d_mask == nullptr || a.d_mask[row0 + r] != 0)) continue;
                            for (int32_t ka = 0; ka < a.k_atoms; ++ka) {
                                uint4* rowp = reinterpret_cast<uint4*>(dst + ka * kDAtom + r * 128);
#pragma unroll
                                for (int c = 0; c < 8; ++c) rowp[(c + lane) & 7] = nan4;  // rotated: 8 rows per phase hit 8 bank groups
                            }
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) arrive_leader(&ctl->d_ready[stage]);
                }
                if (++stage == a.stages) { stage = 0; phase ^= 1u; }
            }
        }
    }
    } else {
        regs_claim<kRegsEpi>();
        // ------------------------------------------------------------ epilogue
        // Warpgroup g owns the M-tiles k = g, g + kEpiGroups, ...; each of its
        // threads owns one query row of each of those M-tiles.
        constexpr int kKPer = kMaxMT / kEpiGroups;
        const float kNegInf = __int_as_float(0xff800000u);
        const float kNaN = __int_as_float(0x7fffffffu);
        const int ew = warp - kEpiWarp0;              // epilogue warp 0..kEpiWarps-1
        const int g = ew >> 2;                        // warpgroup
        const int e = ew & 3;                         // TMEM lane quadrant
        const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..32*kEpiWarps-1
        int64_t buf = 0;                              // global index of the tile's first buffer
        uint32_t epi_phase = 0, grp_phase = 0;
        uint32_t par = 0;  // parity of the documents closed so far (selects the wslot half)
        bool ok = true;
        if (a.inject_wait_ns != 0)  // fault-handling test hook: this wait can only give up
            ok = wait_bar_slow<false>(a, ctl, smem_u32(&ctl->never), 0u, a.inject_wait_ns);
        for (int32_t u = u0; u < n_units && ok; u += u_step) {
            const Unit w = make_unit<kPair>(a, u, rank);
            const RowBlock& rb = w.rb;
            const bool chunked = a.n_chunks > 1;
            int32_t row_i[kKPer], row_s[kKPer];
            bool in_rb[kKPer], real[kKPer], active[kKPer];
            float qsc[kKPer];
#pragma unroll
            for (int q = 0; q < kKPer; ++q) {
                const int k = g + kEpiGroups * q;
                const int32_t r = rb.row0 + k * kBM + e * 32 + lane;
                in_rb[q] = k < rb.mt && r < rb.row_end;
                row_i[q] = r / a.lq_pad;
                row_s[q] = r - row_i[q] * a.lq_pad;
                real[q] = in_rb[q] && (a.q_real == nullptr || a.q_real[r] != 0);
                active[q] = real[q] && (a.q_active == nullptr || a.q_active[r] != 0);
                qsc[q] = (kInt8 && in_rb[q]) ? a.q_scale[r] : 1.f;
            }
            // empty documents: score 0 and argmax -1, written up front
            for (int32_t j = w.j0 + et; j < w.j1 && a.pr_sorted; j += 32 * kEpiWarps) {
                const int32_t p = __ldg(a.pr_sorted + j);
                const int32_t doc = __ldg(a.pr_pairs + 2 * p + 1);
                if (__ldg(a.cu_d + doc + 1) > __ldg(a.cu_d + doc)) continue;
                a.scores[p] = 0.f;
                if (kArg)
                    for (int32_t s = 0; s < a.lq_out; ++s) a.argmax[static_cast<int64_t>(p) * a.lq_out + s] = -1;
            }
            for (int32_t j = w.j0 + et; j < w.j1 && !a.pr_sorted; j += 32 * kEpiWarps) {
                if (doc_start(a, j + 1) > doc_start(a, j)) continue;
                for (int32_t q = 0; q < rb.nqb; ++q) {
                    const int32_t i = rb.q0 + q;
                    if (chunked) a.partial[(static_cast<int64_t>(rb.chunk) * a.nq + i) * a.nd + j] = 0.f;
                    else a.scores[static_cast<int64_t>(i) * a.nd + j] = 0.f;
                }
                if (kArg) {
                    for (int32_t r = rb.row0; r < rb.row_end; ++r) {
                        const int32_t i = r / a.lq_pad, s = r - (r / a.lq_pad) * a.lq_pad;
                        if (s < a.lq_out) a.argmax[(static_cast<int64_t>(i) * a.nd + j) * a.lq_out + s] = -1;
                    }
                }
            }
            float m[kKPer];
            int32_t am[kKPer];
#pragma unroll
            for (int q = 0; q < kKPer; ++q) { m[q] = kNegInf; am[q] = -1; }

            // INT8: this lane's document scales (columns c * 32 + lane) of the
            // next tile, loaded one tile ahead
            float sc_next[4];
            auto load_scales = [&](const TileWalk& t) {
                const int32_t tn = t.ntok(), trow = t.row();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int32_t col = c * 32 + lane;
                    sc_next[c] = col < tn ? __ldg(a.d_scale + trow + col) : 0.f;
                }
            };
            TileWalk tw;
            tw.begin(a, w);
            if (kInt8 && tw.valid()) load_scales(tw);
            for (; tw.valid() && ok; tw.advance(a)) {
                const int32_t n = tw.ntok(), N = mma_n(n);
                const int32_t nfull = N >> 5;
                const bool half = (N & 31) != 0;
                const int32_t nchunks = nfull + (half ? 1 : 0);
                const bool closes = tw.last_of_doc();
                if constexpr (kInt8) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) dscale[ew * kBN + c * 32 + lane] = sc_next[c];
                    __syncwarp();
                    TileWalk nx = tw;
                    nx.advance(a);
                    if (nx.valid()) load_scales(nx);
                }
#pragma unroll
                for (int q = 0; q < kKPer; ++q) {
                    const int k = g + kEpiGroups * q;
                    if (k >= w.mt) break;
                    const int64_t idx = buf + k;
                    const int32_t slot = static_cast<int32_t>(idx % kAccBufs);
                    const uint32_t ph = static_cast<uint32_t>((idx / kAccBufs) & 1);
                    if (!wait_bar(a, ctl, smem_u32(&ctl->acc_full[slot]), ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(e * 32) << 16) +
                                           static_cast<uint32_t>(slot * kBN);
                    // columns in two halves of up to 64 (registers are the limit)
                    auto fold = [&](float (&vc)[32], int c) {
                        if constexpr (kInt8) {
                            const float4* sc = reinterpret_cast<const float4*>(dscale + ew * kBN + c * 32);
#pragma unroll
                            for (int x = 0; x < 8; ++x) {
                                const float4 s4 = sc[x];
                                mul2_rn(vc[4 * x + 0], vc[4 * x + 1], s4.x, s4.y);
                                mul2_rn(vc[4 * x + 2], vc[4 * x + 3], s4.z, s4.w);
                            }
                        }
                        fold_chunk<kArg>(vc, tw.t0 + c * 32, m[q], am[q]);
                    };
                    // the whole row of the buffer in one round, so that it is handed back
                    // to the MMA warp before the reduction
                    float v[4][32];
                    if constexpr (!kInt8) {
                        // 16-bit operands: the chunk maxima come out of tensor memory
                        // with the values (tcgen05.ld.red)
                        float cm[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            cm[c] = kNegInf;
                            if (c < nfull) {
                                cm[c] = tmem_ldmax32(taddr + c * 32, v[c]);
                            } else if (c == nfull && half) {
                                cm[c] = tmem_ldmax16(taddr + c * 32, v[c]);
#pragma unroll
                                for (int x = 16; x < 32; ++x) v[c][x] = kNaN;
                            }
                        }
                        tmem_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) release_acc(&ctl->acc_empty[slot]);
                        if constexpr (!kArg) {
                            m[q] = fmax3(m[q], fmax3(cm[0], cm[1], cm[2]), cm[3]);
                        } else {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (c < nchunks) fold_chunk_max(v[c], cm[c], tw.t0 + c * 32, m[q], am[q]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (c < nfull) {
                                tmem_ld32(taddr + c * 32, v[c]);
                            } else if (c == nfull && half) {
                                tmem_ld16(taddr + c * 32, v[c]);
#pragma unroll
                                for (int x = 16; x < 32; ++x) v[c][x] = kNaN;
                            }
                        }
                        tmem_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) release_acc(&ctl->acc_empty[slot]);
                        if (nchunks == 4) {  // a full tile: no branch between the chunks
#pragma unroll
                            for (int c = 0; c < 4; ++c) fold(v[c], c);
                        } else {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (c < nchunks) fold(v[c], c);
                        }
                    }
                }
                if (!ok) break;
                if (closes) {
                    // The document ends in this tile. Its reductions come after both
                    // M-tiles' loads (they are off the path that hands the accumulator
                    // buffers back to the MMA warps), the M-tiles' shuffles interleaved.
                    float val[kKPer];
#pragma unroll
                    for (int q = 0; q < kKPer; ++q) {
                        const bool has = m[q] > kNegInf;
                        if (kArg && in_rb[q] && row_s[q] < a.lq_out)
                            a.argmax[out_index(a, row_i[q], tw.oj) * a.lq_out + row_s[q]] =
                                (real[q] && has) ? am[q] : -1;
                        val[q] = (active[q] && has) ? m[q] * qsc[q] : 0.f;
                    }
                    const int32_t width = min(a.lq_pad, 32);
                    for (int o = width >> 1; o > 0; o >>= 1) {
#pragma unroll
                        for (int q = 0; q < kKPer; ++q) val[q] += __shfl_xor_sync(0xFFFFFFFFu, val[q], o);
                    }
#pragma unroll
                    for (int q = 0; q < kKPer; ++q) {
                        const int k = g + kEpiGroups * q;
                        if (k >= w.mt) break;
                        if (a.lq_pad < 32 || (a.lq_pad == 32 && !chunked)) {
                            if (in_rb[q] && (lane & (width - 1)) == 0) a.scores[out_index(a, row_i[q], tw.oj)] = val[q];
                        } else if (lane == 0) {
                            ctl->wslot[par][k * 4 + e] = val[q];
                        }
                        m[q] = kNegInf;
                        am[q] = -1;
                    }
                }
                buf += w.mt;
                if (closes && (a.lq_pad > 32 || (a.lq_pad == 32 && chunked))) {
                    // The warps' partial sums of a query are added in slot order by one
                    // thread after a rendezvous of the warps that wrote them: only the
                    // owning warpgroup when every query lies inside one M-tile, else all
                    // epilogue warps. The slots alternate between two halves by document,
                    // so one rendezvous per document keeps a half from being rewritten
                    // before it is read (its next writer has passed the rendezvous that
                    // its reader reaches only after reading).
                    const int32_t wpq = a.lq_pad / 32;  // warps per query (capped by the block)
                    const int32_t rows_w = (rb.row_end - rb.row0) / 32;
                    const float* ws = ctl->wslot[par];
                    auto sum_query = [&](int32_t qi) {
                        const int32_t wb = qi * wpq;
                        const int32_t we = min(wb + wpq, rows_w);
                        float sum = 0.f;
                        for (int32_t ww = wb; ww < we; ++ww) sum += ws[ww];
                        const int32_t i = rb.q0 + qi;
                        if (chunked) a.partial[(static_cast<int64_t>(rb.chunk) * a.nq + i) * a.nd + tw.oj] = sum;
                        else a.scores[out_index(a, i, tw.oj)] = sum;
                    };
                    if (kBM % a.lq_pad == 0) {
                        if (g < w.mt) {
                            if (!epi_sync(a, ctl, &ctl->epi_bar_g[g], grp_phase)) { ok = false; break; }
                            const int32_t qpm = kBM / a.lq_pad;  // queries per M-tile
                            const int32_t tg = e * 32 + lane;
#pragma unroll
                            for (int q = 0; q < kKPer; ++q) {
                                const int32_t qi = (g + kEpiGroups * q) * qpm + tg;
                                if (tg < qpm && qi < rb.nqb) sum_query(qi);
                            }
                        }
                    } else {
                        if (!epi_sync(a, ctl, &ctl->epi_bar, epi_phase)) { ok = false; break; }
                        if (et < rb.nqb) sum_query(et);
                    }
                }
                if (closes) par ^= 1u;
            }
        }
    }


    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();  // no CTA leaves while its pair may still touch it
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc<kG>(tmem_base, kNAcc * kBN);
    }
}

}  // namespace maxsim
