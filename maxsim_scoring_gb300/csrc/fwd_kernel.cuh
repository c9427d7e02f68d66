// Fused MaxSim forward for sm_103a: TMA -> tcgen05.mma -> TMEM -> fused
// mask / running max / argmax / sum epilogue. The [rows, doc tokens]
// similarity tile exists only in tensor memory and registers.
//
// Work decomposition (one persistent CTA per SM):
//  * Query rows are flattened: row r = i * lq_pad + s. A "row block" holds up
//    to 4 M-tiles of 128 rows that stay resident in shared memory. A query
//    longer than a row block is split into chunks whose partial scores are
//    summed afterwards ("late-interaction-kernels" design notes, "Long-query
//    chunking"; the sum of maxima decomposes over query tokens).
//  * Documents are packed token rows (dense D is the special case
//    cu[j] = j * Ld). A "doc range" is a run of whole documents holding about
//    total_d / n_dr tokens. A work unit is (row block, doc range).
//  * Tiles of BN = 128 consecutive document tokens stream through a shared
//    memory ring by TMA. A tile may span several documents: the epilogue folds
//    each document's columns separately, so no MMA work is spent on padding
//    ("Flash-MaxSim" Sec. 4.3.2: work proportional to the real tokens).
//  * For every (tile, M-tile) one MMA chain S = Q_blk * D_tile^T (K = dim)
//    accumulates in one of four 128-column TMEM buffers; the epilogue warps
//    read it with tcgen05.ld while the tensor core fills the next buffer.
//
// Epilogue semantics ("late-interaction-kernels" notes, "Forward" and "Mask
// handling"; "Flash-MaxSim" Sec. 4.1.1):
//  * masked / out-of-document columns are -inf before the max;
//  * running max per query row: m <- max(m, tile max); argmax moves only on a
//    strictly greater tile max, and inside a tile the lowest column wins, so
//    the overall lowest index wins among equal maxima;
//  * at a document end: m <- 0 unless finite and the row is active, then the
//    rows of each query are summed (warp shuffles, then a fixed-order sum of
//    per-warp partials), so the scores are bitwise reproducible.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace maxsim {

constexpr int kBN = 128;          // document tokens per tile (MMA N)
constexpr int kBM = 128;          // query rows per M-tile (MMA M)
constexpr int kMaxMT = 4;         // M-tiles per row block
constexpr int kNAcc = 4;          // TMEM accumulator buffers (4 x 128 columns)
constexpr int kThreads = 256;     // warp 0 TMA, warp 1 MMA, warps 4-7 epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kAtomBytes = 128 * 128;  // one 128-row x 64-element (128 B) swizzled block

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
    int32_t rb_rows;      // rows per row block (multiple of 32, or of lq_pad if smaller)
    int32_t n_chunks;     // row blocks per query (> 1 only when lq_pad > rb_rows)
    int32_t n_rb;
    // documents (packed token rows)
    const int32_t* cu_d;  // [nd + 1] or NULL => cu[j] = j * ld
    int32_t nd;
    int32_t ld;
    int32_t total_d;
    const uint8_t* d_mask;  // [total_d] or NULL
    int32_t n_dr;         // document ranges
    int32_t n_units;      // n_rb * n_dr
    // outputs
    float* scores;        // [nq, nd]
    float* partial;       // [n_chunks, nq, nd] when n_chunks > 1
    int32_t* argmax;      // [nq * nd, lq_out] or NULL
    // operand geometry
    int32_t k_steps;      // dim / 16 MMA instructions per tile
    int32_t k_atoms;      // ceil(dim / 64) swizzled 64-element blocks per row
    int32_t stages;       // D ring depth
    int32_t q_slots;      // M-tiles of Q resident in shared memory (>= every row block's mt)
    uint32_t idesc;       // tcgen05 instruction descriptor
    int* status;          // device status word
    uint64_t timeout_ns;  // bound on any single wait
};

struct RowBlock {
    int32_t row0, row_end;  // global padded rows [row0, row_end)
    int32_t q0, nqb;        // first query, number of queries in the block
    int32_t chunk;          // chunk index within the query (0 if unchunked)
    int32_t mt;             // M-tiles to compute
};

__device__ __forceinline__ RowBlock row_block(const FwdArgs& a, int32_t rb) {
    RowBlock b;
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
    int32_t j0, j1;      // documents [j0, j1)
    int32_t tok0, tok1;  // their tokens [tok0, tok1)
    int32_t ntiles;
};

__device__ __forceinline__ Unit make_unit(const FwdArgs& a, int32_t u) {
    Unit w;
    int32_t rb = u % a.n_rb;
    int32_t dr = u / a.n_rb;
    w.rb = row_block(a, rb);
    w.j0 = range_first_doc(a, dr);
    w.j1 = range_first_doc(a, dr + 1);
    w.tok0 = doc_start(a, w.j0);
    w.tok1 = doc_start(a, w.j1);
    w.ntiles = w.tok1 > w.tok0 ? (w.tok1 - w.tok0 + kBN - 1) / kBN : 0;
    return w;
}

// Shared-memory control block (after the operand buffers).
struct SmemCtl {
    uint64_t q_full, q_empty;
    uint64_t d_full[8], d_empty[8];
    uint64_t acc_full[kNAcc], acc_empty[kNAcc];
    uint64_t mma_done;
    uint64_t epi_bar;  // rendezvous of the four epilogue warps
    uint32_t tmem_base;
    volatile int32_t abort;
    int32_t slot_doc[kBN];
    float wslot[kBN][kMaxMT * 4];
};

__device__ __forceinline__ void record_status(const FwdArgs& a, int code) {
    if (a.status) atomicCAS(a.status, 0, code);
}

// Bounded wait: gives up after timeout_ns (records the status and raises the
// CTA abort flag) or when another role has already aborted.
__device__ __forceinline__ bool wait_bar(const FwdArgs& a, SmemCtl* ctl, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (ctl->abort) return false;
            if (global_timer_ns() - t0 > a.timeout_ns) {
                ctl->abort = 1;
                record_status(a, kStatusTimeout);
                return false;
            }
        }
    }
}

// Bounded rendezvous of the four epilogue warps (an mbarrier phase per use),
// so that a warp that gave up on a wait can never strand the others.
__device__ __forceinline__ bool epi_sync(const FwdArgs& a, SmemCtl* ctl, uint32_t& phase) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&ctl->epi_bar));
    const bool ok = wait_bar(a, ctl, smem_u32(&ctl->epi_bar), phase);
    phase ^= 1u;
    return ok;
}

// ---------------------------------------------------------------- epilogue helpers

__device__ __forceinline__ float chunk_max(const float (&x)[32], float m) {
    float a0 = fmax3(x[0], x[1], x[2]), a1 = fmax3(x[3], x[4], x[5]), a2 = fmax3(x[6], x[7], x[8]);
    float a3 = fmax3(x[9], x[10], x[11]), a4 = fmax3(x[12], x[13], x[14]), a5 = fmax3(x[15], x[16], x[17]);
    float a6 = fmax3(x[18], x[19], x[20]), a7 = fmax3(x[21], x[22], x[23]), a8 = fmax3(x[24], x[25], x[26]);
    float a9 = fmax3(x[27], x[28], x[29]), a10 = fmax3(x[30], x[31], m);
    float b0 = fmax3(a0, a1, a2), b1 = fmax3(a3, a4, a5), b2 = fmax3(a6, a7, a8), b3 = fmax3(a9, a10, b0);
    return fmax3(b1, b2, b3);
}

// Fold columns whose bit is set in `valid` into (m, am). `col0` is the index,
// relative to the document start, of column 0 of the chunk.
template <bool kArg>
__device__ __forceinline__ void fold_chunk(const float (&x)[32], uint32_t valid, int32_t col0, float& m,
                                           int32_t& am) {
    const float kNegInf = __int_as_float(0xff800000u);
    if constexpr (!kArg) {
        if (valid == 0xFFFFFFFFu) {
            m = chunk_max(x, m);
        } else {
            float y[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = (valid >> e) & 1u ? x[e] : kNegInf;
            m = chunk_max(y, m);
        }
    } else {
        float y[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) y[e] = (valid >> e) & 1u ? x[e] : kNegInf;
        const float cm = chunk_max(y, kNegInf);
        const bool upd = cm > m;
        if (__any_sync(0xFFFFFFFFu, upd)) {
            int32_t idx = 31;
#pragma unroll
            for (int e = 30; e >= 0; --e) idx = (y[e] == cm) ? e : idx;
            if (upd) {
                am = col0 + idx;
                m = cm;
            }
        }
    }
}

__device__ __forceinline__ uint32_t seg_bits(int32_t lo, int32_t hi) {  // bits [lo, hi), 0 <= lo < hi <= 32
    uint32_t upto = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
    return upto & ~((1u << lo) - 1u);
}

// ---------------------------------------------------------------- the kernel

template <bool kArg, bool kDMask>
__global__ void __launch_bounds__(kThreads, 1)
    maxsim_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_d,
                      const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int32_t q_tile_bytes = a.k_atoms * kAtomBytes;   // one 128-row M-tile of Q
    const int32_t d_stage_bytes = a.k_atoms * kAtomBytes;  // one 128-token tile of D
    uint8_t* sQ = smem;
    uint8_t* sD = smem + a.q_slots * q_tile_bytes;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(sD + a.stages * d_stage_bytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->q_full), 1);
        mbar_init(smem_u32(&ctl->q_empty), 1);
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(smem_u32(&ctl->d_full[s]), 1);
            mbar_init(smem_u32(&ctl->d_empty[s]), 1);
        }
        for (int b = 0; b < kNAcc; ++b) {
            mbar_init(smem_u32(&ctl->acc_full[b]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[b]), 4);
        }
        mbar_init(smem_u32(&ctl->mma_done), 1);
        mbar_init(smem_u32(&ctl->epi_bar), 4);
        ctl->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_d);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kNAcc * kBN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();
            int32_t stage = 0;
            uint32_t phase = 0;
            uint32_t q_phase = 0;
            bool first_unit = true;
            int64_t issued = 0;
            for (int32_t u = blockIdx.x; u < a.n_units; u += gridDim.x) {
                Unit w = make_unit(a, u);
                if (!first_unit) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->q_empty), q_phase)) break;
                    q_phase ^= 1u;
                }
                first_unit = false;
                uint32_t qbar = smem_u32(&ctl->q_full);
                mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(w.rb.mt * q_tile_bytes));
                for (int32_t k = 0; k < w.rb.mt; ++k)
                    for (int32_t ka = 0; ka < a.k_atoms; ++ka)
                        tma_load_2d(smem_u32(sQ + k * q_tile_bytes + ka * kAtomBytes), &tm_q, qbar, ka * 64,
                                    w.rb.row0 + k * kBM);
                bool ok = true;
                for (int32_t t = 0; t < w.ntiles; ++t) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->d_empty[stage]), phase ^ 1u)) { ok = false; break; }
                    uint32_t dbar = smem_u32(&ctl->d_full[stage]);
                    mbar_arrive_expect_tx(dbar, static_cast<uint32_t>(d_stage_bytes));
                    for (int32_t ka = 0; ka < a.k_atoms; ++ka)
                        tma_load_2d_hint(smem_u32(sD + stage * d_stage_bytes + ka * kAtomBytes), &tm_d, dbar,
                                         ka * 64, w.tok0 + t * kBN, pol_stream);
                    ++issued;
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            if (ctl->abort) {
                // Let every copy still in flight land before the CTA exits.
                int64_t outstanding = issued < a.stages ? issued : a.stages;
                int32_t s = stage;
                uint32_t ph = phase;
                for (int64_t n = 0; n < outstanding; ++n) {
                    if (--s < 0) { s = a.stages - 1; ph ^= 1u; }
                    uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(smem_u32(&ctl->d_full[s]), ph) && global_timer_ns() - t0 < a.timeout_ns) {}
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int32_t stage = 0;
            uint32_t phase = 0;
            int32_t acc = 0;
            uint32_t acc_phase = 0;
            uint32_t q_phase = 0;
            bool ok = true;
            for (int32_t u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
                Unit w = make_unit(a, u);
                if (!wait_bar(a, ctl, smem_u32(&ctl->q_full), q_phase)) break;
                q_phase ^= 1u;
                tc_fence_after();
                for (int32_t t = 0; t < w.ntiles; ++t) {
                    if (!wait_bar(a, ctl, smem_u32(&ctl->d_full[stage]), phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_base = smem_u32(sD + stage * d_stage_bytes);
                    for (int32_t k = 0; k < w.rb.mt; ++k) {
                        if (!wait_bar(a, ctl, smem_u32(&ctl->acc_empty[acc]), acc_phase ^ 1u)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t q_base = smem_u32(sQ + k * q_tile_bytes);
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                        for (int32_t ks = 0; ks < a.k_steps; ++ks) {
                            const uint32_t off = static_cast<uint32_t>((ks >> 2) * kAtomBytes + (ks & 3) * 32);
                            mma_f16_ss(d_tmem, sdesc_k_sw128(q_base + off), sdesc_k_sw128(d_base + off), a.idesc,
                                       ks > 0 ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&ctl->acc_full[acc]));
                        if (++acc == kNAcc) { acc = 0; acc_phase ^= 1u; }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&ctl->d_empty[stage]));
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctl->q_empty));
            }
            // Drain: wait until every MMA issued above has completed.
            mma_commit(smem_u32(&ctl->mma_done));
            uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&ctl->mma_done), 0) && global_timer_ns() - t0 < a.timeout_ns) {}
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const float kNegInf = __int_as_float(0xff800000u);
        const int e = warp - kEpiWarp0;      // TMEM lane quadrant
        const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
        int32_t acc = 0;
        uint32_t acc_phase = 0;
        uint32_t epi_phase = 0;
        bool ok = true;
        for (int32_t u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
            const Unit w = make_unit(a, u);
            const RowBlock& rb = w.rb;
            // per-row facts for each M-tile this thread reads
            int32_t row_i[kMaxMT], row_s[kMaxMT];
            bool in_rb[kMaxMT], real[kMaxMT], active[kMaxMT];
#pragma unroll
            for (int k = 0; k < kMaxMT; ++k) {
                int32_t r = rb.row0 + k * kBM + e * 32 + lane;
                in_rb[k] = k < rb.mt && r < rb.row_end;
                row_i[k] = r / a.lq_pad;
                row_s[k] = r - row_i[k] * a.lq_pad;
                real[k] = in_rb[k] && (a.q_real == nullptr || a.q_real[r] != 0);
                active[k] = real[k] && (a.q_active == nullptr || a.q_active[r] != 0);
            }
            const bool chunked = a.n_chunks > 1;
            // empty documents: score 0 and argmax -1, written up front
            for (int32_t j = w.j0 + et; j < w.j1; j += 128) {
                if (doc_start(a, j + 1) != doc_start(a, j)) continue;
                for (int32_t q = 0; q < rb.nqb; ++q) {
                    int32_t i = rb.q0 + q;
                    if (chunked) a.partial[(static_cast<int64_t>(rb.chunk) * a.nq + i) * a.nd + j] = 0.f;
                    else a.scores[static_cast<int64_t>(i) * a.nd + j] = 0.f;
                }
                if (kArg) {
                    for (int32_t r = rb.row0; r < rb.row_end; ++r) {
                        int32_t i = r / a.lq_pad, s = r - (r / a.lq_pad) * a.lq_pad;
                        if (s < a.lq_out) a.argmax[(static_cast<int64_t>(i) * a.nd + j) * a.lq_out + s] = -1;
                    }
                }
            }
            float m[kMaxMT];
            int32_t am[kMaxMT];
#pragma unroll
            for (int k = 0; k < kMaxMT; ++k) { m[k] = kNegInf; am[k] = -1; }
            // document cursor: first non-empty document at or after j0
            int32_t cj = w.j0;
            int32_t cds = w.tok0;
            int32_t cde = w.j0 < w.j1 ? doc_start(a, w.j0 + 1) : w.tok0;

            for (int32_t t = 0; t < w.ntiles && ok; ++t) {
                const int32_t ts = w.tok0 + t * kBN;
                const int32_t te = min(ts + kBN, w.tok1);
                uint32_t dmw[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (kDMask) {
                        int32_t col = ts + c * 32 + lane;
                        dmw[c] = __ballot_sync(0xFFFFFFFFu, col < te && col < a.total_d && a.d_mask[col] != 0);
                    } else {
                        dmw[c] = 0xFFFFFFFFu;
                    }
                }
                int32_t nslot = 0;
                int32_t end_j = cj, end_ds = cds, end_de = cde;
#pragma unroll
                for (int k = 0; k < kMaxMT; ++k) {
                    if (k >= rb.mt) break;
                    if (!wait_bar(a, ctl, smem_u32(&ctl->acc_full[acc]), acc_phase)) { ok = false; break; }
                    tc_fence_after();
                    float v[4][32];
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(e * 32) << 16) +
                                           static_cast<uint32_t>(acc * kBN);
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(taddr + c * 32, v[c]);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[acc]));
                    if (++acc == kNAcc) { acc = 0; acc_phase ^= 1u; }

                    // walk the documents covered by this tile
                    int32_t jj = cj, ds = cds, de = cde;
                    int32_t pos = ts;
                    int32_t slot = 0;
                    auto flush = [&](int32_t jdoc) {
                        const bool has = m[k] > kNegInf;
                        if (kArg && in_rb[k] && row_s[k] < a.lq_out)
                            a.argmax[(static_cast<int64_t>(row_i[k]) * a.nd + jdoc) * a.lq_out + row_s[k]] =
                                (real[k] && has) ? am[k] : -1;
                        float val = (active[k] && has) ? m[k] : 0.f;
                        if (a.lq_pad >= 32) {
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xFFFFFFFFu, val, o);
                            if (lane == 0) ctl->wslot[slot][k * 4 + e] = val;
                            if (k == 0 && e == 0 && lane == 0) ctl->slot_doc[slot] = jdoc;
                        } else {
                            for (int o = a.lq_pad >> 1; o > 0; o >>= 1) val += __shfl_xor_sync(0xFFFFFFFFu, val, o);
                            if (in_rb[k] && (lane & (a.lq_pad - 1)) == 0)
                                a.scores[static_cast<int64_t>(row_i[k]) * a.nd + jdoc] = val;
                        }
                        ++slot;
                        m[k] = kNegInf;
                        am[k] = -1;
                    };
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int32_t cs = ts + c * 32;
                        if (cs < te) {
                            const int32_t ce = min(cs + 32, te);
                            while (true) {
                                while (jj < w.j1 && de <= pos) {
                                    if (de > ds) flush(jj);
                                    ++jj;
                                    ds = de;
                                    de = jj < w.j1 ? doc_start(a, jj + 1) : de;
                                }
                                if (jj >= w.j1 || pos >= ce) break;
                                const int32_t hi = min(de, ce);
                                const uint32_t valid = seg_bits(pos - cs, hi - cs) & dmw[c];
                                fold_chunk<kArg>(v[c], valid, cs - ds, m[k], am[k]);
                                pos = hi;
                            }
                        }
                    }
                    while (jj < w.j1 && de <= pos) {
                        if (de > ds) flush(jj);
                        ++jj;
                        ds = de;
                        de = jj < w.j1 ? doc_start(a, jj + 1) : de;
                    }
                    nslot = slot;
                    end_j = jj;
                    end_ds = ds;
                    end_de = de;
                }
                if (!ok) break;
                cj = end_j;
                cds = end_ds;
                cde = end_de;
                if (a.lq_pad >= 32 && nslot > 0) {
                    if (!epi_sync(a, ctl, epi_phase)) { ok = false; break; }
                    const int32_t wpq = a.lq_pad / 32;  // warps per query (capped by the block)
                    for (int32_t x = et; x < nslot * rb.nqb; x += 128) {
                        const int32_t sl = x / rb.nqb, q = x - (x / rb.nqb) * rb.nqb;
                        const int32_t wb = q * wpq;
                        const int32_t we = min(wb + wpq, (rb.row_end - rb.row0) / 32);
                        float sum = 0.f;
                        for (int32_t ww = wb; ww < we; ++ww) sum += ctl->wslot[sl][ww];
                        const int32_t jdoc = ctl->slot_doc[sl];
                        const int32_t i = rb.q0 + q;
                        if (chunked) a.partial[(static_cast<int64_t>(rb.chunk) * a.nq + i) * a.nd + jdoc] = sum;
                        else a.scores[static_cast<int64_t>(i) * a.nd + jdoc] = sum;
                    }
                    if (!epi_sync(a, ctl, epi_phase)) { ok = false; break; }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, kNAcc * kBN);
    }
}

}  // namespace maxsim
