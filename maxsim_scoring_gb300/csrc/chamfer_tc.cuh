// Nearest-point search of the Chamfer distance ("Flash-MaxSim" paper, Sec.
// 4.2.4) on the 5th-generation tensor cores, for points of up to 4
// coordinates.
//
// The search value d'(x, y) = ||y||^2 - 2 <x, y> (the squared distance minus
// the constant ||x||^2) is one inner product of augmented rows. fp32 values are
// carried by a split into two tf32 parts (v = v_hi + v_lo, each a tf32 number;
// the product of two tf32 numbers is exact in fp32):
//   source row  [x_hi, 1,    x_hi, 1,    x_lo]          (dim + 1, dim + 1, dim)
//   target row  [a_hi, n_hi, a_lo, n_lo, a_hi]          a = -2 y, n = ||y||^2
//   dot         = x_hi.a_hi + n_hi + x_hi.a_lo + n_lo + x_lo.a_hi
//               = d'(x, y) up to x_lo.a_lo and the tf32 rounding of the low parts
//               (relative size about 2^-21), with K = 16 (3 dim + 2 <= 16).
// One tcgen05.mma kind::tf32 (M = 128 sources, N = 256 targets, K = 8, twice)
// fills a 128 x 256 fp32 block of d' in tensor memory; the epilogue reads it
// back with tcgen05.ld.red.min (the minimum of each 32-column chunk comes out
// of the load) and keeps, per source, the smallest chunk minimum and the chunk
// (strict <: the earlier chunk keeps a tie). The [N, M] table is never
// formed. chamfer_tc_merge_kernel then takes the minimum over the spans of
// targets and, inside the winning chunk, the first target at the smallest
// distance sum_k (x_k - y_k)^2 computed directly in fp32 (a search over 32
// columns per source instead of one per improving chunk in the epilogue).
//
// Roles (one CTA of 640 threads per SM): warp 0 loads operand tiles by TMA
// (8 source M-tiles per work item, once; a 4-stage ring of 256-target tiles),
// warp 1 issues the MMAs into two 256-column accumulators, warps 4-19 (four
// warpgroups, each a 64-column quarter of every accumulator) reduce. A work
// item is (span of targets, direction, pair of sets, 1,024 sources); items run
// span-major so that the short last spans come last. Per item and source the
// kernel writes (minimum, chunk) of its span.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace maxsim {

constexpr int kTcK = 16;               // tf32 elements per augmented row (64 bytes)
constexpr int kTcRowBytes = kTcK * 4;
constexpr int kTcM = 128;              // sources per M-tile
constexpr int kTcMT = 8;               // M-tiles per work item
constexpr int kTcSources = kTcM * kTcMT;
constexpr int kTcN = 256;              // targets per N-tile
constexpr int kTcStages = 4;
constexpr int kTcSpanTiles = 32;       // N-tiles per work item (8,192 targets)
constexpr int kTcSpan = kTcSpanTiles * kTcN;
constexpr int kTcEpiWarp0 = 4;
constexpr int kTcEpiWarps = 16;
constexpr int kTcThreads = (kTcEpiWarp0 + kTcEpiWarps) * 32;
constexpr int kTcMaxDim = 4;           // 3 dim + 2 <= kTcK
constexpr float kTcPadNorm = 1e30f;    // ||y||^2 of padding targets: never the minimum
constexpr int kTcATile = kTcM * kTcRowBytes;    // 8 KB
constexpr int kTcBTile = kTcN * kTcRowBytes;    // 16 KB
static_assert(3 * kTcMaxDim + 2 <= kTcK, "augmented rows");

struct ChamferTcArgs {
    int64_t nx[2], ny[2];        // direction 0: P -> Q, 1: Q -> P
    int64_t s_rows[2], t_rows[2];  // padded operand rows per set (sources: x 1,024; targets: x 256)
    int64_t n_sb[2], n_span[2];
    int64_t B;
    int64_t items;
    float* part_best[2];         // [n_span][B * nx]: smallest chunk minimum of d'
    int32_t* part_idx[2];        // [n_span][B * nx]: its 32-target chunk (global), -1 if none
    int* status;
    uint64_t timeout_ns;
};

struct TcSmemCtl {
    uint64_t a_full, a_empty;
    uint64_t b_full[kTcStages], b_empty[kTcStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t epi_bar, mma_done;
    uint32_t tmem_base;
    volatile int32_t abort;
};

// ---------------------------------------------------------------- operand prep

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Augmented rows of every point of a set of B x n points X [B, n, dim]:
// source form into S [B, s_rows, kTcK], target form into T [B, t_rows, kTcK];
// rows past n are zero sources and padding targets.
__global__ void chamfer_tc_prep_kernel(const float* __restrict__ X, int64_t B, int64_t n, int32_t dim,
                                       int64_t s_rows, int64_t t_rows, float* __restrict__ S,
                                       float* __restrict__ T) {
    const int64_t rows = B * (s_rows > t_rows ? s_rows : t_rows);
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < rows;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t per = s_rows > t_rows ? s_rows : t_rows;
        const int64_t b = e / per, r = e - b * per;
        float x[kTcMaxDim];
        const bool real = r < n;
#pragma unroll
        for (int k = 0; k < kTcMaxDim; ++k) x[k] = (real && k < dim) ? X[(b * n + r) * dim + k] : 0.f;
        float srow[kTcK], trow[kTcK];
#pragma unroll
        for (int k = 0; k < kTcK; ++k) srow[k] = trow[k] = 0.f;
        // ||y||^2 in the order the fp32 kernels use
        float nrm = __fmul_rn(x[0], x[0]);
#pragma unroll
        for (int k = 1; k < kTcMaxDim; ++k)
            if (k < dim) nrm = __fmaf_rn(x[k], x[k], nrm);
        const float n_hi = to_tf32(nrm), n_lo = to_tf32(__fsub_rn(nrm, n_hi));
#pragma unroll
        for (int k = 0; k < kTcMaxDim; ++k) {
            if (k < dim) {
                const float xh = to_tf32(x[k]), xl = to_tf32(__fsub_rn(x[k], xh));
                const float a = __fmul_rn(-2.f, x[k]);
                const float ah = to_tf32(a), al = to_tf32(__fsub_rn(a, ah));
                srow[k] = xh;
                srow[dim + 1 + k] = xh;
                srow[2 * dim + 2 + k] = xl;
                trow[k] = ah;
                trow[dim + 1 + k] = al;
                trow[2 * dim + 2 + k] = ah;
            }
        }
        if (real) {
            srow[dim] = 1.f;
            srow[2 * dim + 1] = 1.f;
            trow[dim] = n_hi;
            trow[2 * dim + 1] = n_lo;
        } else {
            trow[dim] = kTcPadNorm;  // padding target: d' = 1e30 against any real source
        }
        if (r < s_rows) {
            float4* dst = reinterpret_cast<float4*>(S + (b * s_rows + r) * kTcK);
#pragma unroll
            for (int v = 0; v < kTcK / 4; ++v)
                dst[v] = make_float4(srow[4 * v], srow[4 * v + 1], srow[4 * v + 2], srow[4 * v + 3]);
        }
        if (r < t_rows) {
            float4* dst = reinterpret_cast<float4*>(T + (b * t_rows + r) * kTcK);
#pragma unroll
            for (int v = 0; v < kTcK / 4; ++v)
                dst[v] = make_float4(trow[4 * v], trow[4 * v + 1], trow[4 * v + 2], trow[4 * v + 3]);
        }
    }
}

// ---------------------------------------------------------------- kernel helpers

// K-major operand with the 64-byte swizzle: 64-byte rows, 8-row groups 512
// bytes apart, base 512-byte aligned; swizzle mode 4 (64 B) in bits [61,64).
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(512 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(4) << 61;
    return d;
}

// kind::tf32, fp32 D, both operands K-major: D format 1, A / B format 2 (tf32).
__host__ __device__ constexpr uint32_t idesc_tf32_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Two K = 8 steps (K = 16) of D (+)= A * B^T, issued by one elected lane.
__device__ __forceinline__ void mma_tf32_k16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, b1;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "setp.ne.b32 q, 0, 0;\n\t"
        "add.s64 a1, %1, 2;\n\t"
        "add.s64 b1, %2, 2;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, q;\n\t"
        "setp.eq.b32 q, 0, 0;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], a1, b1, %3, q;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc)
        : "memory");
}

// 32 fp32 columns of this thread's TMEM lane and their minimum (NaN ignored).
__device__ __forceinline__ float tmem_ldmin32(uint32_t taddr, float (&v)[32]) {
    uint32_t* u = reinterpret_cast<uint32_t*>(v);
    float m;
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.min.f32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
          "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
          "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]),
          "=f"(m)
        : "r"(taddr));
    return m;
}

__device__ __forceinline__ bool tc_wait(const ChamferTcArgs& a, TcSmemCtl* ctl, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (ctl->abort) return false;
            if (global_timer_ns() - t0 > a.timeout_ns) {
                ctl->abort = 1;
                if (a.status) atomicCAS(a.status, 0, 4);
                return false;
            }
        }
    }
}

// tc_wait for a warp running warp-uniform code (collective tcgen05 and
// elect.sync follow): every lane polls, and the warp agrees on the outcome.
__device__ __forceinline__ bool tc_wait_warp(const ChamferTcArgs& a, TcSmemCtl* ctl, uint32_t bar, uint32_t parity) {
    const bool ok = tc_wait(a, ctl, bar, parity);
    return __all_sync(0xFFFFFFFFu, ok);
}

struct TcItem {
    int dir;
    int64_t span, b, sb;
};

__device__ __forceinline__ TcItem tc_item(const ChamferTcArgs& a, int64_t it) {
    // span-major: every pair of sets and source block of span 0, then span 1, ...
    const int64_t per0 = a.B * a.n_sb[0], per1 = a.B * a.n_sb[1];
    TcItem w{};
    for (int64_t sp = 0;; ++sp) {
        const int64_t c0 = sp < a.n_span[0] ? per0 : 0, c1 = sp < a.n_span[1] ? per1 : 0;
        if (it < c0) {
            w.dir = 0;
            w.span = sp;
            w.b = it / a.n_sb[0];
            w.sb = it - w.b * a.n_sb[0];
            return w;
        }
        it -= c0;
        if (it < c1) {
            w.dir = 1;
            w.span = sp;
            w.b = it / a.n_sb[1];
            w.sb = it - w.b * a.n_sb[1];
            return w;
        }
        it -= c1;
    }
}

// N-tiles of a work item (the last span of a set may be short).
__device__ __forceinline__ int32_t tc_tiles(const ChamferTcArgs& a, const TcItem& w) {
    const int64_t ny = w.dir ? a.ny[1] : a.ny[0];
    const int64_t t0 = w.span * kTcSpan;
    const int64_t left = ny - t0 < kTcSpan ? ny - t0 : kTcSpan;
    return static_cast<int32_t>((left + kTcN - 1) / kTcN);
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(kTcThreads, 1)
    chamfer_tc_kernel(const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_t0,
                      const __grid_constant__ CUtensorMap tm_s1, const __grid_constant__ CUtensorMap tm_t1,
                      const ChamferTcArgs a) {
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                                  // kTcMT M-tiles
    uint8_t* sB = sA + kTcMT * kTcATile;                 // kTcStages N-tiles
    float* sBest = reinterpret_cast<float*>(sB + kTcStages * kTcBTile);          // [4 wg][kTcSources]
    int32_t* sIdx = reinterpret_cast<int32_t*>(sBest + 4 * kTcSources);          // [4 wg][kTcSources]
    TcSmemCtl* ctl = reinterpret_cast<TcSmemCtl*>(sIdx + 4 * kTcSources);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl->a_full), 1);
        mbar_init(smem_u32(&ctl->a_empty), 1);
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_u32(&ctl->b_full[s]), 1);
            mbar_init(smem_u32(&ctl->b_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&ctl->acc_full[s]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[s]), kTcEpiWarps);
        }
        mbar_init(smem_u32(&ctl->epi_bar), kTcEpiWarps);
        mbar_init(smem_u32(&ctl->mma_done), 1);
        ctl->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_s0);
        tma_prefetch_desc(&tm_t0);
        tma_prefetch_desc(&tm_s1);
        tma_prefetch_desc(&tm_t1);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(&ctl->tmem_base), 2 * kTcN);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int32_t stage = 0;
            uint32_t phase = 0, a_phase = 0;
            int64_t issued = 0;
            bool ok = true, first = true;
            for (int64_t it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
                const TcItem w = tc_item(a, it);
                const CUtensorMap* ms = w.dir ? &tm_s1 : &tm_s0;
                const CUtensorMap* mt = w.dir ? &tm_t1 : &tm_t0;
                if (!first) {
                    if (!tc_wait(a, ctl, smem_u32(&ctl->a_empty), a_phase)) break;
                    a_phase ^= 1u;
                }
                first = false;
                const uint32_t abar = smem_u32(&ctl->a_full);
                mbar_arrive_expect_tx(abar, static_cast<uint32_t>(kTcMT * kTcATile));
                const int64_t srow0 = w.b * (w.dir ? a.s_rows[1] : a.s_rows[0]) + w.sb * kTcSources;
                for (int k = 0; k < kTcMT; ++k)
                    tma_load_2d(smem_u32(sA + k * kTcATile), ms, abar, 0, static_cast<int32_t>(srow0 + k * kTcM));
                const int32_t tiles = tc_tiles(a, w);
                const int64_t trow0 = w.b * (w.dir ? a.t_rows[1] : a.t_rows[0]) + w.span * kTcSpan;
                for (int32_t n = 0; n < tiles; ++n) {
                    if (!tc_wait(a, ctl, smem_u32(&ctl->b_empty[stage]), phase ^ 1u)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&ctl->b_full[stage]);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(kTcBTile));
                    tma_load_2d(smem_u32(sB + stage * kTcBTile), mt, fb, 0, static_cast<int32_t>(trow0 + n * kTcN));
                    ++issued;
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (ctl->abort) {
                // let the copies in flight land before the CTA exits
                const int64_t outstanding = issued < kTcStages ? issued : kTcStages;
                int32_t s = stage;
                uint32_t ph = phase;
                for (int64_t n = 0; n < outstanding; ++n) {
                    if (--s < 0) { s = kTcStages - 1; ph ^= 1u; }
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(smem_u32(&ctl->b_full[s]), ph) && global_timer_ns() - t0 < a.timeout_ns) {}
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int32_t stage = 0;
        uint32_t phase = 0, a_phase = 0;
        int64_t q = 0;  // accumulator uses so far
        bool ok = true;
        const uint64_t a_desc0 = sdesc_k_sw64(smem_u32(sA));
        const uint64_t b_desc0 = sdesc_k_sw64(smem_u32(sB));
        constexpr uint32_t idesc = idesc_tf32_f32(kTcM, kTcN);
        for (int64_t it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
            const TcItem w = tc_item(a, it);
            if (!tc_wait_warp(a, ctl, smem_u32(&ctl->a_full), a_phase)) break;
            a_phase ^= 1u;
            tc_fence_after();
            const int32_t tiles = tc_tiles(a, w);
            for (int32_t n = 0; n < tiles && ok; ++n) {
                if (!tc_wait_warp(a, ctl, smem_u32(&ctl->b_full[stage]), phase)) { ok = false; break; }
                tc_fence_after();
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * kTcBTile) >> 4);
                for (int k = 0; k < kTcMT; ++k, ++q) {
                    const int buf = static_cast<int>(q & 1);
                    const uint32_t acc_phase = static_cast<uint32_t>((q >> 1) & 1);
                    if (!tc_wait_warp(a, ctl, smem_u32(&ctl->acc_empty[buf]), acc_phase ^ 1u)) { ok = false; break; }
                    tc_fence_after();
                    mma_tf32_k16(tmem_base + static_cast<uint32_t>(buf * kTcN),
                                 a_desc0 + static_cast<uint64_t>((k * kTcATile) >> 4), bd, idesc);
                    mma_commit_elect<1>(smem_u32(&ctl->acc_full[buf]));
                }
                if (!ok) break;
                mma_commit_elect<1>(smem_u32(&ctl->b_empty[stage]));
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit_elect<1>(smem_u32(&ctl->a_empty));
        }
        // drain: every MMA issued above has completed before TMEM is freed
        mma_commit_elect<1>(smem_u32(&ctl->mma_done), 1);
        if (lane == 0) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&ctl->mma_done), 0) && global_timer_ns() - t0 < a.timeout_ns) {}
        }
        __syncwarp();
    } else if (warp >= kTcEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - kTcEpiWarp0;
        const int wg = ew >> 2;            // column quarter of every accumulator
        const int quarter = warp & 3;      // TMEM lanes 32 * quarter ..
        const int row = quarter * 32 + lane;
        int64_t q = 0;
        uint32_t epi_phase = 0;
        bool ok = true;
        const float kInf = __int_as_float(0x7f800000);
        for (int64_t it = blockIdx.x; it < a.items && ok; it += gridDim.x) {
            const TcItem w = tc_item(a, it);
            const int32_t tiles = tc_tiles(a, w);
            // this thread's running (minimum, chunk) per M-tile lives in its own
            // slots of the merge scratch (registers go to the TMEM loads)
            float* my_best = sBest + wg * kTcSources + row;
            int32_t* my_chunk = sIdx + wg * kTcSources + row;
#pragma unroll
            for (int k = 0; k < kTcMT; ++k) {
                my_best[k * kTcM] = kInf;
                my_chunk[k * kTcM] = -1;
            }
            const int64_t col_base = w.span * kTcSpan + wg * 64;
            for (int32_t n = 0; n < tiles && ok; ++n) {
#pragma unroll 1
                for (int k = 0; k < kTcMT; ++k) {
                    const int buf = static_cast<int>((q + k) & 1);
                    const uint32_t acc_phase = static_cast<uint32_t>(((q + k) >> 1) & 1);
                    if (!tc_wait_warp(a, ctl, smem_u32(&ctl->acc_full[buf]), acc_phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                           static_cast<uint32_t>(buf * kTcN + wg * 64);
                    const int32_t chunk0 = static_cast<int32_t>((col_base + static_cast<int64_t>(n) * kTcN) >> 5);
                    float v0[32], v1[32];
                    const float m0 = tmem_ldmin32(taddr, v0);
                    const float m1 = tmem_ldmin32(taddr + 32, v1);
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
                    // strict: the earlier chunk keeps a tie
                    const float cur = my_best[k * kTcM];
                    const float mm = fminf(m0, m1);
                    if (mm < cur) {
                        my_best[k * kTcM] = mm;
                        my_chunk[k * kTcM] = m0 <= m1 ? chunk0 : chunk0 + 1;
                    }
                }
                q += kTcMT;
            }
            if (!ok) break;
            // merge the four column quarters: (value, chunk), the lower chunk on ties
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->epi_bar));
            if (!tc_wait_warp(a, ctl, smem_u32(&ctl->epi_bar), epi_phase)) break;
            epi_phase ^= 1u;
            const int64_t nx = w.dir ? a.nx[1] : a.nx[0];
            const int64_t base = w.span * a.B * nx + w.b * nx;
            float* pb = (w.dir ? a.part_best[1] : a.part_best[0]) + base;
            int32_t* pi = (w.dir ? a.part_idx[1] : a.part_idx[0]) + base;
            for (int s = ew * 32 + lane; s < kTcSources; s += kTcEpiWarps * 32) {
                float v = sBest[s];
                int32_t ix = sIdx[s];
#pragma unroll
                for (int g = 1; g < 4; ++g) {
                    const float ov = sBest[g * kTcSources + s];
                    const int32_t oi = sIdx[g * kTcSources + s];
                    if (ov < v || (ov == v && oi >= 0 && (ix < 0 || oi < ix))) {
                        v = ov;
                        ix = oi;
                    }
                }
                const int64_t src = w.sb * kTcSources + s;
                if (src < nx) {
                    pb[src] = v;
                    pi[src] = ix;
                }
            }
            // the scratch is free again once every warp has read it
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->epi_bar));
            if (!tc_wait_warp(a, ctl, smem_u32(&ctl->epi_bar), epi_phase)) break;
            epi_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc<1>(tmem_base, 2 * kTcN);
    }
}

// Minimum over the spans (strict <: the earlier span keeps a tie), then the
// first target of the winning 32-target chunk at the smallest distance
// sum_k (x_k - y_k)^2 (fp32, the fixed order of the other kernels), its
// index, its distance, and the block's share of the loss (fixed-order double
// sums). A warp takes 32 sources: lane l merges the spans of source l; then,
// source by source, lane t computes the distance to target t of the chunk.
// Grid (blocks of 256 sources, B, 2).
__global__ void __launch_bounds__(256) chamfer_tc_merge_kernel(const float* __restrict__ P,
                                                               const float* __restrict__ Q, int32_t dim,
                                                               ChamferTcArgs t, ChamferFwdArgs a) {
    const int dir = blockIdx.z;
    const int64_t b = blockIdx.y;
    const int64_t nx = dir ? a.nx[1] : a.nx[0], ny = dir ? a.ny[1] : a.ny[0];
    const int64_t n_mblk = dir ? a.n_mblk[1] : a.n_mblk[0], n_span = dir ? t.n_span[1] : t.n_span[0];
    if (static_cast<int64_t>(blockIdx.x) >= n_mblk) return;
    const float* X = (dir ? Q : P) + b * nx * dim;
    const float* Y = (dir ? P : Q) + b * ny * dim;
    const float* pb = dir ? t.part_best[1] : t.part_best[0];
    const int32_t* pi = dir ? t.part_idx[1] : t.part_idx[0];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t src0 = static_cast<int64_t>(blockIdx.x) * 256 + warp * 32;
    const int64_t my_src = src0 + lane;
    const bool mine = my_src < nx;
    int32_t chunk = -1;
    if (mine) {
        const int64_t stride = t.B * nx;
        float best = __int_as_float(0x7f800000);
        for (int64_t s = 0; s < n_span; ++s) {
            const float v = pb[s * stride + b * nx + my_src];
            if (v < best) {
                best = v;
                chunk = pi[s * stride + b * nx + my_src];
            }
        }
    }
    float my_x[kTcMaxDim];
#pragma unroll
    for (int k = 0; k < kTcMaxDim; ++k) my_x[k] = (mine && k < dim) ? X[my_src * dim + k] : 0.f;
    float my_d2 = 0.f;
    int32_t my_arg = -1;
    for (int i = 0; i < 32; ++i) {
        const int32_t c = __shfl_sync(0xFFFFFFFFu, chunk, i);
        if (c < 0) continue;  // warp-uniform
        float xv[kTcMaxDim];
#pragma unroll
        for (int k = 0; k < kTcMaxDim; ++k) xv[k] = __shfl_sync(0xFFFFFFFFu, my_x[k], i);
        const int64_t tgt = static_cast<int64_t>(c) * 32 + lane;
        float d2 = __int_as_float(0x7f800000);
        if (tgt < ny) {
            const float* y = Y + tgt * dim;
            const float e0 = __fsub_rn(xv[0], y[0]);
            d2 = __fmul_rn(e0, e0);
#pragma unroll
            for (int k = 1; k < kTcMaxDim; ++k) {
                if (k < dim) {
                    const float e = __fsub_rn(xv[k], y[k]);
                    d2 = __fmaf_rn(e, e, d2);
                }
            }
        }
        float m = d2;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, tgt < ny && d2 == m);
        if (lane == i && hit != 0u) {
            my_d2 = m;
            my_arg = static_cast<int32_t>(static_cast<int64_t>(c) * 32 + (__ffs(hit) - 1));
        }
    }
    if (mine) {
        (dir ? a.dist[1] : a.dist[0])[b * nx + my_src] = my_d2;
        (dir ? a.idx[1] : a.idx[0])[b * nx + my_src] = my_arg;
    }
    double sum = static_cast<double>(my_d2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    __shared__ double wsum[8];
    if (lane == 0) wsum[warp] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < 8; ++w) tot += wsum[w];
        (dir ? a.loss_part[1] : a.loss_part[0])[b * n_mblk + blockIdx.x] = tot;
    }
}

}  // namespace maxsim
