// Top-k of score rows, and the glue of the two-stage INT8 -> f16 / bf16
// top-K scan ("Flash-MaxSim" paper, Sec. 4: a two-stage INT8 -> FP16 top-K
// scan is one of the forward variants; TileMaxSim's retrieval pipeline takes
// the top-k of the scores after scoring).
//
// topk_kernel: one block of 1024 threads per row.
//  1. Radix select of the k-th largest value on an order-preserving 32-bit key
//     (larger float -> larger key; -0 and +0 are one key; NaN is the lowest):
//     four passes of 8 bits from the top, each a shared-memory histogram of
//     the keys that match the digits chosen so far. It yields the threshold
//     key T and how many of the keys equal to T belong to the top k.
//  2. Compaction in index order: every key above T, then the first keys equal
//     to T by index (lower index first among equal values).
//  3. A bitonic sort of the k selected (key descending, index ascending) in
//     shared memory, and the write of indices (optionally mapped through an
//     id table) and the original values.
#pragma once

#include <cstdint>

namespace maxsim {

constexpr int kTopkThreads = 1024;
constexpr int kTopkMaxK = 4096;
constexpr int kTopkPer = 4;  // consecutive elements per thread in the compaction

__device__ __forceinline__ uint32_t topk_key(float v) {
    uint32_t b = __float_as_uint(v);
    if ((b & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below every number
    if ((b & 0x7fffffffu) == 0u) b = 0u;             // -0 and +0 are equal
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkArgs {
    const float* scores;  // [rows, row_stride], n used per row
    int64_t n, row_stride;
    int32_t k, pow2;      // pow2: the sort width, a power of two >= k
    const int32_t* id_map;  // optional: output id = id_map[r * map_stride + position]
    int64_t map_stride;
    int32_t* out_idx;     // [rows, out_stride]
    float* out_val;       // optional, [rows, out_stride]
    int64_t out_stride;
};

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
    extern __shared__ uint32_t tk_sel[];  // keys [pow2], then positions [pow2]
    uint32_t* sel_key = tk_sel;
    int32_t* sel_pos = reinterpret_cast<int32_t*>(tk_sel + a.pow2);
    __shared__ int32_t hist[256];
    __shared__ int32_t wsum[kTopkThreads / 32];
    __shared__ uint32_t s_digit;
    __shared__ int32_t s_rem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const float* row = a.scores + r * a.row_stride;
    const int64_t n = a.n;

    // 1. radix select
    uint32_t prefix = 0, mask = 0;
    int32_t remaining = a.k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t i = tid; i < n; i += kTopkThreads) {
            const uint32_t key = topk_key(row[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 8l .. 8l+7; counts from the top down
            int32_t c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[lane * 8 + j];
                tot += c[j];
            }
            int32_t incl = tot;  // sum over lanes >= lane
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                if (lane + o < 32) incl += y;
            }
            const int32_t above = incl - tot;
            if (above < remaining && remaining <= incl) {  // exactly one lane
                int32_t cum = above;
                for (int j = 7; j >= 0; --j) {
                    if (cum + c[j] >= remaining) {
                        s_digit = static_cast<uint32_t>(lane * 8 + j);
                        s_rem = remaining - cum;
                        break;
                    }
                    cum += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        remaining = s_rem;
        __syncthreads();
    }
    const uint32_t T = prefix;
    const int32_t n_gt = a.k - remaining;  // keys above T, all taken

    // 2. compaction in index order (counts packed: above T in the high half)
    int32_t run_gt = 0, run_eq = 0;
    for (int64_t base = 0; base < n; base += static_cast<int64_t>(kTopkThreads) * kTopkPer) {
        const int64_t i0 = base + static_cast<int64_t>(tid) * kTopkPer;
        uint32_t keys[kTopkPer];
        int32_t packed = 0;
#pragma unroll
        for (int e = 0; e < kTopkPer; ++e) {
            keys[e] = i0 + e < n ? topk_key(row[i0 + e]) : 0u;
            const bool ok = i0 + e < n;
            packed += (ok && keys[e] > T) ? (1 << 16) : 0;
            packed += (ok && keys[e] == T) ? 1 : 0;
        }
        int32_t x = packed;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int32_t excl = (warp > 0 ? wsum[warp - 1] : 0) + x - packed;
        int32_t g = run_gt + (excl >> 16), q = run_eq + (excl & 0xFFFF);
#pragma unroll
        for (int e = 0; e < kTopkPer; ++e) {
            if (i0 + e >= n) break;
            if (keys[e] > T) {
                sel_key[g] = keys[e];
                sel_pos[g] = static_cast<int32_t>(i0 + e);
                ++g;
            } else if (keys[e] == T) {
                if (q < remaining) {
                    sel_key[n_gt + q] = keys[e];
                    sel_pos[n_gt + q] = static_cast<int32_t>(i0 + e);
                }
                ++q;
            }
        }
        const int32_t total = wsum[kTopkThreads / 32 - 1];
        run_gt += total >> 16;
        run_eq += total & 0xFFFF;
        __syncthreads();
    }
    for (int i = a.k + tid; i < a.pow2; i += kTopkThreads) {  // padding sorts last
        sel_key[i] = 0u;
        sel_pos[i] = 0x7FFFFFFF;
    }
    __syncthreads();

    // 3. bitonic sort: key descending, position ascending
    for (int size = 2; size <= a.pow2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < a.pow2; i += kTopkThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint32_t ki = sel_key[i], kj = sel_key[j];
                    const int32_t pi = sel_pos[i], pj = sel_pos[j];
                    const bool j_first = kj > ki || (kj == ki && pj < pi);  // j belongs before i
                    const bool up = (i & size) == 0;                       // this run sorts in order
                    if (up == j_first) {
                        sel_key[i] = kj;
                        sel_key[j] = ki;
                        sel_pos[i] = pj;
                        sel_pos[j] = pi;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int j = tid; j < a.k; j += kTopkThreads) {
        const int32_t pos = sel_pos[j];
        a.out_idx[r * a.out_stride + j] = a.id_map ? a.id_map[r * a.map_stride + pos] : pos;
        if (a.out_val) a.out_val[r * a.out_stride + j] = row[pos];
    }
}

// The pair list of the rescoring stage: pairs[i * k1 + c] = (i, cand[i * k1 + c]).
__global__ void two_stage_pairs_kernel(const int32_t* __restrict__ cand, int64_t nq, int64_t k1,
                                       int32_t* __restrict__ pairs) {
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; p < nq * k1;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        pairs[2 * p] = static_cast<int32_t>(p / k1);
        pairs[2 * p + 1] = cand[p];
    }
}

// Row offsets of a dense [Nd, Ld] corpus seen as packed documents: cu[j] = j * Ld.
__global__ void uniform_offsets_kernel(int64_t nd, int64_t ld, int32_t* __restrict__ cu) {
    for (int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; j <= nd;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x)
        cu[j] = static_cast<int32_t>(j * ld);
}

}  // namespace maxsim
