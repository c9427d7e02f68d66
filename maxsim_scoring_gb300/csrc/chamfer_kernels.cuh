// Chamfer distance ("Flash-MaxSim" paper, Sec. 4.2.4) on the CUDA cores:
//   CD(P, Q) = (1/N) sum_p min_q ||p - q||^2 + (1/M) sum_q min_p ||q - p||^2
// for B independent pairs of float32 point sets with 1 <= dim <= 8.
//
// Forward: the MaxSim structure with a min in place of the max. The [N, M]
// distance table is never formed: sources stay in registers, targets stream
// through shared memory, and each source keeps a running minimum. Points of
// a few coordinates give the tensor cores nothing to contract, so this is
// fp32 ALU work, organised to spend about dim FMAs and one min per
// (source, target) pair:
//  * min_t ||x - y_t||^2 = ||x||^2 + min_t (||y_t||^2 - 2 <x, y_t>): the
//    search runs on the shifted value d'(x, y) = fma chain of x_k * (-2 y_k)
//    starting from ||y||^2, which shared memory holds precomputed per target;
//  * targets sit in shared memory in pairs, coordinate-interleaved, so two
//    16-byte broadcast loads feed 2 x kD FMAs per source, and a three-input
//    min folds both targets into the source's running minimum (the packed
//    fma.rn.f32x2 form was measured slower: it occupies the FMA pipe as long
//    as two scalar FMAs and stalls on dispatch);
//  * the argmin is not tracked per pair: every 32 targets (a sub-tile) each
//    source records the sub-tile in which its minimum last dropped; once the
//    search is over, a second kernel recomputes d' bit for bit over that one
//    sub-tile and takes the first target that attains the minimum (lowest
//    index among ties), then the exact distance sum_k (x_k - y_k)^2 of the
//    winner.
// Work items are (direction, set pair, block of sources, span of targets),
// handed out by an atomic counter to a persistent grid; partial results per
// span are merged in span order (strict <, so the earlier span wins ties).
//
// Backward through the saved nearest indices, with the inverse index of
// Sec. 4.2.2 (a stable sort of flattened destinations, then row pointers) and
// the destination-owned reduction of Sec. 4.2.3: one thread owns each point's
// gradient and walks its inverse row in ascending source order: no atomics,
// bitwise reproducible.
#pragma once

#include <cstdint>

namespace maxsim {

constexpr int kChThreads = 256;
constexpr int kChSub = 32;      // targets per sub-tile (argmin bookkeeping unit)
constexpr int kChTile = 2048;   // targets per shared-memory tile
constexpr int kChSpan = 4096;   // targets per work item
constexpr int kChMaxDim = 8;
constexpr int kChMergeThreads = 256;
static_assert(kChSpan % kChTile == 0 && kChTile % kChSub == 0, "tile sizes");

// kD: coordinates held per point (dim padded with zeros: a zero coordinate
// adds fma(0, 0, acc) = acc to every chain, so the padding changes no value).
template <int kD>
struct ChamferShape {
    static constexpr int kSrc = kD <= 3 ? 8 : 4;                  // sources per thread
    static constexpr int kUnroll = kD <= 3 ? 4 : 1;               // target pairs unrolled in the inner loop
    static constexpr int kPairFloats = ((kD + 1) * 2 + 3) / 4 * 4;  // one target pair in shared memory
    static constexpr int kSources = kSrc * kChThreads;            // sources per work item
    static constexpr size_t kSmem = static_cast<size_t>(kChTile / 2) * kPairFloats * sizeof(float);
};

struct ChamferFwdArgs {
    const float* X[2];  // sources of direction 0 (P) and 1 (Q)
    const float* Y[2];  // targets
    int64_t nx[2], ny[2];
    int64_t B;
    int32_t dim;
    int64_t n_sb[2];     // source blocks per set
    int64_t n_span[2];   // target spans per set
    int64_t items0, items;
    float* part_best[2];      // [n_span][B * nx]: minimum of d' over the span
    int32_t* part_sub[2];     // [n_span][B * nx]: global sub-tile index of that minimum, -1 if none
    unsigned long long* counter;
    // merge outputs
    float* dist[2];
    int32_t* idx[2];
    double* loss_part[2];     // [B][n_mblk]
    int64_t n_mblk[2];
    float* loss;
    int* status;
};

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ||y||^2 in the one fixed order both kernels use.
__device__ __forceinline__ float ch_norm2(const float* y, int dim) {
    float n = __fmul_rn(y[0], y[0]);
    for (int k = 1; k < dim; ++k) n = __fmaf_rn(y[k], y[k], n);
    return n;
}

template <int kD>
__global__ void __launch_bounds__(kChThreads, 2) chamfer_nn_kernel(ChamferFwdArgs a) {
    using S = ChamferShape<kD>;
    constexpr int kSrc = S::kSrc;
    constexpr int kV = S::kPairFloats / 4;  // 16-byte vectors per target pair
    extern __shared__ __align__(16) float ch_tile[];
    __shared__ unsigned long long s_item;
    const int tid = threadIdx.x;
    const int dim = a.dim;
    for (;;) {
        __syncthreads();  // the previous item is done with s_item and the tile
        if (tid == 0) s_item = atomicAdd(a.counter, 1ull);
        __syncthreads();
        const int64_t it = static_cast<int64_t>(s_item);
        if (it >= a.items) return;
        const int dir = it >= a.items0 ? 1 : 0;
        int64_t r = it - (dir ? a.items0 : 0);
        const int64_t n_span = dir ? a.n_span[1] : a.n_span[0], n_sb = dir ? a.n_sb[1] : a.n_sb[0];
        const int64_t span = r % n_span;
        r /= n_span;
        const int64_t sb = r % n_sb;
        const int64_t b = r / n_sb;
        // (ternaries, not a[dir]: a dynamic index into the parameter block
        // would copy it to local memory)
        const int64_t nx = dir ? a.nx[1] : a.nx[0], ny = dir ? a.ny[1] : a.ny[0];
        const float* Xb = (dir ? a.X[1] : a.X[0]) + b * nx * dim;
        const float* Yb = (dir ? a.Y[1] : a.Y[0]) + b * ny * dim;

        float xx[kSrc][kD];
        float m[kSrc], best[kSrc];
        int32_t sub_of[kSrc];
#pragma unroll
        for (int s = 0; s < kSrc; ++s) {
            const int64_t src = sb * S::kSources + s * kChThreads + tid;
#pragma unroll
            for (int k = 0; k < kD; ++k) {
                xx[s][k] = (src < nx && k < dim) ? Xb[src * dim + k] : 0.f;
            }
            m[s] = __int_as_float(0x7f800000);
            best[s] = m[s];
            sub_of[s] = -1;
        }

        const int64_t t_begin = span * kChSpan;
        const int64_t t_end = ny - t_begin < kChSpan ? ny : t_begin + kChSpan;
        for (int64_t t0 = t_begin; t0 < t_end; t0 += kChTile) {
            const int n = static_cast<int>(t_end - t0 < kChTile ? t_end - t0 : kChTile);
            const int n_sub = (n + kChSub - 1) / kChSub;
            __syncthreads();
            // fill: target t of the tile -> pair t/2, lane t%2; padding targets
            // get ||y||^2 = +inf and never win
            for (int t = tid; t < n_sub * kChSub; t += kChThreads) {
                float y[kD];
#pragma unroll
                for (int k = 0; k < kD; ++k) y[k] = (t < n && k < dim) ? Yb[(t0 + t) * dim + k] : 0.f;
                float* dst = ch_tile + (t >> 1) * S::kPairFloats + (t & 1);
#pragma unroll
                for (int k = 0; k < kD; ++k) dst[2 * k] = __fmul_rn(-2.f, y[k]);
                // ||y||^2 over all kD slots: the zero padding adds fma(0, 0, n) = n,
                // the same value as over the dim real coordinates
                float nrm = __fmul_rn(y[0], y[0]);
#pragma unroll
                for (int k = 1; k < kD; ++k) nrm = __fmaf_rn(y[k], y[k], nrm);
                dst[2 * kD] = t < n ? nrm : __int_as_float(0x7f800000);
#pragma unroll
                for (int k = 2 * kD + 2; k < S::kPairFloats; k += 2) dst[k] = 0.f;
            }
            __syncthreads();
            const int64_t sub0 = t0 / kChSub;
            for (int st = 0; st < n_sub; ++st) {
                const float4* tp = reinterpret_cast<const float4*>(ch_tile) + static_cast<int64_t>(st) * (kChSub / 2) * kV;
#pragma unroll S::kUnroll
                for (int j = 0; j < kChSub / 2; ++j) {
                    float c[4 * kV];  // (-2 y_k of the two targets) for each k, then the two norms
#pragma unroll
                    for (int v = 0; v < kV; ++v) {
                        const float4 q = tp[j * kV + v];
                        c[4 * v] = q.x;
                        c[4 * v + 1] = q.y;
                        c[4 * v + 2] = q.z;
                        c[4 * v + 3] = q.w;
                    }
#pragma unroll
                    for (int s = 0; s < kSrc; ++s) {
                        float d0 = c[2 * kD], d1 = c[2 * kD + 1];
#pragma unroll
                        for (int k = 0; k < kD; ++k) {
                            d0 = __fmaf_rn(xx[s][k], c[2 * k], d0);
                            d1 = __fmaf_rn(xx[s][k], c[2 * k + 1], d1);
                        }
                        m[s] = min3f(m[s], d0, d1);
                    }
                }
#pragma unroll
                for (int s = 0; s < kSrc; ++s) {
                    if (m[s] < best[s]) sub_of[s] = static_cast<int32_t>(sub0 + st);
                    best[s] = m[s];
                }
            }
        }
        const int64_t base = span * a.B * nx + b * nx;
        float* pb = (dir ? a.part_best[1] : a.part_best[0]) + base;
        int32_t* ps = (dir ? a.part_sub[1] : a.part_sub[0]) + base;
#pragma unroll
        for (int s = 0; s < kSrc; ++s) {
            const int64_t src = sb * S::kSources + s * kChThreads + tid;
            if (src < nx) {
                pb[src] = best[s];
                ps[src] = sub_of[s];
            }
        }
    }
}

// Merge of the spans, exact argmin inside the winning sub-tile, distance of
// the winner, and the block's share of the loss. Grid (blocks, B, 2); a
// block covers kChMergeThreads sources, a warp 32 of them:
//  * lane l merges the spans of source l in span order (strict <: the
//    earliest span keeps a tie);
//  * then, four sources at a time, lane t recomputes d' for target t of each
//    winning sub-tile (the operations of the search, in its order), and the
//    first lane whose value equals the minimum holds the argmin; that lane
//    computes the distance sum_k (x_k - y_k)^2 directly.
constexpr int kChMergeGroup = 4;
__global__ void __launch_bounds__(kChMergeThreads) chamfer_merge_kernel(ChamferFwdArgs a) {
    const int dir = blockIdx.z;
    const int64_t b = blockIdx.y;
    const int64_t nx = dir ? a.nx[1] : a.nx[0], ny = dir ? a.ny[1] : a.ny[0];
    const int64_t n_mblk = dir ? a.n_mblk[1] : a.n_mblk[0], n_span = dir ? a.n_span[1] : a.n_span[0];
    const float* part_best = dir ? a.part_best[1] : a.part_best[0];
    const int32_t* part_sub = dir ? a.part_sub[1] : a.part_sub[0];
    const float* X = (dir ? a.X[1] : a.X[0]) + b * nx * a.dim;
    const float* Yb = (dir ? a.Y[1] : a.Y[0]) + b * ny * a.dim;
    const int dim = a.dim;
    if (static_cast<int64_t>(blockIdx.x) >= n_mblk) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t src0 = static_cast<int64_t>(blockIdx.x) * kChMergeThreads + warp * 32;
    const int64_t my_src = src0 + lane;
    const bool mine = my_src < nx;
    // this lane's source: merge its spans
    float best = __int_as_float(0x7f800000);
    int32_t sub = -1;
    if (mine) {
        const int64_t stride = a.B * nx;
        for (int64_t sp = 0; sp < n_span; ++sp) {
            const float v = part_best[sp * stride + b * nx + my_src];
            if (v < best) {
                best = v;
                sub = part_sub[sp * stride + b * nx + my_src];
            }
        }
    }
    float my_x[kChMaxDim];
#pragma unroll
    for (int k = 0; k < kChMaxDim; ++k) my_x[k] = (mine && k < dim) ? X[my_src * dim + k] : 0.f;
    float my_d2 = 0.f;
    int32_t my_arg = -1;
    for (int i0 = 0; i0 < 32; i0 += kChMergeGroup) {
        float yv[kChMergeGroup][kChMaxDim];
        int32_t sb[kChMergeGroup];
        float bv[kChMergeGroup];
#pragma unroll
        for (int g = 0; g < kChMergeGroup; ++g) {
            sb[g] = __shfl_sync(0xFFFFFFFFu, sub, i0 + g);
            bv[g] = __shfl_sync(0xFFFFFFFFu, best, i0 + g);
            const int64_t t = static_cast<int64_t>(sb[g]) * kChSub + lane;
            const bool ok = sb[g] >= 0 && t < ny;
#pragma unroll
            for (int k = 0; k < kChMaxDim; ++k) yv[g][k] = (ok && k < dim) ? Yb[t * dim + k] : 0.f;
        }
#pragma unroll
        for (int g = 0; g < kChMergeGroup; ++g) {
            if (sb[g] < 0) continue;  // warp-uniform
            float xv[kChMaxDim];
#pragma unroll
            for (int k = 0; k < kChMaxDim; ++k) xv[k] = __shfl_sync(0xFFFFFFFFu, my_x[k], i0 + g);
            const int64_t t = static_cast<int64_t>(sb[g]) * kChSub + lane;
            float acc = __fmul_rn(yv[g][0], yv[g][0]);
#pragma unroll
            for (int k = 1; k < kChMaxDim; ++k)
                if (k < dim) acc = __fmaf_rn(yv[g][k], yv[g][k], acc);
#pragma unroll
            for (int k = 0; k < kChMaxDim; ++k)
                if (k < dim) acc = __fmaf_rn(xv[k], __fmul_rn(-2.f, yv[g][k]), acc);
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, t < ny && acc == bv[g]);
            if (hit == 0u) {
                if (lane == 0 && a.status) atomicCAS(a.status, 0, 6);  // a recomputation that disagrees
                continue;
            }
            const int w = __ffs(hit) - 1;
            float d2 = 0.f;
            if (lane == w) {
                const float e0 = __fsub_rn(xv[0], yv[g][0]);
                d2 = __fmul_rn(e0, e0);
#pragma unroll
                for (int k = 1; k < kChMaxDim; ++k) {
                    if (k < dim) {
                        const float e = __fsub_rn(xv[k], yv[g][k]);
                        d2 = __fmaf_rn(e, e, d2);
                    }
                }
            }
            d2 = __shfl_sync(0xFFFFFFFFu, d2, w);
            if (lane == i0 + g) {
                my_d2 = d2;
                my_arg = static_cast<int32_t>(static_cast<int64_t>(sb[g]) * kChSub + w);
            }
        }
    }
    if (mine) {
        (dir ? a.dist[1] : a.dist[0])[b * nx + my_src] = my_d2;
        (dir ? a.idx[1] : a.idx[0])[b * nx + my_src] = my_arg;
    }
    // the block's share of sum(dist): fixed-order trees in double
    double sum = static_cast<double>(my_d2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    __shared__ double wsum[kChMergeThreads / 32];
    if (lane == 0) wsum[warp] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kChMergeThreads / 32; ++w) t += wsum[w];
        (dir ? a.loss_part[1] : a.loss_part[0])[b * n_mblk + blockIdx.x] = t;
    }
}

// loss[b] = sum(dist_p[b]) / N + sum(dist_q[b]) / M (0 if N or M is 0); one
// block per pair of sets, the partial sums added in a fixed order.
constexpr int kChLossThreads = 256;
__global__ void __launch_bounds__(kChLossThreads) chamfer_loss_kernel(ChamferFwdArgs a) {
    const int64_t b = blockIdx.x;
    __shared__ double red[2][kChLossThreads];
    double s0 = 0.0, s1 = 0.0;
    for (int64_t k = threadIdx.x; k < a.n_mblk[0]; k += kChLossThreads) s0 += a.loss_part[0][b * a.n_mblk[0] + k];
    for (int64_t k = threadIdx.x; k < a.n_mblk[1]; k += kChLossThreads) s1 += a.loss_part[1][b * a.n_mblk[1] + k];
    red[0][threadIdx.x] = s0;
    red[1][threadIdx.x] = s1;
    __syncthreads();
    for (int w = kChLossThreads / 2; w > 0; w >>= 1) {
        if (static_cast<int>(threadIdx.x) < w) {
            red[0][threadIdx.x] += red[0][threadIdx.x + w];
            red[1][threadIdx.x] += red[1][threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int64_t N = a.nx[0], M = a.nx[1];
        a.loss[b] = (N > 0 && M > 0) ? static_cast<float>(red[0][0] / static_cast<double>(N) +
                                                           red[1][0] / static_cast<double>(M))
                                     : 0.f;
    }
}

// ---------------------------------------------------------------- backward

// Flattened destinations of every source. Rows [0, B*M) are the Q points
// (destinations of idx_p), rows [B*M, B*M + B*N) the P points (of idx_q); the
// key R = B*(N+M) marks a source with no destination. The value is the
// source's global row (b*N + p, or b*M + q).
__global__ void ch_keys_kernel(const int32_t* __restrict__ idx_p, const int32_t* __restrict__ idx_q, int64_t B,
                               int64_t N, int64_t M, uint32_t* __restrict__ keys, int32_t* __restrict__ vals,
                               int* status) {
    const int64_t np = B * N, total = B * (N + M);
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < total;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool from_p = s < np;
        const int64_t row = from_p ? s : s - np;
        const int64_t nsrc = from_p ? N : M, ndst = from_p ? M : N;
        const int64_t b = row / nsrc;
        const int32_t d = from_p ? idx_p[row] : idx_q[row];
        const bool ok = d >= 0 && d < ndst;
        if (!ok && d != -1 && status) atomicCAS(status, 0, 6);
        const int64_t base = from_p ? 0 : B * M;
        keys[s] = static_cast<uint32_t>(ok ? base + b * ndst + d : total);
        vals[s] = static_cast<int32_t>(row);
    }
}

constexpr int kRadixBits = 9;
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kRadixThreads = 256;
constexpr int kRadixPerThread = 16;
constexpr int kRadixBlock = kRadixThreads * kRadixPerThread;  // keys per block
static_assert(kRadixBins % kRadixThreads == 0, "bins per thread");

// Per-block counts of one digit, stored bin-major: hist[bin * blocks + block].
__global__ void __launch_bounds__(kRadixThreads) radix_hist_kernel(const uint32_t* __restrict__ keys, int64_t n,
                                                                   int shift, int32_t* __restrict__ hist,
                                                                   int64_t nblocks) {
    __shared__ int32_t h[kRadixBins];
    for (int i = threadIdx.x; i < kRadixBins; i += kRadixThreads) h[i] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixBlock;
#pragma unroll 4
    for (int e = 0; e < kRadixPerThread; ++e) {
        const int64_t i = base + e * kRadixThreads + threadIdx.x;
        if (i < n) atomicAdd(&h[(keys[i] >> shift) & (kRadixBins - 1)], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kRadixBins; i += kRadixThreads)
        hist[static_cast<int64_t>(i) * nblocks + blockIdx.x] = h[i];
}

// Exclusive prefix sum in place over n int32 by one block of 1024 threads,
// 8192 values per pass: warp w scans its 256 consecutive values as 8 rows
// of 32 (coalesced loads, shuffle scans, a running carry), then the 32 warp
// totals are scanned and added.
constexpr int kScanThreads = 1024;
constexpr int kScanRows = 8;
__global__ void __launch_bounds__(kScanThreads) scan_exclusive_kernel(int32_t* __restrict__ a, int64_t n) {
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += static_cast<int64_t>(kScanThreads) * kScanRows) {
        const int64_t w0 = base + static_cast<int64_t>(warp) * 32 * kScanRows;
        int32_t v[kScanRows], incl[kScanRows];
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) {
            const int64_t i = w0 + r * 32 + lane;
            v[r] = i < n ? a[i] : 0;
        }
        int32_t run = 0;
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) {
            int32_t x = v[r];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            incl[r] = run + x;
            run += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        if (lane == 0) wsum[warp] = run;
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
        const int32_t prefix = carry + (warp > 0 ? wsum[warp - 1] : 0);
#pragma unroll
        for (int r = 0; r < kScanRows; ++r) {
            const int64_t i = w0 + r * 32 + lane;
            if (i < n) a[i] = prefix + incl[r] - v[r];
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += wsum[31];
        __syncthreads();
    }
}

// Stable scatter of one digit. A block takes its keys in index order, 256 at
// a time; inside a batch the warps go in turn and lanes are ranked by
// __match_any_sync, so equal digits keep their input order.
__global__ void __launch_bounds__(kRadixThreads) radix_scatter_kernel(
    const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in, int64_t n, int shift,
    const int32_t* __restrict__ offs, int64_t nblocks, uint32_t* __restrict__ keys_out,
    int32_t* __restrict__ vals_out) {
    __shared__ int32_t run[kRadixBins];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kRadixBins; i += kRadixThreads)
        run[i] = offs[static_cast<int64_t>(i) * nblocks + blockIdx.x];
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixBlock;
    for (int e = 0; e < kRadixPerThread; ++e) {
        const int64_t i = base + e * kRadixThreads + threadIdx.x;
        const bool valid = i < n;
        const uint32_t k = valid ? keys_in[i] : 0u;
        const int32_t v = valid ? vals_in[i] : 0;
        const int d = valid ? static_cast<int>((k >> shift) & (kRadixBins - 1)) : -1;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const bool last = (peers >> lane) == 1u;  // highest lane holding this digit
        for (int w = 0; w < kRadixThreads / 32; ++w) {
            if (warp == w && valid) {
                const int32_t slot = run[d] + rank;
                keys_out[slot] = k;
                vals_out[slot] = v;
            }
            __syncwarp();
            if (warp == w && valid && last) run[d] += __popc(peers);
            __syncthreads();
        }
    }
}

// row_ptr[r] = first position of the sorted keys with key >= r, r in [0, R].
__global__ void ch_row_ptr_kernel(const uint32_t* __restrict__ keys, int64_t n, int64_t R,
                                  int32_t* __restrict__ row_ptr) {
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r <= R;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t lo = 0, hi = n;
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (static_cast<int64_t>(keys[mid]) < r) lo = mid + 1;
            else hi = mid;
        }
        row_ptr[r] = static_cast<int32_t>(lo);
    }
}

struct ChamferBwdArgs {
    const float* P;
    const float* Q;
    int64_t B, N, M;
    int32_t dim;
    const int32_t* idx_p;
    const int32_t* idx_q;
    const float* g;
    float* dP;
    float* dQ;
    const int32_t* row_ptr;  // [R + 1]
    const int32_t* col;      // source rows in destination order
};

// Gradient of sum_b g[b] CD(P_b, Q_b), one thread per point. For a point x of
// X with nearest index near[x] in Y, and inverse row {y : near_Y(y) = x}:
//   dX[x] = g (2/|X|) (x - Y[near[x]]) - g (2/|Y|) sum over the row of (y - x)
// Threads [0, B*N) own the P points, the rest the Q points.
template <int kD>
__global__ void chamfer_grad_kernel(ChamferBwdArgs a) {
    const int64_t np = a.B * a.N, total = a.B * (a.N + a.M);
    const int dim = a.dim;
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < total;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool is_p = s < np;
        const int64_t row = is_p ? s : s - np;
        const int64_t nx = is_p ? a.N : a.M, ny = is_p ? a.M : a.N;
        const float* X = is_p ? a.P : a.Q;
        const float* Y = is_p ? a.Q : a.P;
        const int32_t* near = is_p ? a.idx_p : a.idx_q;
        float* dX = is_p ? a.dP : a.dQ;
        const int64_t b = row / nx;
        const float gb = a.g[b];
        const float wx = __fdiv_rn(2.f * gb, static_cast<float>(nx));
        const float wy = ny > 0 ? __fdiv_rn(2.f * gb, static_cast<float>(ny)) : 0.f;
        float x[kD], inv[kD];
#pragma unroll
        for (int k = 0; k < kD; ++k) {
            x[k] = k < dim ? X[row * dim + k] : 0.f;
            inv[k] = 0.f;
        }
        // inverse row: the P point rows follow the B*M Q point rows
        const int64_t r = is_p ? a.B * a.M + row : row;
        const int32_t e0 = a.row_ptr[r], e1 = a.row_ptr[r + 1];
        for (int32_t e = e0; e < e1; ++e) {
            const float* y = Y + static_cast<int64_t>(a.col[e]) * dim;
#pragma unroll
            for (int k = 0; k < kD; ++k)
                if (k < dim) inv[k] = __fadd_rn(inv[k], __fsub_rn(y[k], x[k]));
        }
        const int32_t n = near[row];
        const bool own = n >= 0 && n < ny;
        const float* yn = Y + (b * ny + (own ? n : 0)) * dim;
#pragma unroll
        for (int k = 0; k < kD; ++k) {
            if (k < dim) {
                const float o = own ? __fmul_rn(wx, __fsub_rn(x[k], yn[k])) : 0.f;
                dX[row * dim + k] = __fsub_rn(o, __fmul_rn(wy, inv[k]));
            }
        }
    }
}

}  // namespace maxsim
