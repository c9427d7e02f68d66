// Backward of MaxSim through the saved argmax ("Flash-MaxSim" Sec. 4.2):
//  * inverse-argmax CSR, built per document: sources p = (i*Nd + j)*Lq + s of
//    document j only point at rows of document j, so each document's slice of
//    the CSR is a counting sort of its own Nq*Lq sources (bincount -> prefix
//    sum -> stable placement in ascending p, Sec. 4.2.2);
//  * dD, destination-owned: one warp per document token walks its CSR sources
//    and writes its row once, no atomics (Sec. 4.2.3, Eq. (3));
//  * dQ, row-owned: one warp per query token gathers D at the winners of every
//    document in ascending j (Eq. (2)).
// Everything is deterministic: integer counts, fixed summation orders.
// Packed layouts (the varlen path of Sec. 4.3.2) change only where rows live:
// document j owns D rows cu_d[j] .. cu_d[j+1]-1 (its CSR rows are the same
// row numbers), query i owns Q rows cu_q[i] .. cu_q[i+1]-1; the argmax keeps
// its [Nq*Nd, max_lq] layout with -1 past a query's end.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace maxsim {

struct BwdArgs {
    const uint16_t* Q;     // [Nq, Lq, dim] f16 / bf16 bits
    const uint16_t* D;     // [Nd, Ld, dim]
    int32_t is_bf16;
    int32_t nq, lq, nd, ld, dim;
    const uint8_t* q_mask; // [Nq, Lq] or NULL
    const int32_t* argmax; // [Nq*Nd, Lq]
    const float* g;        // [Nq, Nd]
    float* dQ;             // [Nq, Lq, dim] or NULL
    float* dD;             // [Nd, Ld, dim] or NULL
    int32_t* row_ptr;      // [Nd*Ld + 1]
    int32_t* col;          // [Nq*Nd*Lq]
    int32_t* doc_cnt;      // [Nd]
    int32_t* doc_base;     // [Nd + 1]
    int* status;
    const int32_t* cu_q;   // [Nq + 1] or NULL: dense Q, rows i*lq + s
    const int32_t* cu_d;   // [Nd + 1] or NULL: dense D, rows j*ld + t (packed: ld is the longest document)
    int64_t d_rows;        // rows of D: Nd*ld dense, total_d packed
};

// Length of document j (-1: an inconsistent packed offset, reported, no rows used).
__device__ __forceinline__ int32_t doc_len(const BwdArgs& b, int32_t j) {
    if (!b.cu_d) return b.ld;
    const int32_t n = b.cu_d[j + 1] - b.cu_d[j];
    return (n < 0 || n > b.ld) ? -1 : n;
}
__device__ __forceinline__ int64_t doc_row0(const BwdArgs& b, int32_t j) {
    return b.cu_d ? static_cast<int64_t>(b.cu_d[j]) : static_cast<int64_t>(j) * b.ld;
}
__device__ __forceinline__ int32_t query_len(const BwdArgs& b, int32_t i) {
    return b.cu_q ? b.cu_q[i + 1] - b.cu_q[i] : b.lq;
}
__device__ __forceinline__ int64_t query_row(const BwdArgs& b, int32_t i, int32_t s) {
    return b.cu_q ? static_cast<int64_t>(b.cu_q[i]) + s : static_cast<int64_t>(i) * b.lq + s;
}

__device__ __forceinline__ float bits_to_f32(uint16_t h, int32_t is_bf16) {
    return is_bf16 ? __uint_as_float(static_cast<uint32_t>(h) << 16) : __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ bool argmax_ok(int32_t a, int32_t ld) { return a >= -1 && a < ld; }

// Sources of document j, in ascending p: (i, s) for i < Nq, s < Lq.
__device__ __forceinline__ int64_t src_index(const BwdArgs& b, int32_t j, int32_t n) {
    int32_t i = n / b.lq, s = n - (n / b.lq) * b.lq;
    return (static_cast<int64_t>(i) * b.nd + j) * b.lq + s;
}

// A source past its query's end (packed Q) has no Q row: it may only hold -1.
__device__ __forceinline__ bool src_in_query(const BwdArgs& b, int32_t n) {
    if (!b.cu_q) return true;
    const int32_t i = n / b.lq, s = n - (n / b.lq) * b.lq;
    return s < query_len(b, i);
}

// Per-document count of sources with a valid winner.
__global__ void __launch_bounds__(256) csr_count_kernel(const BwdArgs b) {
    const int32_t j = blockIdx.x;
    const int32_t nsrc = b.nq * b.lq;
    const int32_t ldj = doc_len(b, j);
    int32_t cnt = 0;
    bool bad = ldj < 0;
#pragma unroll 8
    for (int32_t n = threadIdx.x; n < nsrc && ldj >= 0; n += blockDim.x) {
        int32_t a = b.argmax[src_index(b, j, n)];
        if (a >= 0 && !src_in_query(b, n)) {
            bad = true;
            continue;
        }
        if (a >= 0 && a < ldj) ++cnt;
        else if (!argmax_ok(a, ldj)) bad = true;
    }
    if (bad && b.status) atomicCAS(b.status, 0, 6);
    __shared__ int32_t red[8];
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t tot = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
        b.doc_cnt[j] = tot;
    }
}

// Exclusive prefix sum of the per-document counts (one block, fixed order).
__global__ void __launch_bounds__(1024) csr_doc_scan_kernel(const BwdArgs b) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t base = 0; base < b.nd; base += blockDim.x) {
        int32_t j = base + threadIdx.x;
        int32_t v = j < b.nd ? b.doc_cnt[j] : 0;
        int32_t x = v;
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t ws = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xFFFFFFFFu, ws, o);
                if (lane >= o) ws += y;
            }
            warp_sums[lane] = ws;  // inclusive
        }
        __syncthreads();
        int32_t excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
        if (j < b.nd) b.doc_base[j] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        b.doc_base[b.nd] = carry;
        b.row_ptr[b.d_rows] = carry;
    }
}

// Counting sort of one document's sources into its CSR rows. Each of the
// block's `nw` warps owns a contiguous run of the sources; per-warp histograms
// give every warp its starting offset inside each row, and inside a warp the
// lanes holding the same destination are ranked by lane order, so sources land
// in ascending p (a stable sort, as Sec. 4.2.2 requires).
__global__ void __launch_bounds__(256) csr_build_kernel(const BwdArgs b, int32_t nw) {
    extern __shared__ int32_t hist[];  // [nw][ld]
    const int32_t j = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t nsrc = b.nq * b.lq;
    const int32_t per = (nsrc + nw - 1) / nw;
    const int32_t ldj = max(doc_len(b, j), 0);  // an inconsistent document gets no rows
    const int64_t row0 = doc_row0(b, j);
    for (int32_t x = threadIdx.x; x < nw * b.ld; x += blockDim.x) hist[x] = 0;
    __syncthreads();
    if (warp < nw) {
        const int32_t n0 = warp * per, n1 = min(n0 + per, nsrc);
#pragma unroll 4
        for (int32_t n = n0 + lane; n < n1; n += 32) {
            int32_t a = b.argmax[src_index(b, j, n)];
            if (a >= 0 && a < ldj && src_in_query(b, n)) atomicAdd(&hist[warp * b.ld + a], 1);
        }
    }
    __syncthreads();
    // exclusive scan over destinations t of the per-row totals; each thread
    // owns a contiguous range of t
    __shared__ int32_t part[256];
    const int32_t tper = (ldj + blockDim.x - 1) / blockDim.x;
    const int32_t t0 = min(threadIdx.x * tper, ldj), t1 = min(t0 + tper, ldj);
    int32_t local = 0;
    for (int32_t t = t0; t < t1; ++t)
        for (int32_t w = 0; w < nw; ++w) local += hist[w * b.ld + t];
    // exclusive scan of the per-thread totals across the block (warp scans,
    // then a scan of the warp totals)
    {
        int32_t x = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        __shared__ int32_t wsum[8];
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = lane < static_cast<int>(blockDim.x >> 5) ? wsum[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < 8) wsum[lane] = w;  // inclusive
        }
        __syncthreads();
        part[threadIdx.x] = (warp > 0 ? wsum[warp - 1] : 0) + x - local;
        __syncthreads();
    }
    int32_t run = b.doc_base[j] + part[threadIdx.x];
    for (int32_t t = t0; t < t1; ++t) {
        b.row_ptr[row0 + t] = run;
        for (int32_t w = 0; w < nw; ++w) {
            int32_t c = hist[w * b.ld + t];
            hist[w * b.ld + t] = run;  // becomes warp w's next free slot in row t
            run += c;
        }
    }
    __syncthreads();
    if (warp < nw) {
        const int32_t n0 = warp * per, n1 = min(n0 + per, nsrc);
        for (int32_t nb = n0; nb < n1; nb += 32) {
            const int32_t n = nb + lane;
            int32_t a = -1;
            int64_t p = 0;
            if (n < n1) {
                p = src_index(b, j, n);
                a = b.argmax[p];
                if (!(a >= 0 && a < ldj && src_in_query(b, n))) a = -1;
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, a);
            if (a >= 0) {
                const uint32_t lower = peers & ((1u << lane) - 1u);
                const int32_t rank = __popc(lower);
                const int32_t slot = hist[warp * b.ld + a] + rank;
                b.col[slot] = static_cast<int32_t>(p);
                __syncwarp(peers);
                if ((peers >> lane) == 1u) hist[warp * b.ld + a] += __popc(peers);  // highest peer lane
            }
            __syncwarp();
        }
    }
}

// One embedding row into this lane's kVec consecutive elements (lane * kVec
// + v) as fp32; whole-vector loads when the row is exactly 32 * kVec wide.
template <int kVec>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ row, int lane, int32_t dim, int32_t is_bf16,
                                         float (&x)[kVec]) {
    const int k0 = lane * kVec;
    if constexpr (kVec == 2 || kVec == 4 || kVec == 8) {
        if (dim == 32 * kVec) {
            uint32_t w[kVec / 2];
            if constexpr (kVec == 2) {
                w[0] = __ldg(reinterpret_cast<const uint32_t*>(row + k0));
            } else if constexpr (kVec == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + k0));
                w[0] = u.x;
                w[1] = u.y;
            } else {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + k0));
                w[0] = u.x;
                w[1] = u.y;
                w[2] = u.z;
                w[3] = u.w;
            }
#pragma unroll
            for (int h = 0; h < kVec / 2; ++h) {
                x[2 * h] = bits_to_f32(static_cast<uint16_t>(w[h] & 0xFFFFu), is_bf16);
                x[2 * h + 1] = bits_to_f32(static_cast<uint16_t>(w[h] >> 16), is_bf16);
            }
            return;
        }
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
        const int k = k0 + v;
        x[v] = k < dim ? bits_to_f32(row[k], is_bf16) : 0.f;
    }
}

template <int kVec>
__device__ __forceinline__ void store_row(float* __restrict__ out, int lane, int32_t dim, const float (&acc)[kVec]) {
    const int k0 = lane * kVec;
    if constexpr (kVec == 4) {
        if (dim == 128) {
            *reinterpret_cast<float4*>(out + k0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            return;
        }
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
        const int k = k0 + v;
        if (k < dim) out[k] = acc[v];
    }
}

// Rows gathered per batch: their loads are issued together so that their
// latencies overlap; the accumulation order is unchanged.
constexpr int kGather = 4;

// This lane's kVec elements of one row kept as raw 16-bit values (two per
// word) until they are used: a batch of gathers then holds half the
// registers of decoded floats, so twice as many rows can be in flight.
template <int kVec>
struct RawRow {
    uint32_t w[(kVec + 1) / 2];
};

template <int kVec>
__device__ __forceinline__ void load_raw(const uint16_t* __restrict__ row, int lane, int32_t dim, RawRow<kVec>& r) {
    const int k0 = lane * kVec;
    if constexpr (kVec == 2 || kVec == 4 || kVec == 8) {
        if (dim == 32 * kVec) {
            if constexpr (kVec == 2) {
                r.w[0] = __ldg(reinterpret_cast<const uint32_t*>(row + k0));
            } else if constexpr (kVec == 4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + k0));
                r.w[0] = u.x;
                r.w[1] = u.y;
            } else {
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + k0));
                r.w[0] = u.x;
                r.w[1] = u.y;
                r.w[2] = u.z;
                r.w[3] = u.w;
            }
            return;
        }
    }
#pragma unroll
    for (int h = 0; h < (kVec + 1) / 2; ++h) {
        const int k = k0 + 2 * h;
        const uint32_t lo = k < dim ? row[k] : 0u;
        const uint32_t hi = (2 * h + 1 < kVec && k + 1 < dim) ? row[k + 1] : 0u;
        r.w[h] = lo | (hi << 16);
    }
}

// (a0, a1) = w * (x0, x1) + (a0, a1) with one packed instruction; each lane
// is rounded as a plain fp32 fma.
__device__ __forceinline__ void fma2_rn(float& a0, float& a1, float w, float x0, float x1) {
    asm("{\n\t.reg .b64 d, m, x;\n\t"
        "mov.b64 d, {%0, %1};\n\t"
        "mov.b64 m, {%2, %2};\n\t"
        "mov.b64 x, {%3, %4};\n\t"
        "fma.rn.f32x2 d, m, x, d;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(w), "f"(x0), "f"(x1));
}

// Two 16-bit values of one word (element 2h in the low half) as fp32.
template <bool kBf16>
__device__ __forceinline__ void decode2(uint32_t wd, float& lo, float& hi) {
    if constexpr (kBf16) {
        lo = __uint_as_float(wd << 16);
        hi = __uint_as_float(wd & 0xFFFF0000u);
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wd));
        lo = f.x;
        hi = f.y;
    }
}

// acc[v] += wgt * element v, element by element (the same fp32 fmas as with
// decoded rows), two elements per packed instruction.
template <int kVec, bool kBf16>
__device__ __forceinline__ void fma_raw(float wgt, const RawRow<kVec>& r, float (&acc)[kVec]) {
#pragma unroll
    for (int h = 0; h < kVec / 2; ++h) {
        float lo, hi;
        decode2<kBf16>(r.w[h], lo, hi);
        fma2_rn(acc[2 * h], acc[2 * h + 1], wgt, lo, hi);
    }
    if constexpr (kVec & 1) {
        float lo, hi;
        decode2<kBf16>(r.w[kVec / 2], lo, hi);
        acc[kVec - 1] = fmaf(wgt, lo, acc[kVec - 1]);
    }
}

// dD: one warp per destination row (j, t); lanes split the embedding. The
// row's sources are taken 32 at a time: each lane decodes one (index, weight),
// then the warp walks them in CSR order.
template <int kVec>  // floats per lane (dim / 32, rounded up)
__global__ void __launch_bounds__(256) dd_kernel(const BwdArgs b) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= b.d_rows) return;
    float acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
    int32_t e0 = b.row_ptr[r], e1 = b.row_ptr[r + 1];
    // inconsistent packed offsets (reported by the checks) leave rows unset:
    // never read outside the CSR
    const int64_t n_col = static_cast<int64_t>(b.nq) * b.nd * b.lq;
    if (e0 < 0 || e1 < e0 || e1 > n_col) e1 = e0 = 0;
    for (int32_t eb = e0; eb < e1; eb += 32) {
        const int32_t cnt = min(32, e1 - eb);
        int64_t off = 0;  // element offset of this lane's source row in Q
        float wl = 0.f;
        if (lane < cnt) {
            const int32_t p = b.col[eb + lane];  // (i * Nd + j) * lq + s
            const int32_t s = p % b.lq;
            const int32_t i = (p / b.lq) / b.nd, j = (p / b.lq) % b.nd;
            const int64_t qr = query_row(b, i, s);
            wl = b.g[static_cast<int64_t>(i) * b.nd + j];
            if (b.q_mask && !b.q_mask[qr]) wl = 0.f;
            off = qr * b.dim;
        }
        for (int32_t k = 0; k < cnt; k += kGather) {
            float x[kGather][kVec];
            float w[kGather];
#pragma unroll
            for (int u = 0; u < kGather; ++u) {
                const int32_t src = min(k + u, cnt - 1);
                w[u] = __shfl_sync(0xFFFFFFFFu, wl, src);
                const int64_t o = __shfl_sync(0xFFFFFFFFu, off, src);
                load_row<kVec>(b.Q + o, lane, b.dim, b.is_bf16, x[u]);
            }
#pragma unroll
            for (int u = 0; u < kGather; ++u) {
                if (k + u < cnt) {
#pragma unroll
                    for (int v = 0; v < kVec; ++v) acc[v] = fmaf(w[u], x[u][v], acc[v]);
                }
            }
        }
    }
    store_row<kVec>(b.dD + r * b.dim, lane, b.dim, acc);
}

// dD without a materialised CSR (dense D, caller did not ask for the CSR):
// one CTA per (document j, slice of kDdRows of its tokens). The CTA reads
// the Nq*Lq sources of document j, keeps those whose winner lies in its
// slice, and builds the slice's inverse-argmax CSR in shared memory with the
// same stable counting sort as csr_build_kernel (per-warp histograms over
// contiguous runs of sources, ranks within a warp by lane order), so each
// destination row lists its sources in ascending p (Sec. 4.2.2). Each warp
// then owns kDdRows / kDdWarps consecutive destination rows and walks their
// sources as one run (batches of gathers may cross a row boundary; a row is
// stored when its last source is added), in the same order as dd_kernel:
// the result is bitwise the same (Sec. 4.2.3, Eq. (3)).
constexpr int kDdRows = 128;     // destination rows per CTA
constexpr int kDdWarps = 16;     // warps per CTA
constexpr int kDdMaxSrc = 16384; // sources of one document the shared-memory sort takes (Nq * Lq)
constexpr int kDdGather = 16;    // source rows loaded together

inline size_t dd_fused_smem(int32_t nsrc) {
    // slot byte per source, per-warp histograms, row starts, the sorted sources (u16)
    return static_cast<size_t>(nsrc) + kDdWarps * kDdRows * 4 + (kDdRows + 1) * 4 + 2 * static_cast<size_t>(nsrc) +
           16;
}

template <int kVec, bool kBf16>
__global__ void __launch_bounds__(32 * kDdWarps, 2) dd_fused_kernel(const BwdArgs b) {
    constexpr int kG = kVec <= 4 ? kDdGather : kDdGather / 2;  // wide rows: fewer in flight (registers)
    extern __shared__ __align__(16) uint8_t dd_smem[];
    const int32_t nsrc = b.nq * b.lq;
    int32_t* hist = reinterpret_cast<int32_t*>(dd_smem);     // [kDdWarps][kDdRows], then offsets
    int32_t* rs = hist + kDdWarps * kDdRows;                 // [kDdRows + 1] row starts
    uint16_t* list = reinterpret_cast<uint16_t*>(rs + kDdRows + 1);  // [nsrc] sorted sources
    uint8_t* slot_of = reinterpret_cast<uint8_t*>(list + nsrc);      // [nsrc] slot, 0xFF = elsewhere
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t j = blockIdx.x;
    const int32_t t0 = blockIdx.y * kDdRows, t1 = min(t0 + kDdRows, b.ld);
    const int32_t nrows = t1 - t0;
    for (int32_t x = threadIdx.x; x < kDdWarps * kDdRows; x += blockDim.x) hist[x] = 0;
    __syncthreads();
    // 1. slots and per-warp counts; every argmax is checked once (slice 0)
    const int32_t per = (nsrc + kDdWarps - 1) / kDdWarps;
    const int32_t n0 = min(warp * per, nsrc), n1 = min(n0 + per, nsrc);
    bool bad = false;
#pragma unroll 4
    for (int32_t n = n0 + lane; n < n1; n += 32) {
        const int32_t a = b.argmax[src_index(b, j, n)];
        bad |= !argmax_ok(a, b.ld);
        const bool mine = a >= t0 && a < t1;
        slot_of[n] = mine ? static_cast<uint8_t>(a - t0) : 0xFFu;
        if (mine) atomicAdd(&hist[warp * kDdRows + (a - t0)], 1);
    }
    if (bad && blockIdx.y == 0 && b.status) atomicCAS(b.status, 0, 6);
    __syncthreads();
    // 2. exclusive scan over (row, warp), row-major: thread x owns four entries
    {
        constexpr int kPer = kDdRows * kDdWarps / (32 * kDdWarps);  // 4
        int32_t v[kPer], local = 0;
        const int x0 = threadIdx.x * kPer;  // flat index r * kDdWarps + w
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int x = x0 + q, r = x / kDdWarps, w = x % kDdWarps;
            v[q] = hist[w * kDdRows + r];
            local += v[q];
        }
        int32_t incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        __shared__ int32_t wsum[kDdWarps];
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int32_t before = 0;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        int32_t run = before + incl - local;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int x = x0 + q, r = x / kDdWarps, w = x % kDdWarps;
            if (w == 0) rs[r] = run;
            hist[w * kDdRows + r] = run;  // warp w's next free place in row r
            run += v[q];
        }
        if (threadIdx.x == blockDim.x - 1) rs[kDdRows] = run;
    }
    __syncthreads();
    // 3. stable placement: in a warp's run of sources, equal slots rank by lane
    for (int32_t nb = n0; nb < n1; nb += 32) {
        const int32_t n = nb + lane;
        const uint32_t sl = n < n1 ? slot_of[n] : 0xFFu;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, sl);
        if (sl != 0xFFu) {
            const int32_t rank = __popc(peers & ((1u << lane) - 1u));
            list[hist[warp * kDdRows + sl] + rank] = static_cast<uint16_t>(n);
            __syncwarp(peers);
            if ((peers >> lane) == 1u) hist[warp * kDdRows + sl] += __popc(peers);  // highest peer lane
        }
        __syncwarp();
    }
    __syncthreads();
    // 4. destination rows r0 .. r1-1 of this warp, their sources in one run
    constexpr int kRowsPerWarp = kDdRows / kDdWarps;
    const int32_t r0 = warp * kRowsPerWarp, r1 = min(r0 + kRowsPerWarp, nrows);
    if (r0 >= r1) return;
    float* out = b.dD + (static_cast<int64_t>(j) * b.ld + t0) * b.dim;
    float acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
    int32_t row = r0, row_end = rs[r0 + 1];
    const int32_t e_end = rs[r1];
    for (int32_t eb = rs[r0]; eb < e_end; eb += 32) {
        const int32_t cnt = min(32, e_end - eb);
        int32_t rowl = 0;  // Q row of this lane's source
        float wl = 0.f;
        if (lane < cnt) {
            const int32_t n = list[eb + lane];
            const int32_t i = n / b.lq, sq = n - (n / b.lq) * b.lq;
            rowl = i * b.lq + sq;
            wl = b.g[static_cast<int64_t>(i) * b.nd + j];
            if (b.q_mask && !b.q_mask[rowl]) wl = 0.f;
        }
        for (int32_t k = 0; k < cnt; k += kG) {
            RawRow<kVec> x[kG];
            float w[kG];
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                const int32_t src = min(k + u, cnt - 1);
                w[u] = __shfl_sync(0xFFFFFFFFu, wl, src);
                const int32_t r = __shfl_sync(0xFFFFFFFFu, rowl, src);
                load_raw<kVec>(b.Q + static_cast<int64_t>(r) * b.dim, lane, b.dim, x[u]);
            }
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                if (k + u < cnt) {
                    const int32_t e = eb + k + u;
                    while (e >= row_end) {  // the current row is complete (warp-uniform)
                        store_row<kVec>(out + static_cast<int64_t>(row) * b.dim, lane, b.dim, acc);
#pragma unroll
                        for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
                        ++row;
                        row_end = rs[row + 1];
                    }
                    fma_raw<kVec, kBf16>(w[u], x[u], acc);
                }
            }
        }
    }
    for (; row < r1; ++row) {  // the last row with sources, then rows without any
        store_row<kVec>(out + static_cast<int64_t>(row) * b.dim, lane, b.dim, acc);
#pragma unroll
        for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
    }
}

constexpr int kDqGather = 16;  // D rows loaded together by the dQ gather

// dQ: one warp per (query row (i, s), chunk of documents), ascending j. The
// winners and weights of 32 documents are loaded at once, one per lane. With
// one chunk the warp writes dQ; with several (gridDim.y > 1, many documents
// per query row) each chunk writes its partial row to `part` and
// dq_reduce_kernel adds the chunks in order: a fixed summation order either way.
template <int kVec, bool kBf16>
__global__ void __launch_bounds__(256, 4) dq_kernel(const BwdArgs b, float* __restrict__ part) {
    constexpr int kG = kVec <= 4 ? kDqGather : kDqGather / 2;  // wide rows: fewer in flight (registers)
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nrows = static_cast<int64_t>(b.nq) * b.lq;
    if (r >= nrows) return;
    const int32_t i = static_cast<int32_t>(r / b.lq);
    const int32_t s = static_cast<int32_t>(r - static_cast<int64_t>(i) * b.lq);
    if (s >= query_len(b, i)) return;  // no such row in packed Q
    const int64_t qr = query_row(b, i, s);
    const int32_t n_chunks = static_cast<int32_t>(gridDim.y);
    const int32_t per = (b.nd + n_chunks - 1) / n_chunks;
    const int32_t j_lo = static_cast<int32_t>(blockIdx.y) * per, j_hi = min(j_lo + per, b.nd);
    float acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
    for (int32_t jb = j_lo; jb < j_hi; jb += 32) {
        const int32_t cnt = min(32, j_hi - jb);
        int32_t rowl = -1;  // D row of this lane's document's winner (-1: none)
        float wl = 0.f;     // 0 for a document without a winner (argmax -1)
        if (lane < cnt) {
            const int32_t j = jb + lane;
            const int32_t a = b.argmax[(static_cast<int64_t>(i) * b.nd + j) * b.lq + s];
            if (a >= 0 && a < doc_len(b, j)) {
                wl = b.g[static_cast<int64_t>(i) * b.nd + j];
                rowl = static_cast<int32_t>(doc_row0(b, j) + a);
            }
        }
        for (int32_t k = 0; k < cnt; k += kG) {
            RawRow<kVec> x[kG];
            float w[kG];
            bool use[kG];
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                const int32_t src = min(k + u, cnt - 1);
                w[u] = __shfl_sync(0xFFFFFFFFu, wl, src);
                const int32_t r = __shfl_sync(0xFFFFFFFFu, rowl, src);
                use[u] = k + u < cnt && r >= 0;
                load_raw<kVec>(b.D + static_cast<int64_t>(r >= 0 ? r : 0) * b.dim, lane, b.dim, x[u]);
            }
#pragma unroll
            for (int u = 0; u < kG; ++u) {
                if (use[u]) fma_raw<kVec, kBf16>(w[u], x[u], acc);
            }
        }
    }
    const bool active = b.q_mask == nullptr || b.q_mask[qr] != 0;
    if (!active) {
#pragma unroll
        for (int v = 0; v < kVec; ++v) acc[v] = 0.f;
    }
    if (n_chunks == 1) store_row<kVec>(b.dQ + qr * b.dim, lane, b.dim, acc);
    else store_row<kVec>(part + (static_cast<int64_t>(blockIdx.y) * nrows + r) * b.dim, lane, b.dim, acc);
}

// dQ row (i, s) = the chunk partials added in chunk order.
__global__ void __launch_bounds__(256) dq_reduce_kernel(const BwdArgs b, const float* __restrict__ part,
                                                        int32_t n_chunks) {
    const int64_t nrows = static_cast<int64_t>(b.nq) * b.lq;
    const int64_t total = nrows * b.dim;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / b.dim;
        const int32_t i = static_cast<int32_t>(r / b.lq), s = static_cast<int32_t>(r % b.lq);
        if (s >= query_len(b, i)) continue;
        float v = part[e];
        for (int32_t c = 1; c < n_chunks; ++c) v = __fadd_rn(v, part[c * total + e]);
        b.dQ[query_row(b, i, s) * b.dim + (e - r * b.dim)] = v;
    }
}

}  // namespace maxsim
