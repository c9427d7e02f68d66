// Host side of the C ABI declared in include/maxsim.h: argument validation,
// launch planning (row blocks, document ranges, pipeline depth), TMA
// descriptor encoding, and the launches on the caller's stream.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "maxsim.h"
#include "bwd_kernels.cuh"
#include "chamfer_kernels.cuh"
#include "chamfer_tc.cuh"
#include "topk_kernels.cuh"
#include "fwd_kernel.cuh"

namespace maxsim {

// Device status word (first recorded problem wins; read and cleared by
// maxsim_device_status).
__device__ int g_device_status;

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s bound on any single device-side wait
constexpr int kMaxDevices = 64;
constexpr size_t kSmemBudget = 232448;          // 227 KB: opt-in shared memory per block on sm_100 / sm_103

struct DeviceInfo {
    bool init = false;
    int num_sms = 0;
    int smem_optin = 0;
    int* status = nullptr;
    bool attrs_set[16] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Armed by maxsim_debug_inject_wait_timeout; taken (and cleared) by the next
// forward launch.
std::atomic<uint64_t> g_inject_wait_ns{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

maxsim_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAXSIM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) return MAXSIM_ERR_UNSUPPORTED;  // built for sm_103a only
        if (static_cast<size_t>(d.smem_optin) < kSmemBudget) return MAXSIM_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return MAXSIM_ERR_CUDA;
        d.status = static_cast<int*>(p);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return MAXSIM_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.init = true;
    }
    *out = &d;
    return MAXSIM_OK;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline bool aligned16(const void* p) { return aligned(p, 16); }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 2-D row-major [rows, cols] tensor, loaded as box_cols x box_rows boxes with
// the 128-byte swizzle (the layout the tcgen05 descriptors expect).
bool encode_rows(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t cols,
                 uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- planning

struct FwdPlan {
    int64_t lq_pad = 0;
    int32_t rb_rows = 0, n_chunks = 1;
    int64_t n_rb = 0;
    int32_t k_atoms = 0, k8_atoms = 0, k_steps = 0, mt_max = 0, stages = 0, stages8 = 0;
    int64_t rows = 0;  // padded query rows
    bool repack = false, int8 = false, ok = false;
    bool pair = false;   // two-CTA clusters (each CTA loads half of every document tile)
    int64_t n_pr = 0;    // row-block pairs
    size_t smem = 0;
    size_t off_q = 0, off_real = 0, off_active = 0, off_qscale = 0, off_partial = 0, ws_bytes = 0;
};

inline int64_t pad_lq(int64_t lq) {
    if (lq <= 16) {
        int64_t p = 1;
        while (p < lq) p <<= 1;
        return p;
    }
    return (lq + 31) / 32 * 32;
}

size_t fwd_smem_bytes(int32_t mt, int32_t k_atoms, int32_t stages, int32_t k8_atoms, int32_t stages8, bool pair) {
    const size_t d_atom = static_cast<size_t>(pair ? kBN / 2 : kBN) * 128;
    const size_t q_bytes = static_cast<size_t>(mt) * k_atoms * kAtomBytes;
    size_t b = 1024 + q_bytes + static_cast<size_t>(stages) * k_atoms * d_atom + sizeof(SmemCtl);
    if (stages8 > 0) b += static_cast<size_t>(stages8) * k8_atoms * d_atom + kDScaleBytes;
    return b;
}

// Resident query M-tiles and ring depths: the most query rows per pass (up to
// mt_cap M-tiles), then
// the deepest document rings that fit (the 16-bit operand ring keeps two
// stages when it can; wide INT8 rows fall back to one). Returns false when
// nothing fits; the entry points then reject the shape.
bool choose_pipeline(FwdPlan& p, int32_t mt_cap) {
    for (int32_t min_stages = 2; min_stages >= 1; --min_stages) {
        for (int32_t mt = std::min(kMaxMT, mt_cap); mt >= 1; --mt) {
            if (!p.int8) {
                if (min_stages < 2 || fwd_smem_bytes(mt, p.k_atoms, 2, 0, 0, p.pair) > kSmemBudget) continue;
                int32_t s = kMaxStages;
                while (fwd_smem_bytes(mt, p.k_atoms, s, 0, 0, p.pair) > kSmemBudget) --s;
                p.mt_max = mt;
                p.stages = s;
                p.stages8 = 0;
            } else {
                if (fwd_smem_bytes(mt, p.k_atoms, min_stages, p.k8_atoms, 2, p.pair) > kSmemBudget) continue;
                int32_t s8 = kMaxStages;
                while (fwd_smem_bytes(mt, p.k_atoms, min_stages, p.k8_atoms, s8, p.pair) > kSmemBudget) --s8;
                p.mt_max = mt;
                p.stages = min_stages;
                p.stages8 = s8;
            }
            p.smem = fwd_smem_bytes(p.mt_max, p.k_atoms, p.stages, p.k8_atoms, p.stages8, p.pair);
            return true;
        }
    }
    return false;
}

FwdPlan plan_fwd_mode(int64_t nq, int64_t lq, int64_t nd, int64_t dim, bool varlen_q, bool int8, bool pair,
                      bool one_query_units) {
    FwdPlan p;
    p.int8 = int8;
    p.pair = pair;
    p.lq_pad = pad_lq(lq);
    p.k_atoms = static_cast<int32_t>((dim + 63) / 64);
    p.k8_atoms = int8 ? static_cast<int32_t>((dim + 127) / 128) : 0;
    p.k_steps = static_cast<int32_t>(dim / 16);
    // resident query M-tiles: no more than one pass over the call's query rows needs
    // (the memory left goes to the document ring)
    const int64_t pass_rows =
        std::min<int64_t>(std::max<int64_t>(one_query_units ? p.lq_pad : nq * p.lq_pad, 1), kBM * kMaxMT);
    p.ok = choose_pipeline(p, static_cast<int32_t>((pass_rows + kBM - 1) / kBM));
    if (!p.ok) p.mt_max = 1;  // keeps the sizes below defined; the entry points reject the shape
    const int64_t rb_max = static_cast<int64_t>(kBM) * p.mt_max;
    if (p.lq_pad <= rb_max) {
        int64_t qpb = rb_max / p.lq_pad;
        p.rb_rows = static_cast<int32_t>(qpb * p.lq_pad);
        p.n_chunks = 1;
        p.n_rb = (nq + qpb - 1) / qpb;
    } else {
        p.rb_rows = static_cast<int32_t>(rb_max);
        p.n_chunks = static_cast<int32_t>((p.lq_pad + rb_max - 1) / rb_max);
        p.n_rb = nq * p.n_chunks;
    }
    p.rows = nq * p.lq_pad;
    p.n_pr = (p.n_rb + 1) / 2;
    p.repack = int8 || varlen_q || p.lq_pad != lq;
    size_t off = 0;
    if (p.repack) {
        p.off_q = off;
        off = round_up(off + static_cast<size_t>(p.rows) * dim * 2, 256);  // 16-bit operand rows
        p.off_real = off;
        off = round_up(off + static_cast<size_t>(p.rows), 256);
        p.off_active = off;
        off = round_up(off + static_cast<size_t>(p.rows), 256);
    }
    if (int8) {
        p.off_qscale = off;
        off = round_up(off + static_cast<size_t>(p.rows) * sizeof(float), 256);
    }
    if (p.n_chunks > 1) {
        p.off_partial = off;
        off = round_up(off + static_cast<size_t>(p.n_chunks) * nq * nd * sizeof(float), 256);
    }
    p.ws_bytes = off;
    return p;
}

// Pair mode whenever there are at least two row blocks: each SM then reads
// from shared memory its own query rows and only half of every document tile
// per MMA, so the MMAs run at the tensor rate (the single-CTA kernel is bound
// by shared-memory operand reads at the short tiles of varlen documents), and
// for INT8 the staging ring and the 16-bit operand ring fit beside four
// resident query M-tiles. The pair-list walk (pair_list = true) runs on
// single CTAs, one query per unit.
FwdPlan plan_fwd(int64_t nq, int64_t lq, int64_t nd, int64_t dim, bool varlen_q, bool int8, bool pair_list = false) {
    FwdPlan p = plan_fwd_mode(nq, lq, nd, dim, varlen_q, int8, false, pair_list);
    if (!pair_list && p.ok && p.n_rb >= 2) {
        FwdPlan q = plan_fwd_mode(nq, lq, nd, dim, varlen_q, int8, true, false);
        if (q.ok && q.n_rb >= 2) return q;
    }
    return p;
}

// Document ranges per row group. A worker (an SM, or an SM pair) runs units
// u, u + workers, ...: each unit is one row group over 1/n_dr of the document
// tokens, so a worker's load is ceil(units / workers) / n_dr. Among 1, 2, 4 or
// 8 ranges per worker and group ("waves") take the smallest load, and the
// fewest units on a tie (each unit start reloads the query tile and drains
// the MMA pipeline).
int64_t choose_doc_ranges(int64_t n_rb, int64_t total_d, int64_t nd, int num_sms) {
    if (nd == 0) return 1;
    const int64_t workers = std::max(1, num_sms);
    const int64_t cap = std::min<int64_t>(nd, std::max<int64_t>(1, total_d / 256));
    int64_t best = 1;
    double best_load = 0.0;
    for (int64_t waves = 1; waves <= 8; waves *= 2) {
        const int64_t n_dr = std::max<int64_t>(1, std::min<int64_t>((workers * waves + n_rb - 1) / n_rb, cap));
        const int64_t units = n_dr * n_rb;
        const double load = static_cast<double>((units + workers - 1) / workers) / static_cast<double>(n_dr);
        if (waves == 1 || load < best_load * (1.0 - 1e-9)) {
            best = n_dr;
            best_load = load;
        }
    }
    return best;
}

// ---------------------------------------------------------------- small kernels

// Query rows into the padded layout [Nq * lq_pad, dim] of 16-bit values, with
// per-row flags (real token, active token) and, for INT8 queries, the row's
// scale. INT8 values are converted to binary16 exactly.
template <bool kInt8In>
__global__ void repack_q_kernel(const void* __restrict__ q, const int32_t* __restrict__ cu_q, int64_t lq_dense,
                                int64_t lq_pad, int64_t nq, int64_t dim, const uint8_t* __restrict__ q_mask,
                                const float* __restrict__ q_scale_in, uint16_t* __restrict__ qp,
                                uint8_t* __restrict__ real, uint8_t* __restrict__ active,
                                float* __restrict__ q_scale_out) {
    const int64_t rows = nq * lq_pad;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.y) + threadIdx.y; r < rows;
         r += static_cast<int64_t>(gridDim.x) * blockDim.y) {
        const int64_t i = r / lq_pad, s = r - (r / lq_pad) * lq_pad;
        const int64_t start = cu_q ? cu_q[i] : i * lq_dense;
        const int64_t len = cu_q ? static_cast<int64_t>(cu_q[i + 1]) - cu_q[i] : lq_dense;
        const bool is_real = s < len;
        const int64_t src = start + s;
        for (int64_t k = threadIdx.x; k < dim; k += blockDim.x) {
            uint16_t v = 0;
            if (is_real) {
                if constexpr (kInt8In) {
                    v = __half_as_ushort(__int2half_rn(static_cast<const int8_t*>(q)[src * dim + k]));
                } else {
                    v = static_cast<const uint16_t*>(q)[src * dim + k];
                }
            }
            qp[r * dim + k] = v;
        }
        if (threadIdx.x == 0) {
            real[r] = is_real ? 1 : 0;
            active[r] = (is_real && (q_mask == nullptr || q_mask[src] != 0)) ? 1 : 0;
            if (q_scale_out) q_scale_out[r] = is_real ? q_scale_in[src] : 0.f;
        }
    }
}

__global__ void sum_chunks_kernel(const float* __restrict__ partial, int32_t n_chunks, int64_t n,
                                  float* __restrict__ scores) {
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float s = 0.f;
        for (int32_t c = 0; c < n_chunks; ++c) s += partial[c * n + x];
        scores[x] = s;
    }
}

__global__ void check_cu_kernel(const int32_t* __restrict__ cu, int64_t n, int64_t total, int* status) {
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x <= n;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        bool bad = false;
        if (x == 0 && cu[0] != 0) bad = true;
        if (x == n && total >= 0 && cu[n] != total) bad = true;
        if (x < n && cu[x + 1] < cu[x]) bad = true;
        if (bad) atomicCAS(status, 0, kStatusBadInput);
    }
}

__global__ void fill_kernel(float* scores, int64_t ns, int32_t* argmax, int64_t na) {
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < ns + na;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (x < ns) scores[x] = 0.f;
        else argmax[x - ns] = -1;
    }
}

// INT8: the exact integer dot product at each argmax (0 where there is none).
// One thread per (i, j, s), 4-byte dot-product steps.
__global__ void win_dot_kernel(const int8_t* __restrict__ q, const int8_t* __restrict__ d,
                               const int32_t* __restrict__ argmax, int64_t nq, int64_t lq, int64_t nd, int64_t ld,
                               int64_t dim, int32_t* __restrict__ win) {
    const int64_t n = nq * nd * lq;
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t s = x % lq, ij = x / lq;
        const int64_t i = ij / nd, j = ij - (ij / nd) * nd;
        const int32_t a = argmax[x];
        int32_t acc = 0;
        if (a >= 0 && a < ld) {
            const int* qr = reinterpret_cast<const int*>(q + (i * lq + s) * dim);
            const int* dr = reinterpret_cast<const int*>(d + (j * ld + a) * dim);
            for (int64_t k = 0; k < dim / 4; ++k) acc = __dp4a(qr[k], dr[k], acc);
        }
        win[x] = acc;
    }
}

inline int grid_for(int64_t n, int per_block, int num_sms) {
    int64_t g = (n + per_block - 1) / per_block;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, static_cast<int64_t>(num_sms) * 8)));
}

template <bool kArg, bool kInt8, bool kPair>
maxsim_status launch_fwd_kernel(DeviceInfo* dev, int slot, const CUtensorMap& tq, const CUtensorMap& td,
                                const FwdArgs& a, size_t smem, int grid, cudaStream_t st) {
    auto kern = maxsim_fwd_kernel<kArg, kInt8, kPair>;
    if (!dev->attrs_set[slot]) {
        // The kernel moves registers between its warpgroups (setmaxnreg): the
        // split only adds up if every thread was launched with kRegsLaunch.
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return MAXSIM_ERR_CUDA;
        if (fa.numRegs < kRegsLaunch) return MAXSIM_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev->smem_optin) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        dev->attrs_set[slot] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, td, a) != cudaSuccess) return MAXSIM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

// Shared path of the forward entry points once the query rows are 16-bit rows
// in device memory: Q as padded rows [rows, dim] (possibly in the workspace),
// D as packed token rows [total_d, dim] (16-bit, or INT8 in INT8 mode).
struct FwdCall {
    const void* q_rows;
    const uint8_t* q_real;
    const uint8_t* q_active;
    const float* q_scale;
    const void* d_rows;
    const float* d_scale;
    CUtensorMapDataType q_dt, d_dt;
    uint32_t ab_format;   // 0 = f16, 1 = bf16
    uint32_t nan_pair;
    int64_t nq, lq_out, nd, ld, total_d, dim;
    const int32_t* cu_d;
    const uint8_t* d_mask;
    float* scores;
    int32_t* argmax;
    // pair-list mode (score_pairs_packed), else all NULL / 0
    const int32_t* pr_pairs;
    const int32_t* pr_sorted;
    const int32_t* pr_qptr;
    const int32_t* pr_uptr;
    int32_t pr_chunk;
};

maxsim_status run_fwd(DeviceInfo* dev, const FwdPlan& p, const FwdCall& c, uint8_t* ws, cudaStream_t st) {
    if (!p.ok || p.stages < 1 || p.stages > kMaxStages || (p.int8 && (p.stages8 < 1 || p.stages8 > kMaxStages)) ||
        p.smem > kSmemBudget)
        return MAXSIM_ERR_UNSUPPORTED;
    CUtensorMap tq, td;
    if (!encode_rows(&tq, c.q_rows, c.q_dt, 2, static_cast<uint64_t>(c.dim), static_cast<uint64_t>(p.rows), 64, kBM))
        return MAXSIM_ERR_CUDA;
    // With no document tokens the D map is never read; point it at Q.
    const bool has_d = c.total_d > 0;
    const int d_elem = p.int8 ? 1 : 2;
    const uint32_t d_box_rows = p.pair ? kBN / 2 : kBN;
    if (has_d) {
        if (!encode_rows(&td, c.d_rows, c.d_dt, d_elem, static_cast<uint64_t>(c.dim), static_cast<uint64_t>(c.total_d),
                         p.int8 ? 128 : 64, d_box_rows))
            return MAXSIM_ERR_CUDA;
    } else if (!encode_rows(&td, c.q_rows, c.q_dt, 2, static_cast<uint64_t>(c.dim), static_cast<uint64_t>(p.rows), 64,
                            d_box_rows)) {
        return MAXSIM_ERR_CUDA;
    }

    FwdArgs a{};
    a.nq = static_cast<int32_t>(c.nq);
    a.lq_pad = static_cast<int32_t>(p.lq_pad);
    a.lq_out = static_cast<int32_t>(c.lq_out);
    a.q_active = c.q_active;
    a.q_real = c.q_real;
    a.q_scale = c.q_scale;
    a.rb_rows = p.rb_rows;
    a.n_chunks = p.n_chunks;
    a.n_rb = static_cast<int32_t>(p.n_rb);
    a.cu_d = c.cu_d;
    a.nd = static_cast<int32_t>(c.nd);
    a.ld = static_cast<int32_t>(c.ld);
    a.total_d = static_cast<int32_t>(c.total_d);
    a.d_mask = c.d_mask;
    a.d_scale = c.d_scale;
    // workers: SMs, or SM pairs in pair mode; row groups: row blocks, or their pairs
    const int workers = p.pair ? dev->num_sms / 2 : dev->num_sms;
    const int64_t groups = p.pair ? p.n_pr : p.n_rb;
    const int64_t n_dr = choose_doc_ranges(groups, c.total_d, c.nd, workers);
    a.n_dr = static_cast<int32_t>(n_dr);
    a.n_units = static_cast<int32_t>(n_dr * groups);
    a.n_pr = static_cast<int32_t>(p.n_pr);
    a.scores = c.scores;
    a.partial = p.n_chunks > 1 ? reinterpret_cast<float*>(ws + p.off_partial) : nullptr;
    a.argmax = c.argmax;
    a.k_steps = p.k_steps;
    a.k_atoms = p.k_atoms;
    a.k8_atoms = p.k8_atoms;
    a.dim = static_cast<int32_t>(c.dim);
    a.stages = p.stages;
    a.stages8 = p.stages8;
    a.q_slots = p.mt_max;
    a.idesc = idesc_f16_f32(c.ab_format, 0, 0);  // M and N are filled in on the device
    a.nan_pair = c.nan_pair;
    a.status = dev->status;
    a.timeout_ns = kTimeoutNs;
    a.inject_wait_ns = g_inject_wait_ns.exchange(0);
    // One CTA per SM: the request always exceeds half of an SM's shared memory.
    const size_t smem = std::max<size_t>(p.smem, kSmemBudget / 2 + 1024);
    a.pr_pairs = c.pr_pairs;
    a.pr_sorted = c.pr_sorted;
    a.pr_qptr = c.pr_qptr;
    a.pr_uptr = c.pr_uptr;
    a.pr_chunk = c.pr_chunk;
    if (c.pr_sorted && p.pair) return MAXSIM_ERR_UNSUPPORTED;
    // pair-list mode: the unit count is known on the device only; every SM runs
    const int grid = c.pr_sorted ? workers
                   : p.pair ? 2 * static_cast<int>(std::min<int64_t>(a.n_units, workers))
                            : static_cast<int>(std::min<int64_t>(a.n_units, workers));

    maxsim_status rc;
    const bool arg = c.argmax != nullptr;
    if (p.pair) {
        if (p.int8) rc = arg ? launch_fwd_kernel<true, true, true>(dev, 8, tq, td, a, smem, grid, st)
                             : launch_fwd_kernel<false, true, true>(dev, 9, tq, td, a, smem, grid, st);
        else rc = arg ? launch_fwd_kernel<true, false, true>(dev, 10, tq, td, a, smem, grid, st)
                      : launch_fwd_kernel<false, false, true>(dev, 11, tq, td, a, smem, grid, st);
    } else {
        if (p.int8) rc = arg ? launch_fwd_kernel<true, true, false>(dev, 0, tq, td, a, smem, grid, st)
                             : launch_fwd_kernel<false, true, false>(dev, 1, tq, td, a, smem, grid, st);
        else rc = arg ? launch_fwd_kernel<true, false, false>(dev, 2, tq, td, a, smem, grid, st)
                      : launch_fwd_kernel<false, false, false>(dev, 3, tq, td, a, smem, grid, st);
    }
    if (rc != MAXSIM_OK) return rc;
    if (p.n_chunks > 1) {
        const int64_t n = c.nq * c.nd;
        sum_chunks_kernel<<<grid_for(n, 256, dev->num_sms), 256, 0, st>>>(a.partial, p.n_chunks, n, c.scores);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    return MAXSIM_OK;
}

// ---------------------------------------------------------------- pair lists

// Valid pairs counted per query; a pair outside [0, Nq) x [0, Nd) scores 0,
// its argmax row is -1, and it is reported on the device status word. The
// lanes of a warp that hold pairs of the same query add their count with one
// atomic (pair lists usually come grouped by query, so one per warp).
__global__ void pairs_count_kernel(const int32_t* __restrict__ pairs, int64_t np, int64_t nq, int64_t nd,
                                   int32_t* __restrict__ qcnt, float* __restrict__ scores, int32_t* __restrict__ argmax,
                                   int64_t lq_out, int* status) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    // every lane of a warp runs the same iterations (warp-wide match below)
    for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x - lane; base < np;
         base += stride) {
        const int64_t p = base + lane;
        int32_t key = -2;  // -2: no pair in this lane, -1: an invalid pair
        if (p < np) {
            const int32_t q = pairs[2 * p], d = pairs[2 * p + 1];
            key = (q >= 0 && q < nq && d >= 0 && d < nd) ? q : -1;
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        if (key >= 0) {
            if (qcnt && lane == __ffs(peers) - 1) atomicAdd(qcnt + key, __popc(peers));
        } else if (key == -1) {
            scores[p] = 0.f;
            if (argmax)
                for (int64_t s = 0; s < lq_out; ++s) argmax[p * lq_out + s] = -1;
            atomicCAS(status, 0, kStatusBadInput);
        }
    }
}

// One block: exclusive prefix sums over the queries of their pair counts
// (qptr, also copied to the placement cursors) and of their unit counts
// ceil(count / chunk) (uptr); qptr[nq] and uptr[nq] hold the totals.
__global__ void __launch_bounds__(1024) pairs_scan_kernel(const int32_t* __restrict__ qcnt, int64_t nq, int32_t chunk,
                                                          int32_t* __restrict__ qptr, int32_t* __restrict__ uptr,
                                                          int32_t* __restrict__ cursor) {
    __shared__ int32_t wsum[2][32];
    __shared__ int32_t carry[2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    for (int64_t base = 0; base < nq; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const int32_t c = i < nq ? qcnt[i] : 0;
        int32_t v[2] = {c, (c + chunk - 1) / chunk};
        int32_t x[2] = {v[0], v[1]};
#pragma unroll
        for (int h = 0; h < 2; ++h)
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x[h], o);
                if (lane >= o) x[h] += y;
            }
        if (lane == 31) { wsum[0][warp] = x[0]; wsum[1][warp] = x[1]; }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int32_t w = lane < static_cast<int>(blockDim.x >> 5) ? wsum[h][lane] : 0;
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                    if (lane >= o) w += y;
                }
                wsum[h][lane] = w;  // inclusive
            }
        }
        __syncthreads();
        int32_t ex[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) ex[h] = carry[h] + (warp > 0 ? wsum[h][warp - 1] : 0) + x[h] - v[h];
        if (i < nq) {
            qptr[i] = ex[0];
            cursor[i] = ex[0];
            uptr[i] = ex[1];
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            carry[0] = ex[0] + v[0];
            carry[1] = ex[1] + v[1];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        qptr[nq] = carry[0];
        uptr[nq] = carry[1];
    }
}

// Each valid pair to a free slot of its query. The order inside a query's
// group is free: every pair is scored on its own. The lanes of a warp with
// pairs of the same query reserve their slots with one atomic.
__global__ void pairs_place_kernel(const int32_t* __restrict__ pairs, int64_t np, int64_t nq, int64_t nd,
                                   int32_t* __restrict__ cursor, int32_t* __restrict__ sorted) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x - lane; base < np;
         base += stride) {
        const int64_t p = base + lane;
        int32_t key = -1;
        if (p < np) {
            const int32_t q = pairs[2 * p], d = pairs[2 * p + 1];
            if (q >= 0 && q < nq && d >= 0 && d < nd) key = q;
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        if (key >= 0) {
            const int leader = __ffs(peers) - 1;
            int32_t slot = 0;
            if (lane == leader) slot = atomicAdd(cursor + key, __popc(peers));
            slot = __shfl_sync(peers, slot, leader) + __popc(peers & ((1u << lane) - 1u));
            sorted[slot] = static_cast<int32_t>(p);
        }
    }
}

// Workspace of the pair-list forward: the varlen plan's, then the grouping.
struct PairsWs {
    size_t off_qcnt = 0, off_qptr = 0, off_uptr = 0, off_cursor = 0, off_sorted = 0, bytes = 0;
};

PairsWs pairs_ws(size_t base, int64_t nq, int64_t np) {
    PairsWs w;
    size_t off = round_up(base, 256);
    w.off_qcnt = off;
    off = round_up(off + static_cast<size_t>(nq) * 4, 256);
    w.off_qptr = off;
    off = round_up(off + static_cast<size_t>(nq + 1) * 4, 256);
    w.off_uptr = off;
    off = round_up(off + static_cast<size_t>(nq + 1) * 4, 256);
    w.off_cursor = off;
    off = round_up(off + static_cast<size_t>(nq) * 4, 256);
    w.off_sorted = off;
    off = round_up(off + static_cast<size_t>(np) * 4, 256);
    w.bytes = off;
    return w;
}

maxsim_status check_dim(int64_t dim, int64_t multiple) {
    if (dim <= 0) return MAXSIM_ERR_INVALID_ARG;
    if (dim % multiple != 0 || dim > 256) return MAXSIM_ERR_UNSUPPORTED;
    return MAXSIM_OK;
}

constexpr int64_t kI32Max = 2147483647;
constexpr uint32_t kNaNPairF16 = 0x7E007E00u;
constexpr uint32_t kNaNPairBF16 = 0x7FC07FC0u;

inline CUtensorMapDataType half_map(maxsim_dtype dt) {
    return dt == MAXSIM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}


// ---------------------------------------------------------------- Chamfer planning

struct ChamferFwdPlan {
    int64_t n_sb[2] = {0, 0}, n_span[2] = {0, 0}, n_mblk[2] = {0, 0};
    int64_t items0 = 0, items = 0;
    size_t off_counter = 0, off_best[2] = {0, 0}, off_sub[2] = {0, 0}, off_loss[2] = {0, 0}, ws_bytes = 0;
    int kd = 3;
};

ChamferFwdPlan plan_chamfer_fwd(int64_t B, int64_t N, int64_t M, int64_t dim) {
    ChamferFwdPlan p;
    p.kd = dim <= 3 ? 3 : kChMaxDim;
    const int64_t per_item = p.kd == 3 ? ChamferShape<3>::kSources : ChamferShape<kChMaxDim>::kSources;
    const int64_t nx[2] = {N, M}, ny[2] = {M, N};
    size_t off = 256;  // the work counter
    for (int d = 0; d < 2; ++d) {
        p.n_sb[d] = (nx[d] + per_item - 1) / per_item;
        p.n_span[d] = (ny[d] + kChSpan - 1) / kChSpan;
        p.n_mblk[d] = (nx[d] + kChMergeThreads - 1) / kChMergeThreads;
        const size_t n_part = static_cast<size_t>(p.n_span[d]) * static_cast<size_t>(B * nx[d]);
        p.off_best[d] = off;
        off = round_up(off + n_part * 4, 256);
        p.off_sub[d] = off;
        off = round_up(off + n_part * 4, 256);
        p.off_loss[d] = off;
        off = round_up(off + static_cast<size_t>(B * p.n_mblk[d]) * 8, 256);
    }
    p.items0 = B * p.n_sb[0] * p.n_span[0];
    p.items = p.items0 + B * p.n_sb[1] * p.n_span[1];
    p.ws_bytes = off;
    return p;
}

// Tensor-core nearest-point search (dim <= kTcMaxDim): augmented operand rows
// of both sets, partial results per target span, loss partials.
struct ChamferTcPlan {
    int64_t s_rows[2] = {0, 0}, t_rows[2] = {0, 0};  // per set of P (0) and Q (1)
    int64_t n_sb[2] = {0, 0}, n_span[2] = {0, 0}, n_mblk[2] = {0, 0};  // per direction
    int64_t items = 0;
    size_t off_s[2] = {0, 0}, off_t[2] = {0, 0}, off_best[2] = {0, 0}, off_idx[2] = {0, 0}, off_loss[2] = {0, 0};
    size_t ws_bytes = 0;
};

ChamferTcPlan plan_chamfer_tc(int64_t B, int64_t N, int64_t M) {
    ChamferTcPlan p;
    const int64_t n[2] = {N, M};
    size_t off = 0;
    for (int c = 0; c < 2; ++c) {  // operand rows of P and of Q
        p.s_rows[c] = (n[c] + kTcSources - 1) / kTcSources * kTcSources;
        p.t_rows[c] = (n[c] + kTcN - 1) / kTcN * kTcN;
        p.off_s[c] = off;
        off = round_up(off + static_cast<size_t>(B * p.s_rows[c]) * kTcRowBytes, 1024);
        p.off_t[c] = off;
        off = round_up(off + static_cast<size_t>(B * p.t_rows[c]) * kTcRowBytes, 1024);
    }
    const int64_t nx[2] = {N, M}, ny[2] = {M, N};
    for (int d = 0; d < 2; ++d) {
        p.n_sb[d] = (nx[d] + kTcSources - 1) / kTcSources;
        p.n_span[d] = (ny[d] + kTcSpan - 1) / kTcSpan;
        p.n_mblk[d] = (nx[d] + 255) / 256;
        const size_t n_part = static_cast<size_t>(p.n_span[d]) * static_cast<size_t>(B * nx[d]);
        p.off_best[d] = off;
        off = round_up(off + n_part * 4, 256);
        p.off_idx[d] = off;
        off = round_up(off + n_part * 4, 256);
        p.off_loss[d] = off;
        off = round_up(off + static_cast<size_t>(B * p.n_mblk[d]) * 8, 256);
    }
    p.items = (N > 0 && M > 0) ? B * (p.n_sb[0] * p.n_span[0] + p.n_sb[1] * p.n_span[1]) : 0;
    p.ws_bytes = off;
    return p;
}

constexpr size_t kTcSmemBytes = static_cast<size_t>(kTcMT) * kTcATile + static_cast<size_t>(kTcStages) * kTcBTile +
                                2ull * 4 * kTcSources * 4 + sizeof(TcSmemCtl) + 1024;

// [rows, 16] fp32 rows with the 64-byte swizzle, box_rows rows per load.
bool encode_rows_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTcK), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kTcRowBytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct ChamferBwdPlan {
    int64_t K = 0, nblocks = 0, hist_n = 0;
    int passes = 0;
    size_t off_keys[2] = {0, 0}, off_vals[2] = {0, 0}, off_hist = 0, off_row = 0, ws_bytes = 0;
};

ChamferBwdPlan plan_chamfer_bwd(int64_t B, int64_t N, int64_t M) {
    ChamferBwdPlan p;
    p.K = B * (N + M);
    p.nblocks = (p.K + kRadixBlock - 1) / kRadixBlock;
    p.hist_n = p.nblocks * kRadixBins;
    int bits = 0;
    while (bits < 32 && (int64_t(1) << bits) <= p.K) ++bits;  // keys are in [0, K]
    p.passes = (bits + kRadixBits - 1) / kRadixBits;
    size_t off = 0;
    for (int i = 0; i < 2; ++i) {
        p.off_keys[i] = off;
        off = round_up(off + static_cast<size_t>(p.K) * 4, 256);
        p.off_vals[i] = off;
        off = round_up(off + static_cast<size_t>(p.K) * 4, 256);
    }
    p.off_hist = off;
    off = round_up(off + static_cast<size_t>(p.hist_n) * 4, 256);
    p.off_row = off;
    off = round_up(off + static_cast<size_t>(p.K + 1) * 4, 256);
    p.ws_bytes = p.K > 0 ? off : 0;
    return p;
}

maxsim_status check_chamfer_shape(int64_t B, int64_t N, int64_t M, int64_t dim) {
    if (B < 0 || N < 0 || M < 0 || dim <= 0) return MAXSIM_ERR_INVALID_ARG;
    if (dim > kChMaxDim) return MAXSIM_ERR_UNSUPPORTED;
    if (B * (N + M) >= kI32Max || B * (N + M) * dim >= (int64_t(1) << 40)) return MAXSIM_ERR_UNSUPPORTED;
    return MAXSIM_OK;
}

maxsim_status chamfer_fwd_tc(DeviceInfo* dev, const ChamferTcPlan& p, const float* P, const float* Q, int64_t B,
                             int64_t N, int64_t M, int64_t dim, float* dist_p, int32_t* idx_p, float* dist_q,
                             int32_t* idx_q, float* loss, uint8_t* ws, cudaStream_t st) {
    ChamferFwdArgs a{};
    a.X[0] = P; a.Y[0] = Q; a.X[1] = Q; a.Y[1] = P;
    a.nx[0] = N; a.ny[0] = M; a.nx[1] = M; a.ny[1] = N;
    a.B = B;
    a.dim = static_cast<int32_t>(dim);
    a.dist[0] = dist_p; a.idx[0] = idx_p; a.dist[1] = dist_q; a.idx[1] = idx_q;
    a.loss = loss;
    a.status = dev->status;
    ChamferTcArgs t{};
    t.B = B;
    t.items = p.items;
    t.status = dev->status;
    t.timeout_ns = kTimeoutNs;
    const int64_t n[2] = {N, M};
    for (int d = 0; d < 2; ++d) {
        t.nx[d] = a.nx[d];
        t.ny[d] = a.ny[d];
        t.n_sb[d] = p.n_sb[d];
        t.n_span[d] = p.n_span[d];
        t.part_best[d] = reinterpret_cast<float*>(ws + p.off_best[d]);
        t.part_idx[d] = reinterpret_cast<int32_t*>(ws + p.off_idx[d]);
        a.n_mblk[d] = p.n_mblk[d];
        a.loss_part[d] = reinterpret_cast<double*>(ws + p.off_loss[d]);
    }
    // direction 0: sources P, targets Q; direction 1: sources Q, targets P
    t.s_rows[0] = p.s_rows[0]; t.t_rows[0] = p.t_rows[1];
    t.s_rows[1] = p.s_rows[1]; t.t_rows[1] = p.t_rows[0];
    if (p.items > 0) {
        const float* pts[2] = {P, Q};
        for (int c = 0; c < 2; ++c) {
            const int64_t rows = B * std::max(p.s_rows[c], p.t_rows[c]);
            chamfer_tc_prep_kernel<<<grid_for(rows, 256, dev->num_sms), 256, 0, st>>>(
                pts[c], B, n[c], static_cast<int32_t>(dim), p.s_rows[c], p.t_rows[c],
                reinterpret_cast<float*>(ws + p.off_s[c]), reinterpret_cast<float*>(ws + p.off_t[c]));
        }
        CUtensorMap ms0, mt0, ms1, mt1;
        if (!encode_rows_sw64(&ms0, ws + p.off_s[0], static_cast<uint64_t>(B * p.s_rows[0]), kTcM) ||
            !encode_rows_sw64(&mt0, ws + p.off_t[1], static_cast<uint64_t>(B * p.t_rows[1]), kTcN) ||
            !encode_rows_sw64(&ms1, ws + p.off_s[1], static_cast<uint64_t>(B * p.s_rows[1]), kTcM) ||
            !encode_rows_sw64(&mt1, ws + p.off_t[0], static_cast<uint64_t>(B * p.t_rows[0]), kTcN))
            return MAXSIM_ERR_CUDA;
        if (!dev->attrs_set[14]) {
            if (cudaFuncSetAttribute(chamfer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kTcSmemBytes)) != cudaSuccess)
                return MAXSIM_ERR_CUDA;
            dev->attrs_set[14] = true;
        }
        const int64_t grid = std::min<int64_t>(p.items, dev->num_sms);
        chamfer_tc_kernel<<<static_cast<unsigned>(grid), kTcThreads, kTcSmemBytes, st>>>(ms0, mt0, ms1, mt1, t);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    const int64_t mblk = std::max(p.n_mblk[0], p.n_mblk[1]);
    if (mblk > 0)
        chamfer_tc_merge_kernel<<<dim3(static_cast<unsigned>(mblk), static_cast<unsigned>(B), 2), 256, 0, st>>>(
            P, Q, static_cast<int32_t>(dim), t, a);
    chamfer_loss_kernel<<<static_cast<unsigned>(B), kChLossThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

template <int kD>
maxsim_status launch_chamfer_nn(DeviceInfo* dev, int slot, const ChamferFwdArgs& a, int64_t items, cudaStream_t st) {
    auto kern = chamfer_nn_kernel<kD>;
    const size_t smem = ChamferShape<kD>::kSmem;
    if (!dev->attrs_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return MAXSIM_ERR_CUDA;
        dev->attrs_set[slot] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kChThreads, smem) != cudaSuccess || per_sm < 1)
        return MAXSIM_ERR_CUDA;
    const int64_t grid = std::min<int64_t>(items, static_cast<int64_t>(dev->num_sms) * per_sm);
    kern<<<static_cast<unsigned>(grid), kChThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

inline int32_t pow2_at_least(int64_t k) {
    int32_t p = 1;
    while (p < k) p <<= 1;
    return p;
}

maxsim_status launch_topk(DeviceInfo* dev, const float* scores, int64_t rows, int64_t n, int64_t row_stride,
                          int64_t k, const int32_t* id_map, int64_t map_stride, int32_t* out_idx, float* out_val,
                          int64_t out_stride, cudaStream_t st) {
    (void)dev;
    if (rows == 0 || k == 0) return MAXSIM_OK;
    if (rows > 2147483647) return MAXSIM_ERR_UNSUPPORTED;
    TopkArgs t{};
    t.scores = scores;
    t.n = n;
    t.row_stride = row_stride;
    t.k = static_cast<int32_t>(k);
    t.pow2 = pow2_at_least(k);
    t.id_map = id_map;
    t.map_stride = map_stride;
    t.out_idx = out_idx;
    t.out_val = out_val;
    t.out_stride = out_stride;
    const size_t smem = static_cast<size_t>(t.pow2) * 8;  // keys and positions
    topk_kernel<<<static_cast<unsigned>(rows), kTopkThreads, smem, st>>>(t);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

struct TwoStagePlan {
    size_t off_s8 = 0, off_cand = 0, off_pairs = 0, off_cu = 0, off_s16 = 0, off_stage = 0, bytes = 0;
    size_t stage_bytes = 0;
    bool ok = false;
};

TwoStagePlan plan_two_stage(int64_t Nq, int64_t Lq, int64_t Nd, int64_t dim, int64_t k1) {
    TwoStagePlan p;
    const FwdPlan p8 = plan_fwd(Nq, Lq, Nd, dim, false, true);
    const FwdPlan p16 = plan_fwd(Nq, Lq, Nd, dim, true, false, true);
    if (!p8.ok || !p16.ok || p16.n_chunks > 1) return p;
    p.stage_bytes = std::max(p8.ws_bytes, pairs_ws(p16.ws_bytes, Nq, Nq * k1).bytes);
    size_t off = 0;
    p.off_s8 = off;
    off = round_up(off + static_cast<size_t>(Nq * Nd) * 4, 256);
    p.off_cand = off;
    off = round_up(off + static_cast<size_t>(Nq * k1) * 4, 256);
    p.off_pairs = off;
    off = round_up(off + static_cast<size_t>(Nq * k1) * 8, 256);
    p.off_cu = off;
    off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);
    p.off_s16 = off;
    off = round_up(off + static_cast<size_t>(Nq * k1) * 4, 256);
    p.off_stage = off;
    p.bytes = round_up(off + p.stage_bytes, 256);
    p.ok = true;
    return p;
}

struct StreamedPlan {
    int64_t blk = 0;
    size_t buf_bytes = 0, off_buf[2] = {0, 0}, off_scores = 0, off_fwd = 0, fwd_bytes = 0, bytes = 0;
    bool ok = false;
};

StreamedPlan plan_streamed(int64_t Nq, int64_t Lq, int64_t blk, int64_t Ld, int64_t dim, int64_t elem) {
    StreamedPlan p;
    const FwdPlan f = plan_fwd(Nq, Lq, blk, dim, false, false);
    if (!f.ok) return p;
    p.blk = blk;
    p.buf_bytes = static_cast<size_t>(blk * Ld * dim * elem);
    size_t off = 0;
    for (int i = 0; i < 2; ++i) {
        p.off_buf[i] = off;
        off = round_up(off + p.buf_bytes, 256);
    }
    p.off_scores = off;
    off = round_up(off + static_cast<size_t>(Nq * blk) * 4, 256);
    p.off_fwd = off;
    p.fwd_bytes = f.ws_bytes;
    p.bytes = round_up(off + f.ws_bytes, 256);
    p.ok = true;
    return p;
}

// Document chunks of the dQ gather: enough warps to fill the GPU when a query
// row has many documents to visit, at least 64 documents per chunk.
template <int kVec, bool kBf16>
maxsim_status launch_dd_fused(dim3 grid, size_t shm, cudaStream_t st, const BwdArgs& b) {
    if (shm > 48 * 1024 &&
        cudaFuncSetAttribute(dd_fused_kernel<kVec, kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(shm)) != cudaSuccess)
        return MAXSIM_ERR_CUDA;
    dd_fused_kernel<kVec, kBf16><<<grid, 32 * kDdWarps, shm, st>>>(b);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

template <int kVec>
maxsim_status launch_dd_fused_t(dim3 grid, size_t shm, cudaStream_t st, const BwdArgs& b) {
    return b.is_bf16 ? launch_dd_fused<kVec, true>(grid, shm, st, b) : launch_dd_fused<kVec, false>(grid, shm, st, b);
}

template <int kVec>
void launch_dq(dim3 grid, cudaStream_t st, const BwdArgs& b, float* part) {
    if (b.is_bf16) dq_kernel<kVec, true><<<grid, 256, 0, st>>>(b, part);
    else dq_kernel<kVec, false><<<grid, 256, 0, st>>>(b, part);
}

int32_t dq_chunks(int64_t Nq, int64_t lq, int64_t Nd) {
    const int64_t rows = std::max<int64_t>(1, Nq * lq);
    const int64_t want = (16384 + rows - 1) / rows;
    return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(want, Nd / 64)));
}

size_t bwd_ws_bytes(int64_t Nq, int64_t lq, int64_t Nd, int64_t d_rows, int64_t dim, bool have_rp, bool have_col) {
    size_t off = 0;
    off = round_up(off + static_cast<size_t>(Nd) * 4, 256);          // doc_cnt
    off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);      // doc_base
    if (!have_rp) off = round_up(off + static_cast<size_t>(d_rows + 1) * 4, 256);
    if (!have_col) off = round_up(off + static_cast<size_t>(Nq * Nd * lq) * 4, 256);
    const int32_t c = dq_chunks(Nq, lq, Nd);
    if (c > 1) off = round_up(off + static_cast<size_t>(c) * Nq * lq * dim * 4, 256);  // dQ partials
    return off;
}

// The backward's dQ gather and its dD reduction read the same inputs and
// write different outputs, so dQ runs on a library stream of its own beside
// the caller's: forked after the caller's earlier work, joined before the
// caller's later work. One stream and two events per device; the enqueue of a
// whole fork / launch / join sequence holds the lock, so calls from several
// host threads cannot interleave their events.
struct BwdSide {
    bool init = false;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_bwd_mu;
BwdSide g_bwd_side[kMaxDevices];

maxsim_status bwd_side(BwdSide** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAXSIM_ERR_CUDA;
    BwdSide& r = g_bwd_side[dev];
    if (!r.init) {
        if (cudaStreamCreateWithFlags(&r.stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        r.init = true;
    }
    *out = &r;
    return MAXSIM_OK;
}

// Backward for dense (cu_q = cu_d = NULL, ld = the document length) and
// packed layouts (cu_d given, ld = the longest document).
maxsim_status run_bwd(const void* Q, const int32_t* cu_q, int64_t Lq, const void* D, const int32_t* cu_d,
                      int64_t d_rows, int64_t Ld, maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                      const uint8_t* q_mask, const int32_t* argmax, const float* grad_scores, float* dQ, float* dD,
                      int32_t* csr_row_ptr, int32_t* csr_col, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd * Lq > kI32Max || d_rows >= kI32Max || Nd * Ld >= (int64_t(1) << 40)) return MAXSIM_ERR_UNSUPPORTED;
    // destination histograms: at least one warp's worth of Ld counters must fit
    if (Ld * 4 > 200 * 1024) return MAXSIM_ERR_UNSUPPORTED;
    const bool need_csr = dD || csr_row_ptr || csr_col;
    if (need_csr || dQ) {
        if (!argmax || !grad_scores) return MAXSIM_ERR_INVALID_ARG;
        if ((Nq * Lq > 0 && (!Q || !aligned16(Q))) || (d_rows > 0 && (!D || !aligned16(D))))
            return MAXSIM_ERR_INVALID_ARG;
    }
    // the gradient rows are written as whole vectors
    if ((dQ && !aligned16(dQ)) || (dD && !aligned16(dD))) return MAXSIM_ERR_INVALID_ARG;
    size_t off = 0;
    const size_t off_cnt = off;
    off = round_up(off + static_cast<size_t>(Nd) * 4, 256);
    const size_t off_base = off;
    off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);
    size_t off_rp = 0, off_col = 0, off_part = 0;
    if (!csr_row_ptr) { off_rp = off; off = round_up(off + static_cast<size_t>(d_rows + 1) * 4, 256); }
    if (!csr_col) { off_col = off; off = round_up(off + static_cast<size_t>(Nq * Nd * Lq) * 4, 256); }
    const int32_t n_chunks = dQ ? dq_chunks(Nq, Lq, Nd) : 1;
    if (n_chunks > 1) { off_part = off; off = round_up(off + static_cast<size_t>(n_chunks) * Nq * Lq * dim * 4, 256); }
    if ((need_csr || n_chunks > 1) && (workspace_bytes < off || !workspace)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    BwdArgs b{};
    b.Q = static_cast<const uint16_t*>(Q);
    b.D = static_cast<const uint16_t*>(D);
    b.is_bf16 = dtype == MAXSIM_BF16;
    b.nq = static_cast<int32_t>(Nq);
    b.lq = static_cast<int32_t>(Lq);
    b.nd = static_cast<int32_t>(Nd);
    b.ld = static_cast<int32_t>(Ld);
    b.dim = static_cast<int32_t>(dim);
    b.q_mask = q_mask;
    b.argmax = argmax;
    b.g = grad_scores;
    b.dQ = dQ;
    b.dD = dD;
    b.status = dev->status;
    b.cu_q = cu_q;
    b.cu_d = cu_d;
    b.d_rows = d_rows;
    if (cu_d) check_cu_kernel<<<grid_for(Nd + 1, 256, dev->num_sms), 256, 0, st>>>(cu_d, Nd, d_rows, dev->status);
    if (cu_q) check_cu_kernel<<<grid_for(Nq + 1, 256, dev->num_sms), 256, 0, st>>>(cu_q, Nq, -1, dev->status);
    const int vec = static_cast<int>((dim + 31) / 32);
    // dD alone, dense D: the CSR of each document slice is built in shared
    // memory next to the reduction (the same sorted sources, the same sums)
    const bool fused_dd = dD && !csr_row_ptr && !csr_col && !cu_d && !cu_q && Ld > 0 && Nd > 0 &&
                          Nq * Lq <= kDdMaxSrc;
    // dQ beside the CSR and dD work when there is any
    const bool side_dq = dQ && Nq * Lq > 0 && (fused_dd || need_csr || (dD && d_rows > 0));
    std::unique_lock<std::mutex> side_lock(g_bwd_mu, std::defer_lock);
    BwdSide* side = nullptr;
    if (side_dq) {
        side_lock.lock();
        if ((rc = bwd_side(&side)) != MAXSIM_OK) return rc;
        if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
    }
    // every return after the fork joins the side stream back first
    auto join = [&](maxsim_status r) -> maxsim_status {
        if (side && (cudaEventRecord(side->join, side->stream) != cudaSuccess ||
                     cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess))
            return MAXSIM_ERR_CUDA;
        return r;
    };
    if (fused_dd) {
        const dim3 grid(static_cast<unsigned>(Nd), static_cast<unsigned>((Ld + kDdRows - 1) / kDdRows));
        const size_t shm = dd_fused_smem(static_cast<int32_t>(Nq * Lq));
        static_assert(kDdMaxSrc * 3 + kDdWarps * kDdRows * 4 + (kDdRows + 1) * 4 + 16 <= 227 * 1024, "fused dD smem");
        maxsim_status frc = MAXSIM_OK;
        switch (vec) {
        case 1: frc = launch_dd_fused_t<1>(grid, shm, st, b); break;
        case 2: frc = launch_dd_fused_t<2>(grid, shm, st, b); break;
        case 3: frc = launch_dd_fused_t<3>(grid, shm, st, b); break;
        case 4: frc = launch_dd_fused_t<4>(grid, shm, st, b); break;
        case 5: frc = launch_dd_fused_t<5>(grid, shm, st, b); break;
        case 6: frc = launch_dd_fused_t<6>(grid, shm, st, b); break;
        case 7: frc = launch_dd_fused_t<7>(grid, shm, st, b); break;
        default: frc = launch_dd_fused_t<8>(grid, shm, st, b); break;
        }
        if (frc != MAXSIM_OK) return join(frc);
    } else if (need_csr) {
        b.doc_cnt = reinterpret_cast<int32_t*>(ws + off_cnt);
        b.doc_base = reinterpret_cast<int32_t*>(ws + off_base);
        b.row_ptr = csr_row_ptr ? csr_row_ptr : reinterpret_cast<int32_t*>(ws + off_rp);
        b.col = csr_col ? csr_col : reinterpret_cast<int32_t*>(ws + off_col);
        // packed: rows no document covers (inconsistent offsets) stay empty
        if (cu_d && cudaMemsetAsync(b.row_ptr, 0, static_cast<size_t>(d_rows + 1) * 4, st) != cudaSuccess)
            return join(MAXSIM_ERR_CUDA);
        if (Nd > 0) {
            csr_count_kernel<<<static_cast<int>(Nd), 256, 0, st>>>(b);
        }
        csr_doc_scan_kernel<<<1, 1024, 0, st>>>(b);
        if (Nd > 0 && Ld > 0) {
            int32_t nw = static_cast<int32_t>(std::min<int64_t>(8, (200 * 1024) / (Ld * 4)));
            size_t shm = static_cast<size_t>(nw) * Ld * 4;
            if (shm > 48 * 1024)
                cudaFuncSetAttribute(csr_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(shm));
            csr_build_kernel<<<static_cast<int>(Nd), 256, shm, st>>>(b, nw);
        }
        if (cudaGetLastError() != cudaSuccess) return join(MAXSIM_ERR_CUDA);
    }
    if (dD && d_rows > 0 && !fused_dd) {
        const int grid = static_cast<int>((d_rows + 7) / 8);
        switch (vec) {
        case 1: dd_kernel<1><<<grid, 256, 0, st>>>(b); break;
        case 2: dd_kernel<2><<<grid, 256, 0, st>>>(b); break;
        case 3: dd_kernel<3><<<grid, 256, 0, st>>>(b); break;
        case 4: dd_kernel<4><<<grid, 256, 0, st>>>(b); break;
        case 5: dd_kernel<5><<<grid, 256, 0, st>>>(b); break;
        case 6: dd_kernel<6><<<grid, 256, 0, st>>>(b); break;
        case 7: dd_kernel<7><<<grid, 256, 0, st>>>(b); break;
        default: dd_kernel<8><<<grid, 256, 0, st>>>(b); break;
        }
    }
    if (dQ && Nq * Lq > 0) {
        const int64_t rows = Nq * Lq;
        const dim3 grid(static_cast<unsigned>((rows + 7) / 8), static_cast<unsigned>(n_chunks));
        float* part = n_chunks > 1 ? reinterpret_cast<float*>(ws + off_part) : nullptr;
        const cudaStream_t sq = side ? side->stream : st;
        switch (vec) {
        case 1: launch_dq<1>(grid, sq, b, part); break;
        case 2: launch_dq<2>(grid, sq, b, part); break;
        case 3: launch_dq<3>(grid, sq, b, part); break;
        case 4: launch_dq<4>(grid, sq, b, part); break;
        case 5: launch_dq<5>(grid, sq, b, part); break;
        case 6: launch_dq<6>(grid, sq, b, part); break;
        case 7: launch_dq<7>(grid, sq, b, part); break;
        default: launch_dq<8>(grid, sq, b, part); break;
        }
        if (n_chunks > 1)
            dq_reduce_kernel<<<grid_for(rows * dim, 256, dev->num_sms), 256, 0, sq>>>(b, part, n_chunks);
    }
    return join(cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA);
}

}  // namespace
}  // namespace maxsim

using namespace maxsim;

extern "C" {

int maxsim_version(void) { return 200; }

const char* maxsim_status_string(maxsim_status s) {
    switch (s) {
    case MAXSIM_OK: return "ok";
    case MAXSIM_ERR_INVALID_ARG: return "invalid argument";
    case MAXSIM_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MAXSIM_ERR_CUDA: return "CUDA call failed";
    case MAXSIM_ERR_TIMEOUT: return "device-side wait timed out";
    case MAXSIM_ERR_WORKSPACE: return "workspace missing or too small";
    case MAXSIM_ERR_DEVICE_INPUT: return "an input failed a device-side check";
    }
    return "unknown status";
}

maxsim_status maxsim_debug_inject_wait_timeout(uint64_t limit_ns) {
    if (limit_ns == 0 || limit_ns > kTimeoutNs) return MAXSIM_ERR_INVALID_ARG;
    g_inject_wait_ns.store(limit_ns);
    return MAXSIM_OK;
}

maxsim_status maxsim_device_status(void* stream) {
    DeviceInfo* dev = nullptr;
    maxsim_status rc = device_info(&dev);
    if (rc != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MAXSIM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MAXSIM_ERR_CUDA;
    int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MAXSIM_ERR_CUDA;
    return static_cast<maxsim_status>(v);
}

maxsim_status maxsim_last_device_status(void* stream) { return maxsim_device_status(stream); }

size_t maxsim_workspace_size(int op, int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim) {
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0 || dim <= 0) return static_cast<size_t>(-1);
    switch (op) {
    case MAXSIM_OP_FWD:
        return plan_fwd(Nq, Lq, Nd, dim, false, false).ws_bytes;
    case MAXSIM_OP_FWD_VARLEN:
        return plan_fwd(Nq, Lq, Nd, dim, true, false).ws_bytes;
    case MAXSIM_OP_SCORE_PAIRS:  // Ld carries the number of pairs
        return pairs_ws(plan_fwd(Nq, Lq, Nd, dim, true, false, true).ws_bytes, Nq, Ld).bytes;
    case MAXSIM_OP_FWD_INT8:
        return plan_fwd(Nq, Lq, Nd, dim, false, true).ws_bytes;
    case MAXSIM_OP_BWD:
        return bwd_ws_bytes(Nq, Lq, Nd, Nd * Ld, dim, false, false);
    case MAXSIM_OP_BWD_VARLEN:  // (Nq, max_lq, Nd, total_d, dim)
        return bwd_ws_bytes(Nq, Lq, Nd, Ld, dim, false, false);
    case MAXSIM_OP_FWD_VARLEN_STREAMED: {  // (Nq, max_lq, block_docs, block_tokens, dim)
        const FwdPlan f = plan_fwd(Nq, Lq, Nd, dim, true, false);
        if (!f.ok) return static_cast<size_t>(-1);
        size_t off = 0;
        for (int i = 0; i < 2; ++i) {
            off = round_up(off + static_cast<size_t>(Ld * dim * 2), 256);
            off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);
        }
        off = round_up(off + static_cast<size_t>(Nq * Nd) * 4, 256);
        return round_up(off + f.ws_bytes, 256);
    }
    case MAXSIM_OP_FWD_STREAMED: {  // (Nq, Lq, block_docs, Ld, dim)
        const StreamedPlan p = plan_streamed(Nq, Lq, Nd, Ld, dim, 2);
        return p.ok ? p.bytes : static_cast<size_t>(-1);
    }
    case MAXSIM_OP_TWO_STAGE: {  // (Nq, Lq, Nd, Ld, dim), for any k1 <= min(Nd, 4096)
        const TwoStagePlan p = plan_two_stage(Nq, Lq, Nd, dim, std::min<int64_t>(Nd, kTopkMaxK));
        return p.ok ? p.bytes : static_cast<size_t>(-1);
    }
    case MAXSIM_OP_CHAMFER_FWD:  // (B, N, M, unused, dim)
        if (check_chamfer_shape(Nq, Lq, Nd, dim) == MAXSIM_ERR_INVALID_ARG) return static_cast<size_t>(-1);
        return dim <= kTcMaxDim ? plan_chamfer_tc(Nq, Lq, Nd).ws_bytes : plan_chamfer_fwd(Nq, Lq, Nd, dim).ws_bytes;
    case MAXSIM_OP_CHAMFER_BWD:
        if (check_chamfer_shape(Nq, Lq, Nd, dim) == MAXSIM_ERR_INVALID_ARG) return static_cast<size_t>(-1);
        return plan_chamfer_bwd(Nq, Lq, Nd).ws_bytes;
    default: return static_cast<size_t>(-1);
    }
}

maxsim_status maxsim_fwd(const void* Q, const void* D, maxsim_dtype dtype, int64_t Nq, int64_t Lq, int64_t Nd,
                         int64_t Ld, int64_t dim, const uint8_t* q_mask, const uint8_t* d_mask, float* scores,
                         int32_t* argmax, void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd == 0) return MAXSIM_OK;
    if (!scores) return MAXSIM_ERR_INVALID_ARG;
    if ((Lq > 0 && (!Q || !aligned16(Q))) || (Ld > 0 && (!D || !aligned16(D)))) return MAXSIM_ERR_INVALID_ARG;
    if (Nd * Ld > kI32Max || Nq * pad_lq(Lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    if (argmax && Nq * Nd * Lq > (int64_t(1) << 40)) return MAXSIM_ERR_UNSUPPORTED;
    const FwdPlan p = plan_fwd(Nq, Lq, Nd, dim, false, false);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;
    if (workspace_bytes < p.ws_bytes || (p.ws_bytes > 0 && !workspace)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Lq == 0) {  // no query tokens: every score is 0
        fill_kernel<<<grid_for(Nq * Nd, 256, dev->num_sms), 256, 0, st>>>(scores, Nq * Nd, nullptr, 0);
        return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    FwdCall c{};
    c.q_rows = Q;
    c.q_active = q_mask;
    if (p.repack) {
        uint16_t* qp = reinterpret_cast<uint16_t*>(ws + p.off_q);
        dim3 blk(32, 8);
        repack_q_kernel<false><<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(
            Q, nullptr, Lq, p.lq_pad, Nq, dim, q_mask, nullptr, qp, ws + p.off_real, ws + p.off_active, nullptr);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
        c.q_rows = qp;
        c.q_real = ws + p.off_real;
        c.q_active = ws + p.off_active;
    }
    c.d_rows = D;
    c.q_dt = c.d_dt = half_map(dtype);
    c.ab_format = dtype == MAXSIM_BF16 ? 1u : 0u;
    c.nan_pair = dtype == MAXSIM_BF16 ? kNaNPairBF16 : kNaNPairF16;
    c.nq = Nq;
    c.lq_out = Lq;
    c.nd = Nd;
    c.ld = Ld;
    c.total_d = Nd * Ld;
    c.dim = dim;
    c.d_mask = d_mask;
    c.scores = scores;
    c.argmax = argmax;
    return run_fwd(dev, p, c, ws, st);
}

maxsim_status maxsim_fwd_varlen(const void* Q, const int32_t* cu_seqlens_q, int64_t max_lq, const void* D,
                                const int32_t* cu_seqlens_d, int64_t total_d, maxsim_dtype dtype, int64_t Nq,
                                int64_t Nd, int64_t dim, const uint8_t* q_mask, const uint8_t* d_mask,
                                float* scores, int32_t* argmax, void* workspace, size_t workspace_bytes,
                                void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Nd < 0 || max_lq < 0 || total_d < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd == 0) return MAXSIM_OK;
    if (!scores || !cu_seqlens_d) return MAXSIM_ERR_INVALID_ARG;
    if ((max_lq > 0 && (!Q || !aligned16(Q))) || (total_d > 0 && (!D || !aligned16(D))))
        return MAXSIM_ERR_INVALID_ARG;
    if (total_d > kI32Max || Nq * pad_lq(max_lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    const FwdPlan p = plan_fwd(Nq, max_lq, Nd, dim, true, false);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;
    if (workspace_bytes < p.ws_bytes || (p.ws_bytes > 0 && !workspace)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    check_cu_kernel<<<grid_for(Nd + 1, 256, dev->num_sms), 256, 0, st>>>(cu_seqlens_d, Nd, total_d, dev->status);
    if (cu_seqlens_q)
        check_cu_kernel<<<grid_for(Nq + 1, 256, dev->num_sms), 256, 0, st>>>(cu_seqlens_q, Nq, -1, dev->status);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    if (max_lq == 0) {
        fill_kernel<<<grid_for(Nq * Nd, 256, dev->num_sms), 256, 0, st>>>(scores, Nq * Nd, nullptr, 0);
        return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* qp = reinterpret_cast<uint16_t*>(ws + p.off_q);
    dim3 blk(32, 8);
    repack_q_kernel<false><<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(
        Q, cu_seqlens_q, max_lq, p.lq_pad, Nq, dim, q_mask, nullptr, qp, ws + p.off_real, ws + p.off_active, nullptr);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    FwdCall c{};
    c.q_rows = qp;
    c.q_real = ws + p.off_real;
    c.q_active = ws + p.off_active;
    c.d_rows = D;
    c.q_dt = c.d_dt = half_map(dtype);
    c.ab_format = dtype == MAXSIM_BF16 ? 1u : 0u;
    c.nan_pair = dtype == MAXSIM_BF16 ? kNaNPairBF16 : kNaNPairF16;
    c.nq = Nq;
    c.lq_out = max_lq;
    c.nd = Nd;
    c.ld = 0;
    c.total_d = total_d;
    c.dim = dim;
    c.cu_d = cu_seqlens_d;
    c.d_mask = d_mask;
    c.scores = scores;
    c.argmax = argmax;
    return run_fwd(dev, p, c, ws, st);
}

maxsim_status maxsim_score_pairs_packed(const void* Q, const int32_t* cu_seqlens_q, int64_t max_lq, const void* D,
                                        const int32_t* cu_seqlens_d, int64_t total_d, maxsim_dtype dtype, int64_t Nq,
                                        int64_t Nd, int64_t dim, const uint8_t* q_mask, const uint8_t* d_mask,
                                        const int32_t* pairs, int64_t num_pairs, float* scores, int32_t* argmax,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Nd < 0 || max_lq < 0 || total_d < 0 || num_pairs < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (num_pairs == 0) return MAXSIM_OK;
    if (!scores || !pairs || !aligned(pairs, 4) || !cu_seqlens_d) return MAXSIM_ERR_INVALID_ARG;
    if ((max_lq > 0 && (!Q || !aligned16(Q))) || (total_d > 0 && (!D || !aligned16(D))))
        return MAXSIM_ERR_INVALID_ARG;
    if (total_d > kI32Max || Nq * pad_lq(max_lq) > kI32Max || num_pairs > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    const FwdPlan p = plan_fwd(Nq, max_lq, Nd, dim, true, false, true);
    if (!p.ok || p.n_chunks > 1) return MAXSIM_ERR_UNSUPPORTED;  // one query per unit: up to 4 M-tiles
    const PairsWs pw = pairs_ws(p.ws_bytes, Nq, num_pairs);
    if (workspace_bytes < pw.bytes || !workspace) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* qcnt = reinterpret_cast<int32_t*>(ws + pw.off_qcnt);
    int32_t* qptr = reinterpret_cast<int32_t*>(ws + pw.off_qptr);
    int32_t* uptr = reinterpret_cast<int32_t*>(ws + pw.off_uptr);
    int32_t* cursor = reinterpret_cast<int32_t*>(ws + pw.off_cursor);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws + pw.off_sorted);
    const int gp = grid_for(num_pairs, 256, dev->num_sms);
    if (Nq * Nd == 0 || max_lq == 0) {
        // no pair can be valid (reported), or every query is empty (score 0)
        if (Nq * Nd == 0) {
            pairs_count_kernel<<<gp, 256, 0, st>>>(pairs, num_pairs, Nq, Nd, nullptr, scores, argmax, max_lq,
                                                   dev->status);
        } else {
            fill_kernel<<<gp, 256, 0, st>>>(scores, num_pairs, nullptr, 0);
        }
        return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
    }
    check_cu_kernel<<<grid_for(Nd + 1, 256, dev->num_sms), 256, 0, st>>>(cu_seqlens_d, Nd, total_d, dev->status);
    if (cu_seqlens_q)
        check_cu_kernel<<<grid_for(Nq + 1, 256, dev->num_sms), 256, 0, st>>>(cu_seqlens_q, Nq, -1, dev->status);
    // group the pairs by query: count, scan (pairs and units), place
    const int32_t chunk =
        static_cast<int32_t>(std::max<int64_t>(1, (num_pairs + 4 * dev->num_sms - 1) / (4 * dev->num_sms)));
    if (cudaMemsetAsync(qcnt, 0, static_cast<size_t>(Nq) * 4, st) != cudaSuccess) return MAXSIM_ERR_CUDA;
    pairs_count_kernel<<<gp, 256, 0, st>>>(pairs, num_pairs, Nq, Nd, qcnt, scores, argmax, max_lq, dev->status);
    pairs_scan_kernel<<<1, 1024, 0, st>>>(qcnt, Nq, chunk, qptr, uptr, cursor);
    pairs_place_kernel<<<gp, 256, 0, st>>>(pairs, num_pairs, Nq, Nd, cursor, sorted);
    uint16_t* qp = reinterpret_cast<uint16_t*>(ws + p.off_q);
    dim3 blk(32, 8);
    repack_q_kernel<false><<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(
        Q, cu_seqlens_q, max_lq, p.lq_pad, Nq, dim, q_mask, nullptr, qp, ws + p.off_real, ws + p.off_active, nullptr);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    FwdCall c{};
    c.q_rows = qp;
    c.q_real = ws + p.off_real;
    c.q_active = ws + p.off_active;
    c.d_rows = D;
    c.q_dt = c.d_dt = half_map(dtype);
    c.ab_format = dtype == MAXSIM_BF16 ? 1u : 0u;
    c.nan_pair = dtype == MAXSIM_BF16 ? kNaNPairBF16 : kNaNPairF16;
    c.nq = Nq;
    c.lq_out = max_lq;
    c.nd = Nd;
    c.ld = 0;
    c.total_d = total_d;
    c.dim = dim;
    c.cu_d = cu_seqlens_d;
    c.d_mask = d_mask;
    c.scores = scores;
    c.argmax = argmax;
    c.pr_pairs = pairs;
    c.pr_sorted = sorted;
    c.pr_qptr = qptr;
    c.pr_uptr = uptr;
    c.pr_chunk = chunk;
    return run_fwd(dev, p, c, ws, st);
}

maxsim_status maxsim_bwd(const void* Q, const void* D, maxsim_dtype dtype, int64_t Nq, int64_t Lq, int64_t Nd,
                         int64_t Ld, int64_t dim, const uint8_t* q_mask, const int32_t* argmax,
                         const float* grad_scores, float* dQ, float* dD, int32_t* csr_row_ptr, int32_t* csr_col,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0) return MAXSIM_ERR_INVALID_ARG;
    return run_bwd(Q, nullptr, Lq, D, nullptr, Nd * Ld, Ld, dtype, Nq, Nd, dim, q_mask, argmax, grad_scores, dQ, dD,
                   csr_row_ptr, csr_col, workspace, workspace_bytes, stream);
}

maxsim_status maxsim_bwd_varlen(const void* Q, const int32_t* cu_seqlens_q, int64_t max_lq, const void* D,
                                const int32_t* cu_seqlens_d, int64_t total_d, int64_t max_ld, maxsim_dtype dtype,
                                int64_t Nq, int64_t Nd, int64_t dim, const uint8_t* q_mask, const int32_t* argmax,
                                const float* grad_scores, float* dQ, float* dD, int32_t* csr_row_ptr,
                                int32_t* csr_col, void* workspace, size_t workspace_bytes, void* stream) {
    if (Nq < 0 || max_lq < 0 || Nd < 0 || total_d < 0 || max_ld < 0) return MAXSIM_ERR_INVALID_ARG;
    if (!cu_seqlens_d) return MAXSIM_ERR_INVALID_ARG;
    return run_bwd(Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, total_d, max_ld, dtype, Nq, Nd, dim, q_mask, argmax,
                   grad_scores, dQ, dD, csr_row_ptr, csr_col, workspace, workspace_bytes, stream);
}

maxsim_status maxsim_fwd_int8(const int8_t* Q, const float* q_scale, const int8_t* D, const float* d_scale,
                              int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim, const uint8_t* q_mask,
                              const uint8_t* d_mask, float* scores, int32_t* argmax, int32_t* win_dot,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 32);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd == 0) return MAXSIM_OK;
    if (!scores || (win_dot && !argmax)) return MAXSIM_ERR_INVALID_ARG;
    if (Lq > 0 && (!Q || !aligned16(Q) || !q_scale || !aligned(q_scale, 4))) return MAXSIM_ERR_INVALID_ARG;
    if (Ld > 0 && (!D || !aligned16(D) || !d_scale || !aligned(d_scale, 4))) return MAXSIM_ERR_INVALID_ARG;
    if (Nd * Ld > kI32Max || Nq * pad_lq(Lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    const FwdPlan p = plan_fwd(Nq, Lq, Nd, dim, false, true);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;
    if (workspace_bytes < p.ws_bytes || (p.ws_bytes > 0 && !workspace)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Lq == 0) {
        fill_kernel<<<grid_for(Nq * Nd, 256, dev->num_sms), 256, 0, st>>>(scores, Nq * Nd, nullptr, 0);
        return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* qp = reinterpret_cast<uint16_t*>(ws + p.off_q);
    float* qs = reinterpret_cast<float*>(ws + p.off_qscale);
    dim3 blk(32, 8);
    repack_q_kernel<true><<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(
        Q, nullptr, Lq, p.lq_pad, Nq, dim, q_mask, q_scale, qp, ws + p.off_real, ws + p.off_active, qs);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    FwdCall c{};
    c.q_rows = qp;
    c.q_real = ws + p.off_real;
    c.q_active = ws + p.off_active;
    c.q_scale = qs;
    c.d_rows = D;
    c.d_scale = d_scale;
    c.q_dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    c.d_dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    c.ab_format = 0u;
    c.nan_pair = kNaNPairF16;
    c.nq = Nq;
    c.lq_out = Lq;
    c.nd = Nd;
    c.ld = Ld;
    c.total_d = Nd * Ld;
    c.dim = dim;
    c.d_mask = d_mask;
    c.scores = scores;
    c.argmax = argmax;
    rc = run_fwd(dev, p, c, ws, st);
    if (rc != MAXSIM_OK) return rc;
    if (win_dot) {
        const int64_t n = Nq * Nd * Lq;
        win_dot_kernel<<<grid_for(n, 256, dev->num_sms), 256, 0, st>>>(Q, D, argmax, Nq, Lq, Nd, Ld, dim, win_dot);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    return MAXSIM_OK;
}

maxsim_status maxsim_chamfer_fwd(const float* P, const float* Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                                 float* dist_p, int32_t* idx_p, float* dist_q, int32_t* idx_q, float* loss,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    maxsim_status rc = check_chamfer_shape(B, N, M, dim);
    if (rc != MAXSIM_OK) return rc;
    if (B == 0) return MAXSIM_OK;
    if (B > 65535) return MAXSIM_ERR_UNSUPPORTED;  // grid.y of the merge
    if (!loss || !aligned(loss, 4)) return MAXSIM_ERR_INVALID_ARG;
    if (N > 0 && (!P || !aligned(P, 4) || !dist_p || !idx_p || !aligned(dist_p, 4) || !aligned(idx_p, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    if (M > 0 && (!Q || !aligned(Q, 4) || !dist_q || !idx_q || !aligned(dist_q, 4) || !aligned(idx_q, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    if (dim <= kTcMaxDim) {
        const ChamferTcPlan tp = plan_chamfer_tc(B, N, M);
        if (workspace_bytes < tp.ws_bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
        DeviceInfo* dev = nullptr;
        if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
        return chamfer_fwd_tc(dev, tp, P, Q, B, N, M, dim, dist_p, idx_p, dist_q, idx_q, loss,
                              static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
    }
    const ChamferFwdPlan p = plan_chamfer_fwd(B, N, M, dim);
    if (workspace_bytes < p.ws_bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ChamferFwdArgs a{};
    a.X[0] = P; a.Y[0] = Q; a.X[1] = Q; a.Y[1] = P;
    a.nx[0] = N; a.ny[0] = M; a.nx[1] = M; a.ny[1] = N;
    a.B = B;
    a.dim = static_cast<int32_t>(dim);
    a.items0 = p.items0;
    a.items = p.items;
    a.counter = reinterpret_cast<unsigned long long*>(ws + p.off_counter);
    a.dist[0] = dist_p; a.idx[0] = idx_p; a.dist[1] = dist_q; a.idx[1] = idx_q;
    for (int d = 0; d < 2; ++d) {
        a.n_sb[d] = p.n_sb[d];
        a.n_span[d] = p.n_span[d];
        a.n_mblk[d] = p.n_mblk[d];
        a.part_best[d] = reinterpret_cast<float*>(ws + p.off_best[d]);
        a.part_sub[d] = reinterpret_cast<int32_t*>(ws + p.off_sub[d]);
        a.loss_part[d] = reinterpret_cast<double*>(ws + p.off_loss[d]);
    }
    a.loss = loss;
    a.status = dev->status;
    if (p.items > 0) {
        if (cudaMemsetAsync(a.counter, 0, sizeof(unsigned long long), st) != cudaSuccess) return MAXSIM_ERR_CUDA;
        rc = p.kd == 3 ? launch_chamfer_nn<3>(dev, 12, a, p.items, st)
                       : launch_chamfer_nn<kChMaxDim>(dev, 13, a, p.items, st);
        if (rc != MAXSIM_OK) return rc;
    }
    const int64_t mblk = std::max(p.n_mblk[0], p.n_mblk[1]);
    if (mblk > 0) {
        chamfer_merge_kernel<<<dim3(static_cast<unsigned>(mblk), static_cast<unsigned>(B), 2), kChMergeThreads, 0,
                               st>>>(a);
    }
    chamfer_loss_kernel<<<static_cast<unsigned>(B), kChLossThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

maxsim_status maxsim_chamfer_bwd(const float* P, const float* Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                                 const int32_t* idx_p, const int32_t* idx_q, const float* grad_loss, float* dP,
                                 float* dQ, void* workspace, size_t workspace_bytes, void* stream) {
    maxsim_status rc = check_chamfer_shape(B, N, M, dim);
    if (rc != MAXSIM_OK) return rc;
    if (B * (N + M) == 0) return MAXSIM_OK;
    if (!grad_loss || !aligned(grad_loss, 4)) return MAXSIM_ERR_INVALID_ARG;
    if (N > 0 && (!P || !aligned(P, 4) || !idx_p || !aligned(idx_p, 4) || !dP || !aligned(dP, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    if (M > 0 && (!Q || !aligned(Q, 4) || !idx_q || !aligned(idx_q, 4) || !dQ || !aligned(dQ, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    const ChamferBwdPlan p = plan_chamfer_bwd(B, N, M);
    if (workspace_bytes < p.ws_bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(ws + p.off_keys[0]), reinterpret_cast<uint32_t*>(ws + p.off_keys[1])};
    int32_t* vals[2] = {reinterpret_cast<int32_t*>(ws + p.off_vals[0]), reinterpret_cast<int32_t*>(ws + p.off_vals[1])};
    int32_t* hist = reinterpret_cast<int32_t*>(ws + p.off_hist);
    int32_t* row_ptr = reinterpret_cast<int32_t*>(ws + p.off_row);
    ch_keys_kernel<<<grid_for(p.K, 256, dev->num_sms), 256, 0, st>>>(idx_p, idx_q, B, N, M, keys[0], vals[0],
                                                                     dev->status);
    int cur = 0;
    for (int pass = 0; pass < p.passes; ++pass) {
        const int shift = pass * kRadixBits;
        radix_hist_kernel<<<static_cast<unsigned>(p.nblocks), kRadixThreads, 0, st>>>(keys[cur], p.K, shift, hist,
                                                                                     p.nblocks);
        scan_exclusive_kernel<<<1, kScanThreads, 0, st>>>(hist, p.hist_n);
        radix_scatter_kernel<<<static_cast<unsigned>(p.nblocks), kRadixThreads, 0, st>>>(
            keys[cur], vals[cur], p.K, shift, hist, p.nblocks, keys[cur ^ 1], vals[cur ^ 1]);
        cur ^= 1;
    }
    ch_row_ptr_kernel<<<grid_for(p.K + 1, 256, dev->num_sms), 256, 0, st>>>(keys[cur], p.K, p.K, row_ptr);
    ChamferBwdArgs g{};
    g.P = P; g.Q = Q; g.B = B; g.N = N; g.M = M;
    g.dim = static_cast<int32_t>(dim);
    g.idx_p = idx_p; g.idx_q = idx_q; g.g = grad_loss;
    g.dP = dP; g.dQ = dQ;
    g.row_ptr = row_ptr;
    g.col = vals[cur];
    const int grid = grid_for(p.K, 256, dev->num_sms);
    if (dim <= 3) chamfer_grad_kernel<3><<<grid, 256, 0, st>>>(g);
    else chamfer_grad_kernel<kChMaxDim><<<grid, 256, 0, st>>>(g);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

maxsim_status maxsim_topk(const float* scores, int64_t rows, int64_t n, int64_t k, int32_t* top_idx,
                          float* top_scores, void* stream) {
    if (rows < 0 || n < 0 || k < 0) return MAXSIM_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return MAXSIM_OK;
    if (k > n) return MAXSIM_ERR_INVALID_ARG;
    if (k > kTopkMaxK || n > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    if (!scores || !aligned(scores, 4) || !top_idx || !aligned(top_idx, 4) || (top_scores && !aligned(top_scores, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    maxsim_status rc = device_info(&dev);
    if (rc != MAXSIM_OK) return rc;
    return launch_topk(dev, scores, rows, n, n, k, nullptr, 0, top_idx, top_scores, k, static_cast<cudaStream_t>(stream));
}

maxsim_status maxsim_two_stage_topk(const int8_t* Q8, const float* q_scale, const int8_t* D8, const float* d_scale,
                                    const void* Q16, const void* D16, maxsim_dtype dtype, int64_t Nq, int64_t Lq,
                                    int64_t Nd, int64_t Ld, int64_t dim, int64_t k1, int64_t k, int32_t* top_idx,
                                    float* top_scores, float* stage1_scores, int32_t* candidates, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0 || k1 < 0 || k < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 32);
    if (rc != MAXSIM_OK) return rc;
    if (Nq == 0 || k == 0) return MAXSIM_OK;
    if (k1 > Nd || k > k1) return MAXSIM_ERR_INVALID_ARG;
    if (k1 > kTopkMaxK) return MAXSIM_ERR_UNSUPPORTED;
    if (!top_idx || !aligned(top_idx, 4) || (top_scores && !aligned(top_scores, 4)) ||
        (stage1_scores && !aligned(stage1_scores, 4)) || (candidates && !aligned(candidates, 4)))
        return MAXSIM_ERR_INVALID_ARG;
    if (Lq > 0 && (!Q8 || !aligned16(Q8) || !q_scale || !aligned(q_scale, 4) || !Q16 || !aligned16(Q16)))
        return MAXSIM_ERR_INVALID_ARG;
    if (Ld > 0 && (!D8 || !aligned16(D8) || !d_scale || !aligned(d_scale, 4) || !D16 || !aligned16(D16)))
        return MAXSIM_ERR_INVALID_ARG;
    if (Nd * Ld > kI32Max || Nq * pad_lq(Lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    const TwoStagePlan p = plan_two_stage(Nq, Lq, Nd, dim, k1);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;  // the rescoring stage takes queries of up to 512 rows
    if (workspace_bytes < p.bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* s8 = stage1_scores ? stage1_scores : reinterpret_cast<float*>(ws + p.off_s8);
    int32_t* cand = candidates ? candidates : reinterpret_cast<int32_t*>(ws + p.off_cand);
    int32_t* pairs = reinterpret_cast<int32_t*>(ws + p.off_pairs);
    int32_t* cu = reinterpret_cast<int32_t*>(ws + p.off_cu);
    float* s16 = reinterpret_cast<float*>(ws + p.off_s16);
    void* stage = ws + p.off_stage;
    // 1. INT8 scores of every (query, document)
    rc = maxsim_fwd_int8(Q8, q_scale, D8, d_scale, Nq, Lq, Nd, Ld, dim, nullptr, nullptr, s8, nullptr, nullptr, stage,
                         p.stage_bytes, stream);
    if (rc != MAXSIM_OK) return rc;
    // 2. the k1 best documents of each query
    if ((rc = launch_topk(dev, s8, Nq, Nd, Nd, k1, nullptr, 0, cand, nullptr, k1, st)) != MAXSIM_OK) return rc;
    // 3. rescore the candidates from the f16 / bf16 embeddings (dense documents as packed rows)
    two_stage_pairs_kernel<<<grid_for(Nq * k1, 256, dev->num_sms), 256, 0, st>>>(cand, Nq, k1, pairs);
    uniform_offsets_kernel<<<grid_for(Nd + 1, 256, dev->num_sms), 256, 0, st>>>(Nd, Ld, cu);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    rc = maxsim_score_pairs_packed(Q16, nullptr, Lq, D16, cu, Nd * Ld, dtype, Nq, Nd, dim, nullptr, nullptr, pairs,
                                   Nq * k1, s16, nullptr, stage, p.stage_bytes, stream);
    if (rc != MAXSIM_OK) return rc;
    // 4. the k best rescored candidates, as document indices
    return launch_topk(dev, s16, Nq, k1, k1, k, cand, k1, top_idx, top_scores, k, st);
}

}  // extern "C"
// ---------------------------------------------------------------- allocation-free varlen forward
//
// Scratch for callers that cannot allocate device memory: a fixed array in
// this module's device image. Every GPU that loads the library holds it until
// the process exits; all calls on a device share it, so calls that overlap on
// the GPU race on it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MAXSIM_NOALLOC_SCRATCH_BYTES];

namespace maxsim {
namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device (with that device current). The host-side symbol is only a
// stand-in and must never be handed to a kernel.
maxsim_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAXSIM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MAXSIM_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MAXSIM_OK;
}

}  // namespace
}  // namespace maxsim

extern "C" maxsim_status maxsim_fwd_varlen_noalloc(const void* Q, const int32_t* cu_seqlens_q, int64_t max_lq,
                                                   const void* D, const int32_t* cu_seqlens_d, int64_t total_d,
                                                   maxsim_dtype dtype, int64_t Nq, int64_t Nd, int64_t dim,
                                                   const uint8_t* q_mask, const uint8_t* d_mask, float* scores,
                                                   int32_t* argmax, void* stream) {
    const size_t need = maxsim_workspace_size(MAXSIM_OP_FWD_VARLEN, Nq, max_lq, Nd, total_d, dim);
    if (need == static_cast<size_t>(-1)) return MAXSIM_ERR_INVALID_ARG;
    if (need > static_cast<size_t>(MAXSIM_NOALLOC_SCRATCH_BYTES)) return MAXSIM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        const maxsim_status rc = noalloc_scratch(&scratch);
        if (rc != MAXSIM_OK) return rc;
    }
    return maxsim_fwd_varlen(Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, total_d, dtype, Nq, Nd, dim, q_mask, d_mask,
                             scores, argmax, scratch, need > 0 ? static_cast<size_t>(MAXSIM_NOALLOC_SCRATCH_BYTES) : 0,
                             stream);
}

// ---------------------------------------------------------------- out-of-core forward
//
// A corpus held in host memory is scored block by block ("Flash-MaxSim" Sec.
// 5.3: peak device memory is one streamed document block): the copy of block
// b + 1 into one of two device buffers runs on the library's copy stream
// while block b is scored on the caller's stream. Events order the two
// streams: a buffer is refilled only after the forward that read it, and a
// forward starts only after its block has arrived.

namespace maxsim {
namespace {

struct StreamRes {
    bool init = false;
    cudaStream_t copy = nullptr;
    cudaEvent_t start = nullptr, copied[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
};

std::mutex g_stream_mu;  // also serialises the enqueue of whole streamed calls
StreamRes g_stream_res[kMaxDevices];

maxsim_status stream_res(StreamRes** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAXSIM_ERR_CUDA;
    StreamRes& r = g_stream_res[dev];
    if (!r.init) {
        if (cudaStreamCreateWithFlags(&r.copy, cudaStreamNonBlocking) != cudaSuccess) return MAXSIM_ERR_CUDA;
        cudaEvent_t* evs[5] = {&r.start, &r.copied[0], &r.copied[1], &r.done[0], &r.done[1]};
        for (cudaEvent_t* e : evs)
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return MAXSIM_ERR_CUDA;
        r.init = true;
    }
    *out = &r;
    return MAXSIM_OK;
}

}  // namespace
}  // namespace maxsim

extern "C" maxsim_status maxsim_fwd_streamed(const void* Q, const void* D_host, maxsim_dtype dtype, int64_t Nq,
                                             int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim, int64_t block_docs,
                                             const uint8_t* q_mask, float* scores, void* workspace,
                                             size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0 || block_docs <= 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd == 0) return MAXSIM_OK;
    if (!scores || !aligned(scores, 4) || (Lq > 0 && (!Q || !aligned16(Q))) || (Ld > 0 && !D_host))
        return MAXSIM_ERR_INVALID_ARG;
    const int64_t blk = std::min(block_docs, Nd);
    if (blk * Ld > kI32Max || Nq * pad_lq(Lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    const StreamedPlan p = plan_streamed(Nq, Lq, blk, Ld, dim, 2);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;
    if (workspace_bytes < p.bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
    std::lock_guard<std::mutex> lock(g_stream_mu);
    StreamRes* res = nullptr;
    if ((rc = stream_res(&res)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t doc_bytes = static_cast<size_t>(Ld * dim * 2);
    const uint8_t* host = static_cast<const uint8_t*>(D_host);
    // the copy stream starts after everything already queued on the caller's stream
    if (cudaEventRecord(res->start, st) != cudaSuccess || cudaStreamWaitEvent(res->copy, res->start, 0) != cudaSuccess)
        return MAXSIM_ERR_CUDA;
    const int64_t n_blocks = (Nd + blk - 1) / blk;
    for (int64_t b = 0; b < n_blocks; ++b) {
        const int s = static_cast<int>(b & 1);
        const int64_t j0 = b * blk, nb = std::min(blk, Nd - j0);
        void* buf = ws + p.off_buf[s];
        if (b >= 2 && cudaStreamWaitEvent(res->copy, res->done[s], 0) != cudaSuccess) return MAXSIM_ERR_CUDA;
        if (nb * Ld > 0 && cudaMemcpyAsync(buf, host + static_cast<size_t>(j0) * doc_bytes,
                                           static_cast<size_t>(nb) * doc_bytes, cudaMemcpyHostToDevice,
                                           res->copy) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaEventRecord(res->copied[s], res->copy) != cudaSuccess ||
            cudaStreamWaitEvent(st, res->copied[s], 0) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        // one query: its block of scores is contiguous in the output
        float* out = Nq == 1 ? scores + j0 : reinterpret_cast<float*>(ws + p.off_scores);
        rc = maxsim_fwd(Q, buf, dtype, Nq, Lq, nb, Ld, dim, q_mask, nullptr, out, nullptr, ws + p.off_fwd,
                        p.fwd_bytes, stream);
        if (rc != MAXSIM_OK) return rc;
        if (Nq > 1 && cudaMemcpy2DAsync(scores + j0, static_cast<size_t>(Nd) * 4, out, static_cast<size_t>(nb) * 4,
                                        static_cast<size_t>(nb) * 4, static_cast<size_t>(Nq),
                                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaEventRecord(res->done[s], st) != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    return MAXSIM_OK;
}

// ---------------------------------------------------------------- out-of-core packed forward
//
// The packed corpus stays in host memory with its offsets; blocks of whole
// documents (at most block_docs documents and block_tokens rows) are copied
// into one of two device buffers on the copy stream while the previous block
// is scored by maxsim_fwd_varlen on the caller's stream. A block's offsets are
// copied as they are and rebased on the device.

namespace maxsim {
namespace {

__global__ void rebase_offsets_kernel(int32_t* __restrict__ cu, int64_t n, int32_t base) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i <= n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        cu[i] -= base;
}

struct VarlenStreamedPlan {
    size_t off_buf[2] = {0, 0}, off_cu[2] = {0, 0}, off_scores = 0, off_fwd = 0, fwd_bytes = 0, bytes = 0;
    bool ok = false;
};

VarlenStreamedPlan plan_varlen_streamed(int64_t Nq, int64_t max_lq, int64_t block_docs, int64_t block_tokens,
                                        int64_t dim) {
    VarlenStreamedPlan p;
    const FwdPlan f = plan_fwd(Nq, max_lq, block_docs, dim, true, false);
    if (!f.ok) return p;
    size_t off = 0;
    for (int i = 0; i < 2; ++i) {
        p.off_buf[i] = off;
        off = round_up(off + static_cast<size_t>(block_tokens * dim * 2), 256);
        p.off_cu[i] = off;
        off = round_up(off + static_cast<size_t>(block_docs + 1) * 4, 256);
    }
    p.off_scores = off;
    off = round_up(off + static_cast<size_t>(Nq * block_docs) * 4, 256);
    p.off_fwd = off;
    p.fwd_bytes = f.ws_bytes;
    p.bytes = round_up(off + f.ws_bytes, 256);
    p.ok = true;
    return p;
}

}  // namespace
}  // namespace maxsim

extern "C" maxsim_status maxsim_fwd_varlen_streamed(const void* Q, const int32_t* cu_seqlens_q, int64_t max_lq,
                                                    const void* D_host, const int32_t* cu_seqlens_d_host,
                                                    int64_t total_d, maxsim_dtype dtype, int64_t Nq, int64_t Nd,
                                                    int64_t dim, const uint8_t* q_mask, int64_t block_docs,
                                                    int64_t block_tokens, float* scores, void* workspace,
                                                    size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Nd < 0 || max_lq < 0 || total_d < 0 || block_docs <= 0 || block_tokens <= 0)
        return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd == 0) return MAXSIM_OK;
    if (!scores || !aligned(scores, 4) || !cu_seqlens_d_host || (max_lq > 0 && (!Q || !aligned16(Q))) ||
        (total_d > 0 && !D_host))
        return MAXSIM_ERR_INVALID_ARG;
    if (total_d > kI32Max || Nq * pad_lq(max_lq) > kI32Max || Nq * Nd > kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    // the host offsets are read here: they must describe total_d rows, every document fitting a block
    if (cu_seqlens_d_host[0] != 0 || cu_seqlens_d_host[Nd] != total_d) return MAXSIM_ERR_INVALID_ARG;
    for (int64_t j = 0; j < Nd; ++j) {
        const int64_t len = static_cast<int64_t>(cu_seqlens_d_host[j + 1]) - cu_seqlens_d_host[j];
        if (len < 0) return MAXSIM_ERR_INVALID_ARG;
        if (len > block_tokens) return MAXSIM_ERR_UNSUPPORTED;
    }
    const int64_t bdocs = std::min(block_docs, Nd);
    const VarlenStreamedPlan p = plan_varlen_streamed(Nq, max_lq, bdocs, block_tokens, dim);
    if (!p.ok) return MAXSIM_ERR_UNSUPPORTED;
    if (workspace_bytes < p.bytes || !workspace || !aligned(workspace, 256)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    std::lock_guard<std::mutex> lock(g_stream_mu);
    StreamRes* res = nullptr;
    if ((rc = stream_res(&res)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t row_bytes = static_cast<size_t>(dim * 2);
    const uint8_t* host = static_cast<const uint8_t*>(D_host);
    if (cudaEventRecord(res->start, st) != cudaSuccess || cudaStreamWaitEvent(res->copy, res->start, 0) != cudaSuccess)
        return MAXSIM_ERR_CUDA;
    int64_t j0 = 0;
    for (int64_t b = 0; j0 < Nd; ++b) {
        // the next block: whole documents within both limits
        int64_t j1 = j0;
        while (j1 < Nd && j1 - j0 < bdocs &&
               static_cast<int64_t>(cu_seqlens_d_host[j1 + 1]) - cu_seqlens_d_host[j0] <= block_tokens)
            ++j1;
        const int64_t nb = j1 - j0;
        const int32_t t0 = cu_seqlens_d_host[j0];
        const int64_t ntok = static_cast<int64_t>(cu_seqlens_d_host[j1]) - t0;
        const int s = static_cast<int>(b & 1);
        void* buf = ws + p.off_buf[s];
        int32_t* cu = reinterpret_cast<int32_t*>(ws + p.off_cu[s]);
        if (b >= 2 && cudaStreamWaitEvent(res->copy, res->done[s], 0) != cudaSuccess) return MAXSIM_ERR_CUDA;
        if (ntok > 0 && cudaMemcpyAsync(buf, host + static_cast<size_t>(t0) * row_bytes,
                                        static_cast<size_t>(ntok) * row_bytes, cudaMemcpyHostToDevice,
                                        res->copy) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaMemcpyAsync(cu, cu_seqlens_d_host + j0, static_cast<size_t>(nb + 1) * 4, cudaMemcpyHostToDevice,
                            res->copy) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaEventRecord(res->copied[s], res->copy) != cudaSuccess ||
            cudaStreamWaitEvent(st, res->copied[s], 0) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        rebase_offsets_kernel<<<grid_for(nb + 1, 256, dev->num_sms), 256, 0, st>>>(cu, nb, t0);
        float* out = Nq == 1 ? scores + j0 : reinterpret_cast<float*>(ws + p.off_scores);
        rc = maxsim_fwd_varlen(Q, cu_seqlens_q, max_lq, ntok > 0 ? buf : ws + p.off_buf[s], cu, ntok, dtype, Nq, nb,
                               dim, q_mask, nullptr, out, nullptr, ws + p.off_fwd, p.fwd_bytes, stream);
        if (rc != MAXSIM_OK) return rc;
        if (Nq > 1 && cudaMemcpy2DAsync(scores + j0, static_cast<size_t>(Nd) * 4, out, static_cast<size_t>(nb) * 4,
                                        static_cast<size_t>(nb) * 4, static_cast<size_t>(Nq),
                                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaEventRecord(res->done[s], st) != cudaSuccess) return MAXSIM_ERR_CUDA;
        j0 = j1;
    }
    return MAXSIM_OK;
}
