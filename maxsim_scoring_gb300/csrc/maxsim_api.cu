// Host side of the C ABI declared in include/maxsim.h: argument validation,
// launch planning (row blocks, document ranges, pipeline depth), TMA
// descriptor encoding, and the launches on the caller's stream.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/maxsim.h"
#include "bwd_kernels.cuh"
#include "fwd_kernel.cuh"

namespace maxsim {

// Device status word (first recorded problem wins; read and cleared by
// maxsim_device_status).
__device__ int g_device_status;

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s bound on any single device-side wait
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    int num_sms = 0;
    int smem_optin = 0;
    int* status = nullptr;
    bool attrs_set[8] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 2-D row-major [rows, cols] tensor, loaded as 64-element x box_rows boxes with
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
    int32_t k_atoms = 0, k_steps = 0, mt_max = 0;
    int64_t rows = 0;  // padded query rows
    bool repack = false;
    size_t off_q = 0, off_real = 0, off_active = 0, off_partial = 0, ws_bytes = 0;
};

inline int64_t pad_lq(int64_t lq) {
    if (lq <= 16) {
        int64_t p = 1;
        while (p < lq) p <<= 1;
        return p;
    }
    return (lq + 31) / 32 * 32;
}

// mt_max by operand width: the resident query block plus two document stages
// must fit in shared memory.
inline int32_t mt_for_atoms(int32_t k_atoms) { return k_atoms <= 2 ? 4 : (k_atoms == 3 ? 2 : 1); }

FwdPlan plan_fwd(int64_t nq, int64_t lq, int64_t nd, int64_t dim, int elem_bytes, bool varlen_q, bool int8) {
    FwdPlan p;
    p.lq_pad = pad_lq(lq);
    p.k_atoms = static_cast<int32_t>((dim + 63) / 64);
    p.k_steps = static_cast<int32_t>(dim / 16);
    p.mt_max = mt_for_atoms(p.k_atoms);
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
    p.repack = int8 || varlen_q || p.lq_pad != lq;
    size_t off = 0;
    if (p.repack) {
        p.off_q = off;
        off = round_up(off + static_cast<size_t>(p.rows) * dim * 2, 256);  // bf16/f16 operand
        p.off_real = off;
        off = round_up(off + static_cast<size_t>(p.rows), 256);
        p.off_active = off;
        off = round_up(off + static_cast<size_t>(p.rows), 256);
    }
    if (p.n_chunks > 1) {
        p.off_partial = off;
        off = round_up(off + static_cast<size_t>(p.n_chunks) * nq * nd * sizeof(float), 256);
    }
    (void)elem_bytes;
    p.ws_bytes = off;
    return p;
}

size_t fwd_smem_bytes(int32_t mt_max, int32_t k_atoms, int32_t stages) {
    return 1024 + static_cast<size_t>(mt_max) * k_atoms * kAtomBytes +
           static_cast<size_t>(stages) * k_atoms * kAtomBytes + sizeof(SmemCtl);
}

// Deepest document ring (2..8 stages) that fits; 0 if even two do not fit.
int32_t fwd_stages(int32_t mt_max, int32_t k_atoms, int smem_optin) {
    int32_t s = 8;
    while (s >= 2 && fwd_smem_bytes(mt_max, k_atoms, s) > static_cast<size_t>(smem_optin)) --s;
    return s >= 2 ? s : 0;
}

int64_t choose_doc_ranges(int64_t n_rb, int64_t total_d, int64_t nd, int num_sms) {
    if (nd == 0) return 1;
    int64_t waves = (total_d * n_rb >= static_cast<int64_t>(num_sms) * 4 * 2048) ? 4 : 1;
    int64_t n_dr = (static_cast<int64_t>(num_sms) * waves + n_rb - 1) / n_rb;
    n_dr = std::min<int64_t>(n_dr, std::max<int64_t>(1, total_d / 256));
    n_dr = std::min<int64_t>(n_dr, nd);
    return std::max<int64_t>(1, n_dr);
}

// ---------------------------------------------------------------- small kernels

__global__ void repack_q_kernel(const uint16_t* __restrict__ q, const int32_t* __restrict__ cu_q, int64_t lq_dense,
                                int64_t lq_pad, int64_t nq, int64_t dim, const uint8_t* __restrict__ q_mask,
                                uint16_t* __restrict__ qp, uint8_t* __restrict__ real, uint8_t* __restrict__ active) {
    const int64_t rows = nq * lq_pad;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.y) + threadIdx.y; r < rows;
         r += static_cast<int64_t>(gridDim.x) * blockDim.y) {
        const int64_t i = r / lq_pad, s = r - (r / lq_pad) * lq_pad;
        const int64_t start = cu_q ? cu_q[i] : i * lq_dense;
        const int64_t len = cu_q ? static_cast<int64_t>(cu_q[i + 1]) - cu_q[i] : lq_dense;
        const bool is_real = s < len;
        const int64_t src = start + s;
        for (int64_t k = threadIdx.x; k < dim; k += blockDim.x) qp[r * dim + k] = is_real ? q[src * dim + k] : 0;
        if (threadIdx.x == 0) {
            real[r] = is_real ? 1 : 0;
            active[r] = (is_real && (q_mask == nullptr || q_mask[src] != 0)) ? 1 : 0;
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

inline int grid_for(int64_t n, int per_block, int num_sms) {
    int64_t g = (n + per_block - 1) / per_block;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, static_cast<int64_t>(num_sms) * 8)));
}

template <bool kArg, bool kDMask>
maxsim_status launch_fwd_kernel(DeviceInfo* dev, int slot, const CUtensorMap& tq, const CUtensorMap& td,
                                const FwdArgs& a, size_t smem, int grid, cudaStream_t st) {
    auto kern = maxsim_fwd_kernel<kArg, kDMask>;
    if (!dev->attrs_set[slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev->smem_optin) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        dev->attrs_set[slot] = true;
    }
    kern<<<grid, kThreads, smem, st>>>(tq, td, a);
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

// Shared path of the three forward entry points once the operands are
// f16/bf16 rows in device memory: Q as padded rows [rows, dim] (possibly in the
// workspace), D as packed token rows [total_d, dim].
maxsim_status run_fwd(DeviceInfo* dev, const FwdPlan& p, const void* q_rows, const uint8_t* q_real,
                      const uint8_t* q_active, const void* d_rows, CUtensorMapDataType tdt, uint32_t ab_format,
                      int64_t nq, int64_t lq_out, int64_t nd, int64_t ld, const int32_t* cu_d, int64_t total_d,
                      int64_t dim, const uint8_t* d_mask, float* scores, int32_t* argmax, uint8_t* ws,
                      cudaStream_t st) {
    CUtensorMap tq, td;
    if (!encode_rows(&tq, q_rows, tdt, 2, static_cast<uint64_t>(dim), static_cast<uint64_t>(p.rows), 64, kBM))
        return MAXSIM_ERR_CUDA;
    // With no document tokens the D map is never read; point it at Q.
    const void* dbase = total_d > 0 ? d_rows : q_rows;
    const uint64_t drows = total_d > 0 ? static_cast<uint64_t>(total_d) : static_cast<uint64_t>(p.rows);
    if (!encode_rows(&td, dbase, tdt, 2, static_cast<uint64_t>(dim), drows, 64, kBN)) return MAXSIM_ERR_CUDA;

    FwdArgs a{};
    a.nq = static_cast<int32_t>(nq);
    a.lq_pad = static_cast<int32_t>(p.lq_pad);
    a.lq_out = static_cast<int32_t>(lq_out);
    a.q_active = q_active;
    a.q_real = q_real;
    a.rb_rows = p.rb_rows;
    a.n_chunks = p.n_chunks;
    a.n_rb = static_cast<int32_t>(p.n_rb);
    a.cu_d = cu_d;
    a.nd = static_cast<int32_t>(nd);
    a.ld = static_cast<int32_t>(ld);
    a.total_d = static_cast<int32_t>(total_d);
    a.d_mask = d_mask;
    const int64_t n_dr = choose_doc_ranges(p.n_rb, total_d, nd, dev->num_sms);
    a.n_dr = static_cast<int32_t>(n_dr);
    a.n_units = static_cast<int32_t>(n_dr * p.n_rb);
    a.scores = scores;
    a.partial = p.n_chunks > 1 ? reinterpret_cast<float*>(ws + p.off_partial) : nullptr;
    a.argmax = argmax;
    a.k_steps = p.k_steps;
    a.k_atoms = p.k_atoms;
    a.stages = fwd_stages(p.mt_max, p.k_atoms, dev->smem_optin);
    if (a.stages == 0) return MAXSIM_ERR_UNSUPPORTED;
    a.q_slots = p.mt_max;
    a.idesc = idesc_f16_f32(ab_format, kBM, kBN);
    a.status = dev->status;
    a.timeout_ns = kTimeoutNs;
    // One CTA per SM: the request below always exceeds half of an SM's shared memory.
    size_t smem = std::max<size_t>(fwd_smem_bytes(p.mt_max, p.k_atoms, a.stages),
                                   static_cast<size_t>(dev->smem_optin / 2 + 1024));
    smem = std::min<size_t>(smem, static_cast<size_t>(dev->smem_optin));
    const int grid = static_cast<int>(std::min<int64_t>(a.n_units, dev->num_sms));

    maxsim_status rc;
    const bool arg = argmax != nullptr, dm = d_mask != nullptr;
    if (arg && dm) rc = launch_fwd_kernel<true, true>(dev, 0, tq, td, a, smem, grid, st);
    else if (arg) rc = launch_fwd_kernel<true, false>(dev, 1, tq, td, a, smem, grid, st);
    else if (dm) rc = launch_fwd_kernel<false, true>(dev, 2, tq, td, a, smem, grid, st);
    else rc = launch_fwd_kernel<false, false>(dev, 3, tq, td, a, smem, grid, st);
    if (rc != MAXSIM_OK) return rc;
    if (p.n_chunks > 1) {
        const int64_t n = nq * nd;
        sum_chunks_kernel<<<grid_for(n, 256, dev->num_sms), 256, 0, st>>>(a.partial, p.n_chunks, n, scores);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    return MAXSIM_OK;
}

maxsim_status check_dim(int64_t dim, int64_t multiple) {
    if (dim <= 0) return MAXSIM_ERR_INVALID_ARG;
    if (dim % multiple != 0 || dim > 256) return MAXSIM_ERR_UNSUPPORTED;
    return MAXSIM_OK;
}

constexpr int64_t kI32Max = 2147483647;

}  // namespace
}  // namespace maxsim

using namespace maxsim;

extern "C" {

int maxsim_version(void) { return 100; }

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

size_t maxsim_workspace_size(int op, int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim) {
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0 || dim <= 0) return static_cast<size_t>(-1);
    switch (op) {
    case MAXSIM_OP_FWD:
        return plan_fwd(Nq, Lq, Nd, dim, 2, false, false).ws_bytes;
    case MAXSIM_OP_FWD_VARLEN:
        return plan_fwd(Nq, Lq, Nd, dim, 2, true, false).ws_bytes;
    case MAXSIM_OP_FWD_INT8:
        return plan_fwd(Nq, Lq, Nd, dim, 1, false, true).ws_bytes;
    case MAXSIM_OP_BWD: {
        size_t off = 0;
        off = round_up(off + static_cast<size_t>(Nd) * 4, 256);          // doc_cnt
        off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);      // doc_base
        off = round_up(off + static_cast<size_t>(Nd * Ld + 1) * 4, 256); // row_ptr
        off = round_up(off + static_cast<size_t>(Nq * Nd * Lq) * 4, 256);  // col
        return off;
    }
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
    const FwdPlan p = plan_fwd(Nq, Lq, Nd, dim, 2, false, false);
    if (workspace_bytes < p.ws_bytes || (p.ws_bytes > 0 && !workspace)) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev)) != MAXSIM_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Lq == 0) {  // no query tokens: every score is 0
        fill_kernel<<<grid_for(Nq * Nd, 256, dev->num_sms), 256, 0, st>>>(scores, Nq * Nd, nullptr, 0);
        return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const void* q_rows = Q;
    const uint8_t* q_real = nullptr;
    const uint8_t* q_active = q_mask;
    if (p.repack) {
        uint16_t* qp = reinterpret_cast<uint16_t*>(ws + p.off_q);
        uint8_t* real = ws + p.off_real;
        uint8_t* act = ws + p.off_active;
        dim3 blk(32, 8);
        repack_q_kernel<<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(
            static_cast<const uint16_t*>(Q), nullptr, Lq, p.lq_pad, Nq, dim, q_mask, qp, real, act);
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
        q_rows = qp;
        q_real = real;
        q_active = act;
    }
    const CUtensorMapDataType tdt = dtype == MAXSIM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return run_fwd(dev, p, q_rows, q_real, q_active, D, tdt, dtype == MAXSIM_BF16 ? 1u : 0u, Nq, Lq, Nd, Ld,
                   nullptr, Nd * Ld, dim, d_mask, scores, argmax, ws, st);
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
    const FwdPlan p = plan_fwd(Nq, max_lq, Nd, dim, 2, true, false);
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
    uint8_t* real = ws + p.off_real;
    uint8_t* act = ws + p.off_active;
    dim3 blk(32, 8);
    repack_q_kernel<<<grid_for(p.rows, 8, dev->num_sms), blk, 0, st>>>(static_cast<const uint16_t*>(Q), cu_seqlens_q,
                                                                       max_lq, p.lq_pad, Nq, dim, q_mask, qp, real,
                                                                       act);
    if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    const CUtensorMapDataType tdt = dtype == MAXSIM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return run_fwd(dev, p, qp, real, act, D, tdt, dtype == MAXSIM_BF16 ? 1u : 0u, Nq, max_lq, Nd, 0, cu_seqlens_d,
                   total_d, dim, d_mask, scores, argmax, ws, st);
}

maxsim_status maxsim_bwd(const void* Q, const void* D, maxsim_dtype dtype, int64_t Nq, int64_t Lq, int64_t Nd,
                         int64_t Ld, int64_t dim, const uint8_t* q_mask, const int32_t* argmax,
                         const float* grad_scores, float* dQ, float* dD, int32_t* csr_row_ptr, int32_t* csr_col,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != MAXSIM_F16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_INVALID_ARG;
    if (Nq < 0 || Lq < 0 || Nd < 0 || Ld < 0) return MAXSIM_ERR_INVALID_ARG;
    maxsim_status rc = check_dim(dim, 16);
    if (rc != MAXSIM_OK) return rc;
    if (Nq * Nd * Lq > kI32Max || Nd * Ld >= kI32Max) return MAXSIM_ERR_UNSUPPORTED;
    // destination histograms: at least one warp's worth of Ld counters must fit
    if (Ld * 4 > 200 * 1024) return MAXSIM_ERR_UNSUPPORTED;
    const bool need_csr = dD || csr_row_ptr || csr_col;
    if (need_csr || dQ) {
        if (!argmax || !grad_scores) return MAXSIM_ERR_INVALID_ARG;
        if ((Nq * Lq > 0 && !Q) || (Nd * Ld > 0 && !D)) return MAXSIM_ERR_INVALID_ARG;
    }
    size_t off = 0;
    const size_t off_cnt = off;
    off = round_up(off + static_cast<size_t>(Nd) * 4, 256);
    const size_t off_base = off;
    off = round_up(off + static_cast<size_t>(Nd + 1) * 4, 256);
    size_t off_rp = 0, off_col = 0;
    if (!csr_row_ptr) { off_rp = off; off = round_up(off + static_cast<size_t>(Nd * Ld + 1) * 4, 256); }
    if (!csr_col) { off_col = off; off = round_up(off + static_cast<size_t>(Nq * Nd * Lq) * 4, 256); }
    if (need_csr && (workspace_bytes < off || !workspace)) return MAXSIM_ERR_WORKSPACE;
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
    if (need_csr) {
        b.doc_cnt = reinterpret_cast<int32_t*>(ws + off_cnt);
        b.doc_base = reinterpret_cast<int32_t*>(ws + off_base);
        b.row_ptr = csr_row_ptr ? csr_row_ptr : reinterpret_cast<int32_t*>(ws + off_rp);
        b.col = csr_col ? csr_col : reinterpret_cast<int32_t*>(ws + off_col);
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
        if (cudaGetLastError() != cudaSuccess) return MAXSIM_ERR_CUDA;
    }
    const int vec = static_cast<int>((dim + 31) / 32);
    if (dD && Nd * Ld > 0) {
        const int64_t rows = Nd * Ld;
        const int grid = static_cast<int>((rows + 7) / 8);
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
        const int grid = static_cast<int>((rows + 7) / 8);
        switch (vec) {
        case 1: dq_kernel<1><<<grid, 256, 0, st>>>(b); break;
        case 2: dq_kernel<2><<<grid, 256, 0, st>>>(b); break;
        case 3: dq_kernel<3><<<grid, 256, 0, st>>>(b); break;
        case 4: dq_kernel<4><<<grid, 256, 0, st>>>(b); break;
        case 5: dq_kernel<5><<<grid, 256, 0, st>>>(b); break;
        case 6: dq_kernel<6><<<grid, 256, 0, st>>>(b); break;
        case 7: dq_kernel<7><<<grid, 256, 0, st>>>(b); break;
        default: dq_kernel<8><<<grid, 256, 0, st>>>(b); break;
        }
    }
    return cudaGetLastError() == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

maxsim_status maxsim_fwd_int8(const int8_t* Q, const float* q_scale, const int8_t* D, const float* d_scale,
                              int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim, const uint8_t* q_mask,
                              const uint8_t* d_mask, float* scores, int32_t* argmax, int32_t* win_dot,
                              void* workspace, size_t workspace_bytes, void* stream) {
    (void)Q; (void)q_scale; (void)D; (void)d_scale; (void)Nq; (void)Lq; (void)Nd; (void)Ld; (void)dim;
    (void)q_mask; (void)d_mask; (void)scores; (void)argmax; (void)win_dot; (void)workspace;
    (void)workspace_bytes; (void)stream;
    return MAXSIM_ERR_UNSUPPORTED;
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
