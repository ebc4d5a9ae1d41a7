// api.cu -- the extern "C" entry points of libqgemv: argument validation,
// kernel selection and launch on the caller's stream. Nothing here allocates
// device memory; the only device state is the status word below.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "qgemv_internal.h"

namespace qg {

__device__ int g_status_word = 0;

namespace {

std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_starve{0};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_sm_count[kMaxDevices] = {0};
int* g_status_ptr[kMaxDevices] = {nullptr};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

int current_device()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qg_status check_dense(const void* w0, const void* w1, const void* x, const void* y, const void* residual, int M,
                      int N, int K)
{
    if (!w0 || !w1 || !x || !y) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxTokens || N < 1 || K < 32 || (K % 32) != 0) return QG_ERR_INVALID_ARG;
    if (!aligned16(w0) || !aligned16(w1) || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)))
        return QG_ERR_MISALIGNED;
    return QG_OK;
}

}  // namespace

DebugState debug_state() { return DebugState{g_wait_ns.load(), g_starve.load()}; }

int sm_count(int device)
{
    if (device < 0) device = current_device();
    if (device < 0 || device >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_sm_count[device] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) v = 148;
        g_sm_count[device] = v;
    }
    return g_sm_count[device];
}

int* device_status_ptr()
{
    const int device = current_device();
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_ptr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[device] = static_cast<int*>(p);
    }
    return g_status_ptr[device];
}

static EncodeTiledFn tmap_encoder()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                    uint64_t inner_elems, uint64_t rows, uint32_t box_inner, uint32_t box_rows, bool swizzle128)
{
    if (!tmap_encoder()) return false;
    const cuuint64_t dims[2] = {inner_elems, rows};
    const cuuint64_t strides[1] = {inner_elems * static_cast<uint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A row-major [rows][chunks * inner] matrix viewed as (inner, rows, chunks),
// so that one box brings box_chunks consecutive chunks of box_rows rows,
// laid out chunk-major in shared memory ([chunk][row][inner]).
bool encode_tmap_chunks(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                        uint64_t inner_elems, uint64_t rows, uint64_t chunks, uint32_t box_rows, uint32_t box_chunks,
                        bool swizzle128)
{
    if (!tmap_encoder()) return false;
    const uint64_t inner_bytes = inner_elems * static_cast<uint64_t>(elem_bytes);
    const cuuint64_t dims[3] = {inner_elems, rows, chunks};
    const cuuint64_t strides[2] = {inner_bytes * chunks, inner_bytes};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(inner_elems), box_rows, box_chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace qg

using namespace qg;

namespace {

// NVFP4 with K a multiple of 256: one or two tokens on the CUDA-core kernel,
// three to eight on the warp-MMA kernel (its cost does not grow with the
// tokens); shapes neither plan fits go to the tcgen05 kernel, then the
// mma.sync one.
qg_status dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y, int f32,
                      const void* residual, int M, int N, int K, int swiglu, cudaStream_t stream)
{
    qg_status s = launch_cc_dense_nvfp4(codes, scales, g, x, y, f32, residual, M, N, K, swiglu, stream);
    if (s != QG_ERR_UNSUPPORTED) return s;
    if (M >= 3) {
        s = launch_mt_dense_nvfp4(codes, scales, g, x, y, f32, residual, M, N, K, swiglu, stream);
        if (s != QG_ERR_UNSUPPORTED) return s;
    }
    s = launch_tc_dense_nvfp4(codes, scales, g, x, y, f32, residual, M, N, K, swiglu, stream);
    if (s != QG_ERR_UNSUPPORTED) return s;
    return launch_dense_nvfp4(codes, scales, g, x, y, f32, residual, M, N, K, swiglu, stream);
}

// Q4/Q5 with 3..8 tokens: the warp-MMA kernel up to six tokens. It converts
// every token's activations at its start, which at seven and eight tokens
// costs more than its faster stage saves over the groupwise mma.sync kernel
// (raw bf16 activations brought in with each stage): measured on one box for
// the Q4/Q5 layer, 130 vs 154 us at M = 3, 146 vs 151 us at M = 6, 161 vs
// 150 us at M = 8.
qg_status q45_multi_token(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                          const void* x, void* y, int f32, const void* residual, int M, int N, int K,
                          cudaStream_t stream)
{
    if (M < 3 || M > 6) return QG_ERR_UNSUPPORTED;
    return launch_mt_dense_q45(q_lo, q_hi, scale, min, bits, x, y, f32, residual, M, N, K, stream);
}

// Validation of one qg_gemv_op record (qgemv_chain, qgemv_swiglu_q45).
qg_status check_op(const qg_gemv_op& g, int M)
{
    if (g.format != QG_FMT_NVFP4 && g.format != QG_FMT_Q4 && g.format != QG_FMT_Q5) return QG_ERR_INVALID_ARG;
    if (g.epilogue != QG_EPI_NONE && g.epilogue != QG_EPI_RESIDUAL && g.epilogue != QG_EPI_SWIGLU)
        return QG_ERR_INVALID_ARG;
    if (g.y_dtype != QG_OUT_BF16 && g.y_dtype != QG_OUT_F32) return QG_ERR_INVALID_ARG;
    if ((g.epilogue == QG_EPI_RESIDUAL) != (g.residual != nullptr)) return QG_ERR_INVALID_ARG;
    const bool sep_up = g.up_codes != nullptr;
    if (g.epilogue == QG_EPI_SWIGLU) {
        if (g.y_dtype != QG_OUT_BF16) return QG_ERR_INVALID_ARG;
        // NVFP4: gate and up rows in one matrix; groupwise int: a separate up matrix
        if (g.format == QG_FMT_NVFP4 ? (sep_up || g.N % 2) : !sep_up) return QG_ERR_INVALID_ARG;
    } else if (sep_up) {
        return QG_ERR_INVALID_ARG;
    }
    qg_status s = check_dense(g.codes, g.scales, g.x, g.y, g.residual, M, g.N, g.K);
    if (s != QG_OK) return s;
    if (g.format == QG_FMT_NVFP4) {
        if (g.q_hi || g.mins) return QG_ERR_INVALID_ARG;
    } else {
        if (!g.mins || ((g.format == QG_FMT_Q5) != (g.q_hi != nullptr))) return QG_ERR_INVALID_ARG;
        if (!aligned16(g.mins) || (g.q_hi && !aligned16(g.q_hi))) return QG_ERR_MISALIGNED;
    }
    if (sep_up) {
        if (g.up_format != QG_FMT_Q4 && g.up_format != QG_FMT_Q5) return QG_ERR_INVALID_ARG;
        if (!g.up_scales || !g.up_mins || ((g.up_format == QG_FMT_Q5) != (g.up_q_hi != nullptr)))
            return QG_ERR_INVALID_ARG;
        if (!aligned16(g.up_codes) || !aligned16(g.up_scales) || !aligned16(g.up_mins) ||
            (g.up_q_hi && !aligned16(g.up_q_hi)))
            return QG_ERR_MISALIGNED;
    } else if (g.up_q_hi || g.up_scales || g.up_mins) {
        return QG_ERR_INVALID_ARG;
    }
    if (g.norm_weight && !aligned16(g.norm_weight)) return QG_ERR_MISALIGNED;
    return QG_OK;
}

// The exact warp-per-row kernel for a record (any M and K).
qg_status run_op_simple(const qg_gemv_op& g, int M, cudaStream_t stream)
{
    const bool swiglu = g.epilogue == QG_EPI_SWIGLU;
    const bool sep_up = g.up_codes != nullptr;
    SimpleArgs a{};
    a.fmt = g.format == QG_FMT_NVFP4 ? FMT_NVFP4 : g.format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4;
    a.codes = g.codes;
    a.q_hi = g.q_hi;
    a.scales = g.scales;
    a.mins = g.mins;
    a.g = g.format == QG_FMT_NVFP4 ? g.global_scale : 1.f;
    if (sep_up) {
        a.ufmt = g.up_format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4;
        a.ucodes = g.up_codes;
        a.uq_hi = g.up_q_hi;
        a.uscales = g.up_scales;
        a.umins = g.up_mins;
        a.ug = 1.f;
    }
    a.x = static_cast<const uint16_t*>(g.x);
    a.y = g.y;
    a.out_f32 = g.y_dtype == QG_OUT_F32 && !swiglu;
    a.residual = static_cast<const uint16_t*>(g.residual);
    a.norm_w = static_cast<const uint16_t*>(g.norm_weight);
    a.norm_eps = g.norm_eps;
    a.M = M;
    a.n_out = swiglu && !sep_up ? g.N / 2 : g.N;
    a.K = g.K;
    a.swiglu = swiglu ? 1 : 0;
    return launch_simple_args(a, stream);
}

// One validated record on the kernel that serves it.
qg_status run_op(const qg_gemv_op& g, int M, cudaStream_t stream)
{
    const int f32 = g.y_dtype == QG_OUT_F32;
    const bool swiglu = g.epilogue == QG_EPI_SWIGLU;
    const bool full_chunks = g.K % kChunkK == 0;
    if (g.format == QG_FMT_NVFP4) {
        const uint8_t* sc = static_cast<const uint8_t*>(g.scales);
        if (!g.norm_weight) {
            if (!full_chunks)
                return launch_simple(FMT_NVFP4, g.codes, nullptr, sc, nullptr, g.global_scale, g.x, g.y,
                                     swiglu ? 0 : f32, g.residual, M, g.N, g.K, swiglu ? 1 : 0, stream);
            return dense_nvfp4(g.codes, sc, g.global_scale, g.x, g.y, swiglu ? 0 : f32, g.residual, M, g.N, g.K,
                               swiglu ? 1 : 0, stream);
        }
        if (full_chunks) {
            qg_status s = launch_cc_dense_nvfp4(g.codes, sc, g.global_scale, g.x, g.y, swiglu ? 0 : f32, g.residual,
                                                M, g.N, g.K, swiglu ? 1 : 0, stream, g.norm_weight, g.norm_eps);
            if (s != QG_ERR_UNSUPPORTED) return s;
            if (M >= 3) {
                s = launch_mt_dense_nvfp4(g.codes, sc, g.global_scale, g.x, g.y, swiglu ? 0 : f32, g.residual, M,
                                          g.N, g.K, swiglu ? 1 : 0, stream, g.norm_weight, g.norm_eps);
                if (s != QG_ERR_UNSUPPORTED) return s;
            }
            s = launch_tc_dense_nvfp4(g.codes, sc, g.global_scale, g.x, g.y, swiglu ? 0 : f32, g.residual, M, g.N,
                                      g.K, swiglu ? 1 : 0, stream, g.norm_weight, g.norm_eps);
            if (s != QG_ERR_UNSUPPORTED) return s;
        }
        return run_op_simple(g, M, stream);
    }
    const int bits = g.format == QG_FMT_Q5 ? 5 : 4;
    if (swiglu) {
        if (full_chunks) {
            const Q45Matrix gate{g.codes, g.q_hi, g.scales, g.mins, bits};
            const Q45Matrix up{g.up_codes, g.up_q_hi, g.up_scales, g.up_mins, g.up_format == QG_FMT_Q5 ? 5 : 4};
            qg_status s = launch_cc_swiglu_q45(gate, up, g.x, g.y, M, g.N, g.K, stream, g.norm_weight,
                                               g.norm_eps);
            if (s != QG_ERR_UNSUPPORTED) return s;
            if (M >= 3) {
                s = launch_mt_swiglu_q45(gate, up, g.x, g.y, M, g.N, g.K, stream, g.norm_weight, g.norm_eps);
                if (s != QG_ERR_UNSUPPORTED) return s;
            }
        }
        return run_op_simple(g, M, stream);
    }
    if (full_chunks) {
        qg_status s = launch_cc_dense_q45(g.codes, g.q_hi, g.scales, g.mins, bits, g.x, g.y, f32, g.residual, M,
                                          g.N, g.K, stream, g.norm_weight, g.norm_eps);
        if (s != QG_ERR_UNSUPPORTED) return s;
        if (!g.norm_weight) {
            s = q45_multi_token(g.codes, g.q_hi, g.scales, g.mins, bits, g.x, g.y, f32, g.residual, M, g.N, g.K,
                                stream);
            if (s != QG_ERR_UNSUPPORTED) return s;
            return launch_dense_q45(g.codes, g.q_hi, g.scales, g.mins, bits, g.x, g.y, f32, g.residual, M, g.N,
                                    g.K, stream);
        }
        // with the RMSNorm prologue: the warp-MMA kernel at every M >= 3 (the
        // groupwise mma.sync kernel has no prologue)
        if (M >= 3) {
            s = launch_mt_dense_q45(g.codes, g.q_hi, g.scales, g.mins, bits, g.x, g.y, f32, g.residual, M, g.N,
                                    g.K, stream, g.norm_weight, g.norm_eps);
            if (s != QG_ERR_UNSUPPORTED) return s;
        }
    }
    return run_op_simple(g, M, stream);
}

}  // namespace

extern "C" {

qg_status qgemv_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale, const void* x, void* y,
                      qg_out y_dtype, const void* residual, int M, int N, int K, cudaStream_t stream)
{
    qg_status s = check_dense(codes, scales, x, y, residual, M, N, K);
    if (s != QG_OK) return s;
    if (y_dtype != QG_OUT_BF16 && y_dtype != QG_OUT_F32) return QG_ERR_INVALID_ARG;
    const int f32 = y_dtype == QG_OUT_F32;
    if (K % kChunkK == 0)
        return dense_nvfp4(codes, scales, global_scale, x, y, f32, residual, M, N, K, 0, stream);
    return launch_simple(FMT_NVFP4, codes, nullptr, scales, nullptr, global_scale, x, y, f32, residual, M, N, K, 0,
                         stream);
}

qg_status qgemv_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                    const void* x, void* y, qg_out y_dtype, const void* residual, int M, int N, int K,
                    cudaStream_t stream)
{
    qg_status s = check_dense(q_lo, scale, x, y, residual, M, N, K);
    if (s != QG_OK) return s;
    if (!min) return QG_ERR_INVALID_ARG;
    if (bits != 4 && bits != 5) return QG_ERR_INVALID_ARG;
    if ((bits == 5) != (q_hi != nullptr)) return QG_ERR_INVALID_ARG;
    if (!aligned16(min) || (q_hi && !aligned16(q_hi))) return QG_ERR_MISALIGNED;
    if (y_dtype != QG_OUT_BF16 && y_dtype != QG_OUT_F32) return QG_ERR_INVALID_ARG;
    const int f32 = y_dtype == QG_OUT_F32;
    if (K % kChunkK == 0) {
        s = launch_cc_dense_q45(q_lo, q_hi, scale, min, bits, x, y, f32, residual, M, N, K, stream);
        if (s != QG_ERR_UNSUPPORTED) return s;
        s = q45_multi_token(q_lo, q_hi, scale, min, bits, x, y, f32, residual, M, N, K, stream);
        if (s != QG_ERR_UNSUPPORTED) return s;
        return launch_dense_q45(q_lo, q_hi, scale, min, bits, x, y, f32, residual, M, N, K, stream);
    }
    return launch_simple(bits == 5 ? FMT_Q5 : FMT_Q4, q_lo, q_hi, scale, min, 1.f, x, y, f32, residual, M, N, K, 0,
                         stream);
}

qg_status qgemv_swiglu_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale, const void* x,
                             void* y, int M, int N, int K, cudaStream_t stream)
{
    qg_status s = check_dense(codes, scales, x, y, nullptr, M, N, K);
    if (s != QG_OK) return s;
    if (N % 2 != 0) return QG_ERR_INVALID_ARG;
    if (K % kChunkK == 0)
        return dense_nvfp4(codes, scales, global_scale, x, y, 0, nullptr, M, N, K, 1, stream);
    return launch_simple(FMT_NVFP4, codes, nullptr, scales, nullptr, global_scale, x, y, 0, nullptr, M, N, K, 1,
                         stream);
}

qg_status moe_route_topk(const float* logits, int M, int E, int topk, int32_t* topk_ids, float* topk_w,
                         cudaStream_t stream)
{
    if (!logits || !topk_ids || !topk_w) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxTokens || topk < 1 || topk > 8 || E < topk || E > 1024) return QG_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return QG_ERR_MISALIGNED;
    return launch_route(logits, M, E, topk, topk_ids, topk_w, stream);
}

qg_status moe_qgemv_nvfp4_workspace_size(int M, int topk, int H, int I, int E, size_t* bytes)
{
    if (!bytes) return QG_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxTokens || topk < 1 || topk > 8 || E < topk || H < 256 || I < 256 || H % 256 || I % 256)
        return QG_ERR_INVALID_ARG;
    *bytes = moe_workspace_bytes(M, topk, H, I, E);
    return QG_OK;
}

qg_status moe_qgemv_nvfp4(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_gscale,
                          const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_gscale, const void* x,
                          const int32_t* topk_ids, const float* topk_w, void* y, void* workspace,
                          size_t workspace_bytes, int M, int H, int I, int E, int topk, cudaStream_t stream)
{
    if (!gu_codes || !gu_scales || !gu_gscale || !dn_codes || !dn_scales || !dn_gscale || !x || !topk_ids ||
        !topk_w || !y)
        return QG_ERR_INVALID_ARG;
    size_t need = 0;
    qg_status s = moe_qgemv_nvfp4_workspace_size(M, topk, H, I, E, &need);
    if (s != QG_OK) return s;
    const void* ptrs[] = {gu_codes, gu_scales, gu_gscale, dn_codes, dn_scales, dn_gscale, x, topk_ids, topk_w, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return QG_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QG_ERR_MISALIGNED;
    return launch_moe(gu_codes, gu_scales, gu_gscale, dn_codes, dn_scales, dn_gscale, x, topk_ids, topk_w, y,
                      workspace, workspace_bytes, M, H, I, E, topk, stream);
}

qg_status qgemv_chain_workspace_size(const qg_gemv_op* ops, int n_ops, int M, size_t* bytes)
{
    if (!ops || !bytes || n_ops < 1 || n_ops > 8 || M < 1 || M > kMaxTokens) return QG_ERR_INVALID_ARG;
    for (int o = 0; o < n_ops; ++o)
        if (ops[o].K < 1) return QG_ERR_INVALID_ARG;
    *bytes = chain_workspace_bytes(ops, n_ops, M);
    return QG_OK;
}

qg_status qgemv_chain(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, cudaStream_t stream)
{
    return qgemv_chain_ws(ops, n_ops, M, sync, nullptr, 0, stream);
}

qg_status qgemv_chain_ws(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream)
{
    if (!ops || n_ops < 1 || n_ops > 8 || M < 1 || M > kMaxTokens) return QG_ERR_INVALID_ARG;
    bool any_dep = false;
    for (int o = 0; o < n_ops; ++o) {
        const qg_status s = check_op(ops[o], M);
        if (s != QG_OK) return s;
        any_dep = any_dep || (o > 0 && ops[o].after_previous);
    }
    if (sync && !aligned16(sync)) return QG_ERR_MISALIGNED;
    if (any_dep && !sync) return QG_ERR_INVALID_ARG;
    qg_status s = QG_ERR_UNSUPPORTED;
    if (workspace) {
        if (workspace_bytes < chain_workspace_bytes(ops, n_ops, M)) return QG_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QG_ERR_MISALIGNED;
        if (M >= 3) s = launch_chain_ws(ops, n_ops, M, sync, workspace, stream);
    }
    if (s == QG_ERR_UNSUPPORTED) s = launch_chain(ops, n_ops, M, sync, stream);
    if (s != QG_ERR_UNSUPPORTED) return s;
    // One launch per op, in stream order (which also orders dependent ops).
    for (int o = 0; o < n_ops; ++o) {
        s = run_op(ops[o], M, stream);
        if (s != QG_OK) return s;
    }
    return QG_OK;
}

qg_status qgemv_swiglu_q45(const uint8_t* gate_lo, const uint8_t* gate_hi, const void* gate_scale,
                           const void* gate_min, int gate_bits, const uint8_t* up_lo, const uint8_t* up_hi,
                           const void* up_scale, const void* up_min, int up_bits, const void* x,
                           const void* norm_weight, float norm_eps, void* y, int M, int I, int K, cudaStream_t stream)
{
    if ((gate_bits != 4 && gate_bits != 5) || (up_bits != 4 && up_bits != 5)) return QG_ERR_INVALID_ARG;
    qg_gemv_op g{};
    g.format = gate_bits == 5 ? QG_FMT_Q5 : QG_FMT_Q4;
    g.epilogue = QG_EPI_SWIGLU;
    g.y_dtype = QG_OUT_BF16;
    g.N = I;
    g.K = K;
    g.codes = gate_lo;
    g.q_hi = gate_hi;
    g.scales = gate_scale;
    g.mins = gate_min;
    g.global_scale = 1.f;
    g.x = x;
    g.y = y;
    g.norm_weight = norm_weight;
    g.norm_eps = norm_eps;
    g.up_format = up_bits == 5 ? QG_FMT_Q5 : QG_FMT_Q4;
    g.up_codes = up_lo;
    g.up_q_hi = up_hi;
    g.up_scales = up_scale;
    g.up_mins = up_min;
    const qg_status s = check_op(g, M);
    if (s != QG_OK) return s;
    return run_op(g, M, stream);
}

qg_status qdequant_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale, float* w, int N, int K,
                         cudaStream_t stream)
{
    if (!codes || !scales || !w || N < 1 || K < 32 || K % 32) return QG_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(w)) return QG_ERR_MISALIGNED;
    return launch_dequant(FMT_NVFP4, codes, nullptr, scales, nullptr, global_scale, w, N, K, stream);
}

qg_status qdequant_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                       float* w, int N, int K, cudaStream_t stream)
{
    if (!q_lo || !scale || !min || !w || N < 1 || K < 32 || K % 32) return QG_ERR_INVALID_ARG;
    if (bits != 4 && bits != 5) return QG_ERR_INVALID_ARG;
    if ((bits == 5) != (q_hi != nullptr)) return QG_ERR_INVALID_ARG;
    if (!aligned16(q_lo) || !aligned16(scale) || !aligned16(min) || !aligned16(w) || (q_hi && !aligned16(q_hi)))
        return QG_ERR_MISALIGNED;
    return launch_dequant(bits == 5 ? FMT_Q5 : FMT_Q4, q_lo, q_hi, scale, min, 1.f, w, N, K, stream);
}

qg_status qg_read_probe(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream)
{
    if (!sink || bytes % 16 || (!buf && bytes)) return QG_ERR_INVALID_ARG;
    if (bytes == 0) return QG_OK;
    if (!aligned16(buf) || (reinterpret_cast<uintptr_t>(sink) & 3u)) return QG_ERR_MISALIGNED;
    return launch_read_probe(buf, bytes, sink, stream);
}

qg_status qg_last_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return QG_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return QG_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return QG_ERR_CUDA;
    return static_cast<qg_status>(v);
}

const char* qg_status_string(qg_status status)
{
    switch (status) {
    case QG_OK: return "QG_OK";
    case QG_ERR_INVALID_ARG: return "QG_ERR_INVALID_ARG";
    case QG_ERR_UNSUPPORTED: return "QG_ERR_UNSUPPORTED";
    case QG_ERR_MISALIGNED: return "QG_ERR_MISALIGNED";
    case QG_ERR_WORKSPACE: return "QG_ERR_WORKSPACE";
    case QG_ERR_CUDA: return "QG_ERR_CUDA";
    case QG_ERR_DEVICE_TIMEOUT: return "QG_ERR_DEVICE_TIMEOUT";
    }
    return "QG_ERR_UNKNOWN";
}

qg_status qg_debug_set_wait(uint64_t limit_ns, int starve)
{
    g_wait_ns.store(limit_ns ? limit_ns : kDefaultWaitNs);
    g_starve.store(starve ? 1 : 0);
    return QG_OK;
}

}  // extern "C"
