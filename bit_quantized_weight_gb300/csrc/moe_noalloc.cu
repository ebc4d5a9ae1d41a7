// moe_noalloc.cu -- the MoE entry point for callers that cannot allocate
// device memory.
//
// moe_qgemv_nvfp4 needs a caller-provided workspace. Some callers have no way
// to provide one: a plugin inside a host framework that owns all device
// memory and hands out no allocator, or a latency-critical decode loop that
// may not call cudaMalloc (which can synchronise the device and take
// milliseconds). This entry point takes no workspace: its scratch is a
// file-scope device array of fixed size, part of the library image, which every
// GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "qgemv_internal.h"

namespace qg {
namespace {

// Largest workspace the no-alloc entry point serves. At M = 8 tokens and
// top-8 this covers, e.g., H = 4096 with I = 2048.
constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB

__device__ __align__(256) unsigned char g_moe_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current. With lazy
// module loading (the CUDA default) that first lookup is also what makes the
// driver load the library's device code, and with it reserve the 4 MiB, on
// that device. The cached address is only valid while the device's primary
// context lives: after cudaDeviceReset the library must not be called again
// on that device in the same process.
void* scratch_on_current_device()
{
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_moe_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[device] = p;
    }
    return g_scratch_ptr[device];
}

}  // namespace
}  // namespace qg

extern "C" qg_status moe_qgemv_nvfp4_noalloc(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                              const float* gu_gscale, const uint8_t* dn_codes,
                                              const uint8_t* dn_scales, const float* dn_gscale, const void* x,
                                              const int32_t* topk_ids, const float* topk_w, void* y, int M, int H,
                                              int I, int E, int topk, cudaStream_t stream)
{
    // Same checks, in the same order, as moe_qgemv_nvfp4: pointers and sizes
    // first, so a call is rejected before anything touches CUDA.
    if (!gu_codes || !gu_scales || !gu_gscale || !dn_codes || !dn_scales || !dn_gscale || !x || !topk_ids ||
        !topk_w || !y)
        return QG_ERR_INVALID_ARG;
    size_t need = 0;
    const qg_status s = moe_qgemv_nvfp4_workspace_size(M, topk, H, I, E, &need);
    if (s != QG_OK) return s;
    const void* ptrs[] = {gu_codes, gu_scales, gu_gscale, dn_codes, dn_scales, dn_gscale, x, topk_ids, topk_w, y};
    for (const void* p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return QG_ERR_MISALIGNED;
    if (need > qg::kNoAllocScratchBytes) return QG_ERR_WORKSPACE;
    void* scratch = qg::scratch_on_current_device();
    if (!scratch) return QG_ERR_CUDA;
    // Every byte of the scratch that the MoE kernels read is written earlier
    // in the same call (group lists, unit lists, h rows, per-slot outputs),
    // so nothing needs clearing between calls.
    return moe_qgemv_nvfp4(gu_codes, gu_scales, gu_gscale, dn_codes, dn_scales, dn_gscale, x, topk_ids, topk_w, y,
                           scratch, qg::kNoAllocScratchBytes, M, H, I, E, topk, stream);
}
