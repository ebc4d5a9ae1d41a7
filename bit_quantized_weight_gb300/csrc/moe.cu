// moe.cu -- MoE router (softmax, top-k, renormalised weights) and the
// expert-gathered NVFP4 FFN. Router: Decapybara README, moe.cu ("Top-8 门控和
// softmax"); expert FFN shape: the 35B-A3B-class decode layer the NInfer
// article and memra list.
#include "common.cuh"

namespace qg {
namespace {

// One warp per token. Top-k of softmax(l) is the top-k of l itself (softmax is
// monotone); ties go to the lower expert id. The renormalised weights are
// w_i = exp(l_i - l_max) / sum_{j in top-k} exp(l_j - l_max), which equals
// p_i / sum_{top} p_j for p = softmax(l) because the full denominator cancels.
__global__ void route_kernel(const float* logits, int M, int E, int topk, int32_t* ids, float* w)
{
    const int m = blockIdx.x;
    const int lane = threadIdx.x;
    if (m >= M) return;
    const float* l = logits + static_cast<size_t>(m) * E;
    uint32_t taken[32];  // bit i of taken[j]: expert lane + 32 * (32 * j + i)... kept per lane
#pragma unroll
    for (int j = 0; j < 32; ++j) taken[j] = 0;
    float sel_l[8];
    int sel_id[8];
    for (int i = 0; i < topk; ++i) {
        float best = -INFINITY;
        int best_id = 0x7FFFFFFF;
        for (int e = lane, j = 0; e < E; e += 32, ++j) {
            if ((taken[j >> 5] >> (j & 31)) & 1u) continue;
            const float v = l[e];
            if (v > best || (v == best && e < best_id)) {
                best = v;
                best_id = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oid = __shfl_xor_sync(0xffffffffu, best_id, o);
            if (ov > best || (ov == best && oid < best_id)) {
                best = ov;
                best_id = oid;
            }
        }
        if ((best_id & 31) == lane) {
            const int j = best_id >> 5;
            taken[j >> 5] |= 1u << (j & 31);
        }
        sel_l[i] = best;
        sel_id[i] = best_id;
    }
    if (lane != 0) return;
    const float lmax = sel_l[0];
    float z = 0.f;
    float ex[8];
    for (int i = 0; i < topk; ++i) {
        ex[i] = expf(sel_l[i] - lmax);
        z += ex[i];
    }
    for (int i = 0; i < topk; ++i) {
        ids[m * topk + i] = sel_id[i];
        w[m * topk + i] = ex[i] / z;
    }
}

}  // namespace

qg_status launch_route(const float* logits, int M, int E, int topk, int32_t* ids, float* w, cudaStream_t stream)
{
    route_kernel<<<M, 32, 0, stream>>>(logits, M, E, topk, ids, w);
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

size_t moe_workspace_bytes(int M, int topk, int H, int I, int E)
{
    (void)E;
    const size_t pairs = static_cast<size_t>(M) * topk;
    size_t b = (pairs * I * 2 + 255) / 256 * 256;  // h, bf16 [M][topk][I]
    b += (pairs * H * 4 + 255) / 256 * 256;        // per-slot down outputs, fp32
    b += 64 * 1024;                                // expert lists and work units
    return b;
}

qg_status launch_moe(const uint8_t*, const uint8_t*, const float*, const uint8_t*, const uint8_t*, const float*,
                     const void*, const int32_t*, const float*, void*, void*, size_t, int, int, int, int, int,
                     cudaStream_t)
{
    return QG_ERR_UNSUPPORTED;
}

}  // namespace qg
