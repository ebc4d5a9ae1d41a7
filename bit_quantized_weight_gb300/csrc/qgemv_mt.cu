// qgemv_mt.cu -- NVFP4 and groupwise-int Q4/Q5 decode GEMV for 3..8 tokens:
// the one-token kernel's weight stream and plan, with each compute warp
// turning a 16-row block of decoded weights into mma.sync fragments for all
// the tokens at once.
//
// What is computed follows the pages' NVFP4 format (NVIDIA NVFP4 blog, "How
// NVFP4 works": E2M1 codes, one E4M3 scale per 16 values, one FP32 tensor
// scale) and the decode fusions (NInfer article, section 2: fused residual
// and SwiGLU epilogues; section 1: 1..8 lanes per decode round).
//
// Why a warp-level MMA: the CUDA-core kernel spends one multiply-add per
// weight and token, so its instruction count grows with the tokens and at
// two tokens it no longer keeps pace with HBM. Here one m16n8k16 MMA takes
// 16 rows x 16 k of exactly decoded weights against the (up to) 8 tokens, so
// the decode -- one cvt.rn.f16x2.e2m1x2 and one exact f16 multiply by the
// block scale per weight pair (e2m1 x e4m3 has at most 6 significant bits
// and lies in [2^-10, 2688]) -- is the whole per-weight cost, for any M <= 8.
//
//   * Units, phases, ring and TMA producer are the one-token kernel's
//     (qgemv_cc.cu); box rows are padded to 16 in
//     shared memory (zero rows), and warp w takes 16-row block w % NRB of
//     box w / NRB for the box's 256-k chunk of the stage.
//   * ldmatrix.x4 reads a 16-row x 64-k tile of the 128B-swizzled codes:
//     register j holds the 8 codes k = 32 * (j / 2) + 8 * (lane % 4) + 0..7
//     of row lane / 4 + 8 * (j % 2). The MMA's k slots 2c, 2c+1, 2c+8, 2c+9
//     of thread c = lane % 4 take that thread's k + 0..3 (first MMA) or
//     k + 4..7 (second); the activations are loaded in the same order, so the
//     permutation of k is the same on both sides and the products are the
//     dot product's.
//   * Activations: every token's chunk of 256 k is prescaled exactly into
//     f16 (maximum in [2^14, 2^15)), as in the one-token kernel; a chunk
//     that any token cannot carry exactly stays raw bf16 for all tokens and
//     its stages run bf16 MMAs on weights converted to bf16 (also exact).
//     Per stage the MMAs accumulate in fp32, then acc += D * 2^-prescale of
//     each token.
//   * Q4/Q5 (NInfer article, section 2: the groupwise-int recipe): a masked
//     nibble pair of a code word is an f16 pair of subnormals (q_j, q_j+4) *
//     2^-24 with no conversion (Q5 ORs the fifth bit from its plane), the
//     activations are stored paired (x_j, x_j+4) to match, and the two MMAs
//     of one 32-k half-tile are exactly one group of 32: per row and token
//     acc += 2^24 * scale * D * 2^-prescale + min * sum(x), with sum(x) per
//     (token, group) taken once per window from the values the projection
//     reads. A raw-bf16 chunk runs bf16 MMAs on the codes as bf16 integers
//     (128 + q - 128, exact).
//   * At a unit's end the warps' sums meet in shared memory and are added
//     over phases in index order; the epilogue applies g, SwiGLU or the
//     residual and rounds once. Every sum runs in a fixed order.
#include <algorithm>
#include <cstring>

#include "mt_core.cuh"

namespace qg {

namespace {

template <int EPI, bool MIXED, int BITS, int BITS_U, bool NORM>
__device__ __forceinline__ void mt_units(const MtArgs& m, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                         volatile int* abort_flag, volatile int* any_bf, int warp, int lane)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    const CcArgs& a = m.a;
    const int M = m.M;
    const int b2 = warp / m.NRB;
    const int rb = warp % m.NRB;
    const bool active = b2 < a.P * NGU;
    const int p = active ? b2 / NGU : 0;
    const int n_mine = active ? max(0, (a.C - p + a.P - 1) / a.P) : 0;
    const int g = lane >> 2, c = lane & 3;
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const uint8_t* fl = smem + a.smem_fl;
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const uint32_t ring = smem_u32(smem + a.smem_ring);
    const uint32_t box_off = static_cast<uint32_t>(b2 * a.R8 + 16 * rb) * 128u;
    const uint32_t sbox_off = a.scales_off + static_cast<uint32_t>(b2 * a.R8 + 16 * rb) * 16u;
    const uint32_t mbox_off = a.mins_off + static_cast<uint32_t>(b2 * a.R8 + 16 * rb) * 16u;
    const uint32_t hbox_off = a.hi_off + static_cast<uint32_t>(b2 * a.R8 + 16 * rb) * 32u;
    const float* gx_all = reinterpret_cast<const float*>(smem + a.smem_gx);
    const uint32_t x0 = smem_u32(smem + a.smem_x) + static_cast<uint32_t>(g) * m.x_tok;
    const int t0 = 2 * c, t1 = 2 * c + 1;

    bool aborted = false;
    int slot = 0, lap = 0, cur_win = 0;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cc = 0; cc < a.Cp; ++cc) {
            const int win = (cc * a.P) / m.W;  // the stage's chunks lie in one window
            if (win != cur_win) {
                named_barrier_sync(1, kCcThreads);
                mt_convert_any<BITS != 0, false, NORM>(m, smem, warp, lane, any_bf, win * m.W);
                named_barrier_sync(1, kCcThreads);
                cur_win = win;
            }
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && cc < n_mine) {
                const int kc = cc * a.P + p;
                const int j = kc - win * m.W;
                const uint32_t stage = ring + slot * a.stage_bytes;
                const uint32_t xc = x0 + static_cast<uint32_t>(j) * (kChunkK * 2u);
                const float pe0 = t0 < M ? pe_all[t0 * m.W + j] : 0.f;
                const float pe1 = t1 < M ? pe_all[t1 * m.W + j] : 0.f;
                if constexpr (BITS == 0) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    if (MIXED && fl[j] != 0)
                        mt_stage<true>(stage + box_off, stage + sbox_off, xc, lane, M, d);
                    else
                        mt_stage<false>(stage + box_off, stage + sbox_off, xc, lane, M, d);
                    acc[0] = fmaf(d[0], pe0, acc[0]);
                    acc[1] = fmaf(d[1], pe1, acc[1]);
                    acc[2] = fmaf(d[2], pe0, acc[2]);
                    acc[3] = fmaf(d[3], pe1, acc[3]);
                } else {
                    float aq[4] = {0.f, 0.f, 0.f, 0.f}, am[4] = {0.f, 0.f, 0.f, 0.f};
                    // tokens >= M: any row (their sums are never written)
                    const float* g0 = gx_all + ((t0 < M ? t0 : 0) * m.W + j) * 8;
                    const float* g1 = gx_all + ((t1 < M ? t1 : 0) * m.W + j) * 8;
                    const bool bf = MIXED && fl[j] != 0;
                    // a SwiGLU's odd boxes hold the up matrix (BITS_U-bit codes)
                    if (EPI == EPI_SWIGLU && (b2 & 1)) {
                        if (bf)
                            mtq_stage<BITS_U, true>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                    stage + hbox_off, xc, g0, g1, lane, M, aq, am);
                        else
                            mtq_stage<BITS_U, false>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                     stage + hbox_off, xc, g0, g1, lane, M, aq, am);
                    } else if (bf) {
                        mtq_stage<BITS, true>(stage + box_off, stage + sbox_off, stage + mbox_off, stage + hbox_off,
                                              xc, g0, g1, lane, M, aq, am);
                    } else {
                        mtq_stage<BITS, false>(stage + box_off, stage + sbox_off, stage + mbox_off, stage + hbox_off,
                                               xc, g0, g1, lane, M, aq, am);
                    }
                    // subnormal codes carry 2^-24 (not on the bf16 path)
                    const float f0 = bf ? 1.0f : 16777216.0f * pe0, f1 = bf ? 1.0f : 16777216.0f * pe1;
                    acc[0] = fmaf(aq[0], f0, acc[0]) + am[0];
                    acc[1] = fmaf(aq[1], f1, acc[1]) + am[1];
                    acc[2] = fmaf(aq[2], f0, acc[2]) + am[2];
                    acc[3] = fmaf(aq[3], f1, acc[3]) + am[3];
                }
            }
            mbar_arrive(&empty[slot]);
            if (++slot == a.n_stages) {
                slot = 0;
                ++lap;
            }
        }

        // the warps' sums by (box, row, token), then phases in index order
        if (active) {
            const int r = 16 * rb + g;
            float* rw = red + static_cast<size_t>(b2 * a.R8 + r) * kMtTokens;
            rw[t0] = acc[0];
            rw[t1] = acc[1];
            rw[8 * kMtTokens + t0] = acc[2];
            rw[8 * kMtTokens + t1] = acc[3];
        }
        named_barrier_sync(1, kCcThreads);
        if (!aborted) {
            const int r0 = u * a.R;
            for (int it = threadIdx.x; it < a.R * M; it += kCcThreads) {
                const int r = it % a.R, t = it / a.R;
                if (r0 + r >= a.n_out) continue;
                float v[NGU];
#pragma unroll
                for (int gg = 0; gg < NGU; ++gg) {
                    float s = 0.f;
                    for (int pp = 0; pp < a.P; ++pp) s += red[static_cast<size_t>((pp * NGU + gg) * a.R8 + r) * 8 + t];
                    v[gg] = s * a.g;
                }
                float val = v[0];
                if (EPI == EPI_SWIGLU) val = (val / (1.0f + expf(-val))) * v[NGU - 1];
                const size_t o = static_cast<size_t>(t) * a.n_out + r0 + r;
                if (EPI == EPI_RESID) val += bf16_bits_to_f32(a.residual[o]);
                if (a.out_f32)
                    reinterpret_cast<float*>(a.y)[o] = val;
                else
                    reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(val);
            }
        }
        named_barrier_sync(1, kCcThreads);  // red is rewritten by the next unit
    }
}

template <int EPI, int BITS, int BITS_U, bool NORM>
__global__ void __launch_bounds__(kCcAllThreads, 1)
    mt_gemv_kernel(const __grid_constant__ MtArgs m, const __grid_constant__ MtMaps maps)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    const CcArgs& a = m.a;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCcMaxStages);
    volatile int* any_bf = abort_flag + 1;

    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCcThreads);
        }
        *abort_flag = 0;
        *any_bf = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kCcTmaWarp) {
        // ------------------------------------------------------------ producer (qgemv_cc.cu's)
        if (elect_one()) {
            for (int i = 0; i < (BITS == 0 ? 2 : BITS == 4 ? 3 : 4); ++i) prefetch_tensormap(&maps.m[i]);
            if (BITS != 0 && NGU == 2)
                for (int i = 0; i < (BITS_U == 4 ? 3 : 4); ++i) prefetch_tensormap(&maps.m[4 + i]);
        }
        __syncwarp();
        int slot = 0, lap = 0, issued = 0;
        bool stop = false;
        for (int u = blockIdx.x; u < a.n_units && !stop; u += gridDim.x) {
            const int row0 = u * a.R;
            for (int c = 0; c < a.Cp; ++c) {
                if (lap > 0 && !cc_wait_warp(&empty[slot], (lap - 1) & 1, a, abort_flag)) {
                    stop = true;
                    break;
                }
                if (issued == kCcLeadStages) asm volatile("griddepcontrol.wait;" ::: "memory");
                if (*abort_flag || a.starve) {
                    stop = true;
                    break;
                }
                int live = 0;
                for (int pp = 0; pp < a.P; ++pp) live += (c * a.P + pp < a.C) ? 1 : 0;
                uint8_t* sb = smem + a.smem_ring + slot * a.stage_bytes;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(live) * a.box_tx);  // bytes per phase
                    for (int pp = 0; pp < a.P; ++pp) {
                        const int kc = c * a.P + pp;
                        if (kc >= a.C) continue;
#pragma unroll
                        for (int gg = 0; gg < NGU; ++gg) {
                            const int b2 = pp * NGU + gg;
                            const int row = row0 + gg * a.up_row_offset;
                            // a groupwise-int SwiGLU's up box comes from the up matrix's maps
                            const CUtensorMap* mp = &maps.m[(BITS != 0 && gg == 1) ? 4 : 0];
                            tma_load_2d(sb + b2 * a.R8 * 128, mp, kc * (kChunkK / 2), row, &full[slot]);
                            if constexpr (BITS == 0) {
                                tma_load_2d(sb + a.scales_off + b2 * a.R8 * 16, mp + 1, kc * (kChunkK / 16), row,
                                            &full[slot]);
                            } else {
                                tma_load_2d(sb + a.scales_off + b2 * a.R8 * 16, mp + 1, kc * (kChunkK / 32), row,
                                            &full[slot]);
                                tma_load_2d(sb + a.mins_off + b2 * a.R8 * 16, mp + 2, kc * (kChunkK / 32), row,
                                            &full[slot]);
                                if ((gg ? BITS_U : BITS) == 5)
                                    tma_load_2d(sb + a.hi_off + b2 * a.R8 * 32, mp + 3, kc * (kChunkK / 8), row,
                                                &full[slot]);
                            }
                        }
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == a.n_stages) {
                    slot = 0;
                    ++lap;
                }
            }
        }
        if (lane == 0)
            for (int g = max(0, issued - a.n_stages); g < issued; ++g)
                mbar_wait_bounded(&full[g % a.n_stages], (g / a.n_stages) & 1, a.wait_ns, a.status);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- compute warps
    {
        const uint32_t roff[4] = {0u, a.scales_off, a.mins_off, a.hi_off}, rbytes[4] = {128u, 16u, 16u, 32u};
        cc_zero_padding(a, smem, a.P * NGU, roff, rbytes, BITS == 0 ? 2 : BITS == 4 ? 3 : 4);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (NORM) mt_norm_factors<false>(m, smem, warp, lane);
    mt_convert_any<BITS != 0, false, NORM>(m, smem, warp, lane, any_bf, 0);
    named_barrier_sync(1, kCcThreads);
    // with several windows a later one may hold raw-bf16 chunks: the mixed loop
    if (*any_bf || m.W < a.C)
        mt_units<EPI, true, BITS, BITS_U, NORM>(m, smem, full, empty, abort_flag, any_bf, warp, lane);
    else
        mt_units<EPI, false, BITS, BITS_U, NORM>(m, smem, full, empty, abort_flag, any_bf, warp, lane);
}

constexpr uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

template <int EPI, int BITS, int BITS_U = BITS>
qg_status mt_launch(MtArgs m, const MtMaps& maps, int grid, cudaStream_t stream)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    CcArgs& a = m.a;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;

    const uint32_t nbox = static_cast<uint32_t>(a.P * NGU);
    a.scales_off = nbox * a.R8 * 128u;
    if constexpr (BITS == 0) {
        a.stage_bytes = align_up(a.scales_off + nbox * a.R8 * 16u, 1024);
        a.box_tx = static_cast<uint32_t>(NGU) * static_cast<uint32_t>(a.R) * (128u + 16u);  // per phase
    } else {
        constexpr bool any5 = BITS == 5 || (NGU == 2 && BITS_U == 5);
        a.mins_off = a.scales_off + nbox * a.R8 * 16u;
        a.hi_off = a.mins_off + nbox * a.R8 * 16u;
        a.stage_bytes = align_up(a.hi_off + (any5 ? nbox * a.R8 * 32u : 0u), 1024);
        // bytes per phase: its gate (or only) box, and a SwiGLU's up box (Q5 gate, Q4 up may differ)
        a.box_tx = static_cast<uint32_t>(a.R) * (128u + 16u + 16u + (BITS == 5 ? 32u : 0u));
        if (NGU == 2) a.box_tx += static_cast<uint32_t>(a.R) * (128u + 16u + 16u + (BITS_U == 5 ? 32u : 0u));
    }
    const uint32_t red_bytes = align_up(nbox * a.R8 * 4u * kMtTokens, 128);
    const uint32_t bar_bytes = 2 * kCcMaxStages * 8 + 16;
    // the activation window: all of K if it fits beside a ring of at least
    // four stages, else the largest multiple of P chunks that leaves three
    auto win_bytes = [&](int W) {
        const uint32_t xt = static_cast<uint32_t>(W) * kChunkK * 2u + kMtXPad;
        return align_up(static_cast<uint32_t>(m.M) * xt, 128) + align_up(static_cast<uint32_t>(m.M * W) * 4u, 16) +
               align_up(static_cast<uint32_t>(W), 16) +
               (BITS != 0 ? align_up(static_cast<uint32_t>(m.M * W) * 32u, 16) : 0u);
    };
    const uint32_t other = red_bytes + bar_bytes +
                           (a.norm_w ? align_up(static_cast<uint32_t>(m.M * (a.C + 1)) * 4u, 16) : 0u);
    int W = a.C;
    if (win_bytes(W) + other + 4 * a.stage_bytes > kCcSmemMax) {
        W = (a.C / a.P) * a.P;
        while (W > a.P && win_bytes(W) + other + 3 * a.stage_bytes > kCcSmemMax) W -= a.P;
    }
    if (win_bytes(W) + other + 3 * a.stage_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    m.W = W;
    m.x_tok = static_cast<uint32_t>(W) * kChunkK * 2u + kMtXPad;
    const uint32_t x_bytes = align_up(static_cast<uint32_t>(m.M) * m.x_tok, 128);
    const uint32_t pe_bytes = align_up(static_cast<uint32_t>(m.M * W) * 4u, 16);
    const uint32_t fl_bytes = align_up(static_cast<uint32_t>(W), 16);
    const uint32_t gx_bytes = BITS != 0 ? align_up(static_cast<uint32_t>(m.M * W) * 32u, 16) : 0u;
    const uint32_t ss_bytes = a.norm_w ? align_up(static_cast<uint32_t>(m.M * (a.C + 1)) * 4u, 16) : 0u;
    const uint32_t fixed = x_bytes + pe_bytes + fl_bytes + gx_bytes + ss_bytes + red_bytes + bar_bytes;
    a.n_stages = std::min<int>(kCcMaxStages, static_cast<int>((kCcSmemMax - fixed) / a.stage_bytes));
    uint32_t so = 0;
    a.smem_ring = so;
    so += a.n_stages * a.stage_bytes;
    a.smem_x = so;
    so += x_bytes;
    a.smem_pe = so;
    so += pe_bytes;
    a.smem_fl = so;
    so += fl_bytes;
    a.smem_gx = so;
    so += gx_bytes;
    a.smem_ss = so;
    so += ss_bytes;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;

    auto kern = a.norm_w ? mt_gemv_kernel<EPI, BITS, BITS_U, true> : mt_gemv_kernel<EPI, BITS, BITS_U, false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[a.norm_w ? 1 : 0][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[a.norm_w ? 1 : 0][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCcAllThreads);
    cfg.dynamicSmemBytes = so;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, m, maps) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace

namespace {

// The plan shared by both formats: the one-token rule for R (equal bytes per
// SM), then 16-row blocks, at most 16 warps' worth of (phase, gate/up, block)
// per stage.
MtArgs mt_plan(const void* x, void* y, int out_f32, const void* residual, int M, int n_out, int ngu, int K,
               int sms)
{
    int R = 1;
    for (int U = 1;; ++U) {
        R = (n_out + sms * U - 1) / (sms * U);
        if (ngu * ((R + 15) / 16) <= kCcWarps) break;
    }
    R = std::max(R, 1);
    MtArgs m{};
    CcArgs& a = m.a;
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.residual = static_cast<const uint16_t*>(residual);
    a.K = K;
    a.C = K / kChunkK;
    a.n_out = n_out;
    a.R = R;
    a.R8 = (R + 15) / 16 * 16;
    m.NRB = a.R8 / 16;
    a.P = std::max(1, std::min(kCcWarps / (ngu * m.NRB), a.C));
    a.Cp = (a.C + a.P - 1) / a.P;
    a.up_row_offset = ngu == 2 ? n_out : 0;
    a.out_f32 = ngu == 2 ? 0 : out_f32;
    a.g = 1.0f;
    a.n_units = (n_out + R - 1) / R;
    m.M = M;
    return m;
}

}  // namespace

// 1..8 tokens, K a multiple of 256; QG_ERR_UNSUPPORTED otherwise or when the
// plan does not fit shared memory.
qg_status launch_mt_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > kMtTokens || K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    MtArgs m = mt_plan(x, y, out_f32, residual, M, swiglu ? N / 2 : N, swiglu ? 2 : 1, K, sms);
    m.a.g = g;
    m.a.norm_w = static_cast<const uint16_t*>(norm_w);
    m.a.norm_eps = norm_eps;
    const int grid = std::min(sms, m.a.n_units);
    MtMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!encode_tmap_2d(&maps.m[0], codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, m.a.R, true) ||
        !encode_tmap_2d(&maps.m[1], scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, N, 16, m.a.R, false))
        return QG_ERR_CUDA;
    if (swiglu) return mt_launch<EPI_SWIGLU, 0>(m, maps, grid, stream);
    if (residual) return mt_launch<EPI_RESID, 0>(m, maps, grid, stream);
    return mt_launch<EPI_NONE, 0>(m, maps, grid, stream);
}

// Q4/Q5 with 1..8 tokens (plain or residual epilogue), K a multiple of 256.
qg_status launch_mt_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                              const void* x, void* y, int out_f32, const void* residual, int M, int N, int K,
                              cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > kMtTokens || K % kChunkK != 0 || (bits != 4 && bits != 5)) return QG_ERR_UNSUPPORTED;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    MtArgs m = mt_plan(x, y, out_f32, residual, M, N, 1, K, sms);
    m.a.norm_w = static_cast<const uint16_t*>(norm_w);
    m.a.norm_eps = norm_eps;
    const int grid = std::min(sms, m.a.n_units);
    const int R = m.a.R;
    MtMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!encode_tmap_2d(&maps.m[0], q_lo, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, R, true) ||
        !encode_tmap_2d(&maps.m[1], scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false) ||
        !encode_tmap_2d(&maps.m[2], min, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false))
        return QG_ERR_CUDA;
    if (bits == 5 &&
        !encode_tmap_2d(&maps.m[3], q_hi, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, N, 32, R, false))
        return QG_ERR_CUDA;
    if (bits == 5) return residual ? mt_launch<EPI_RESID, 5>(m, maps, grid, stream)
                                   : mt_launch<EPI_NONE, 5>(m, maps, grid, stream);
    return residual ? mt_launch<EPI_RESID, 4>(m, maps, grid, stream) : mt_launch<EPI_NONE, 4>(m, maps, grid, stream);
}

// Q4/Q5 SwiGLU (separate gate and up matrices, each Q4 or Q5) with 1..8
// tokens, K a multiple of 256, optional RMSNorm prologue.
qg_status launch_mt_swiglu_q45(const Q45Matrix& gate, const Q45Matrix& up, const void* x, void* y, int M, int I, int K,
                               cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > kMtTokens || K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
    if ((gate.bits != 4 && gate.bits != 5) || (up.bits != 4 && up.bits != 5)) return QG_ERR_UNSUPPORTED;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    MtArgs m = mt_plan(x, y, 0, nullptr, M, I, 2, K, sms);
    m.a.up_row_offset = 0;  // the up rows are the same rows of the up matrix
    m.a.norm_w = static_cast<const uint16_t*>(norm_w);
    m.a.norm_eps = norm_eps;
    const int grid = std::min(sms, m.a.n_units);
    const int R = m.a.R;
    MtMaps maps;
    memset(&maps, 0, sizeof(maps));
    const Q45Matrix* mats[2] = {&gate, &up};
    for (int gg = 0; gg < 2; ++gg) {
        const Q45Matrix& q = *mats[gg];
        CUtensorMap* mm = &maps.m[4 * gg];
        if (!encode_tmap_2d(&mm[0], q.q_lo, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, I, 128, R, true) ||
            !encode_tmap_2d(&mm[1], q.scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, I, 8, R, false) ||
            !encode_tmap_2d(&mm[2], q.min, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, I, 8, R, false))
            return QG_ERR_CUDA;
        if (q.bits == 5 &&
            !encode_tmap_2d(&mm[3], q.q_hi, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, I, 32, R, false))
            return QG_ERR_CUDA;
    }
    if (gate.bits == 5 && up.bits == 4) return mt_launch<EPI_SWIGLU, 5, 4>(m, maps, grid, stream);
    if (gate.bits == 5) return mt_launch<EPI_SWIGLU, 5, 5>(m, maps, grid, stream);
    if (up.bits == 5) return mt_launch<EPI_SWIGLU, 4, 5>(m, maps, grid, stream);
    return mt_launch<EPI_SWIGLU, 4, 4>(m, maps, grid, stream);
}

}  // namespace qg
