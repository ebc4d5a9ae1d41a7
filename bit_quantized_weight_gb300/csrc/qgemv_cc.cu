// qgemv_cc.cu -- NVFP4 decode GEMV for one token (M = 1) on the CUDA cores,
// with fused residual-add and SwiGLU epilogues.
//
// What is computed follows the pages' NVFP4 format (NVIDIA NVFP4 blog, "How
// NVFP4 works": E2M1 codes, one E4M3 scale per 16 values, one FP32 tensor
// scale) and decode fusions (NInfer article, section 2). For one token the
// dot products are a plain streaming reduction; the tensor cores would need
// the weights padded into a GEMM, so here every weight is consumed by one
// CUDA-core multiply-add instead:
//
//   * codes become f16 pairs with cvt.rn.f16x2.e2m1x2 (exact);
//   * the activations sit in shared memory as f16 after an exact
//     power-of-two prescale per 256-k chunk (the chunk maximum lands in
//     [2^14, 2^15)); a chunk whose smallest nonzero value f16 cannot carry
//     under that scale stays raw bf16 and takes the bf16 path below;
//   * fma.rn.f32.f16 multiplies an f16 weight by an f16 activation into an
//     fp32 accumulator: the product (at most 13 significant bits) is exact,
//     one rounding per add. The 16 products of a block are summed, then
//     scaled by the block's E4M3 scale times 2^-prescale (an exact fp32
//     product) and added to the row's accumulator.
//
// Work split. As in the tensor-core kernel, a CTA owns units of R output
// rows (gate and up rows of a SwiGLU pair both) and streams all of K for
// them; the 256-k chunks of K are dealt to P phases (phase p takes chunks p,
// p + P, ...) so that P * (gate/up) * R rows -- up to 256 -- fill the CTA's
// 16 compute warps, and the P boxes of one stage are adjacent in memory. One
// warp streams the stages (codes 128B-swizzled, scales) of every (phase,
// gate/up) box into a shared-memory ring with 2-D TMA loads. A compute
// thread takes 4 consecutive rows of a box and a 32-k (or 16-k) segment of
// the stage: it loads its activation segment once and reuses it for the 4
// rows; a warp's code loads are conflict-free under the swizzle. Each thread keeps its rows' partial sums across the
// stages of a unit; at the unit's end they are reduced over segments and
// phases in a fixed order, and the epilogue applies g, SwiGLU or the
// residual and rounds once.
#include <algorithm>
#include <cstring>

#include "cc_core.cuh"

namespace qg {

namespace {

// The compute warps' unit loop. MIXED: some chunk of x stayed raw bf16, so
// each stage picks the f16 or the bf16 stage code; otherwise the loop holds
// the f16 stage code alone. MT tokens (1 or 2) share every decoded code;
// token t's outputs and residuals start t * n_out into y and residual.
template <int EPI, int NSEG, bool MIXED, int MT = 1>
__device__ __forceinline__ void cc_units(const CcArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                         volatile int* abort_flag)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    constexpr int KS = kChunkK / NSEG;
    // this thread's rows and segment: item = (box, row group, segment); the
    // row groups cover rows 0 .. R rounded up to 4
    const int rg_per_box = (a.R + kCcRows - 1) / kCcRows;
    const int item = threadIdx.x;
    const int seg = item % NSEG;
    const int bg = item / NSEG;
    const int b2 = bg / rg_per_box;
    const int row0 = (bg % rg_per_box) * kCcRows;
    const bool active = b2 < a.P * NGU;
    const int p = active ? b2 / NGU : 0;
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(smem + a.smem_x);
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const uint8_t* fl = smem + a.smem_fl;
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const uint32_t ring = smem_u32(smem + a.smem_ring);
    // phase p takes chunks p, p + P, p + 2P, ... (the P boxes of a stage are
    // adjacent in k): n_mine of them in every unit
    const int n_mine = active ? max(0, (a.C - p + a.P - 1) / a.P) : 0;
    const uint32_t x0 = smem_u32(xs + p * (kChunkK / 2) + seg * 4);
    const uint32_t x_step = static_cast<uint32_t>(a.P) * (kChunkK * 2u);
    const uint32_t x_tok = static_cast<uint32_t>(a.C) * (kChunkK * 2u);  // bytes per token's activations

    // residual of the first unit's rows, read now rather than in the epilogue
    float res_first[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        res_first[t] = 0.f;
        if (EPI == EPI_RESID && threadIdx.x < a.R && blockIdx.x * a.R + static_cast<int>(threadIdx.x) < a.n_out)
            res_first[t] = bf16_bits_to_f32(a.residual[t * a.n_out + blockIdx.x * a.R + threadIdx.x]);
    }

    bool aborted = false;
    int slot = 0, lap = 0;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        float acc[kCcRows * MT];
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i) acc[i] = 0.f;
        for (int c = 0; c < a.Cp; ++c) {
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && c < n_mine) {
                const uint32_t stage = ring + slot * a.stage_bytes;
                const uint32_t xc = x0 + static_cast<uint32_t>(c) * x_step;
                const int kc = c * a.P + p;
                if constexpr (MT == 1) {
                    uint32_t xw[KS / 2];
#pragma unroll
                    for (int i = 0; i < KS / 8; ++i) {
                        const uint4 v = lds128(xc + i * NSEG * 16);
                        xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
                    }
                    if (!MIXED || fl[kc] == 0)
                        cc_stage<NSEG, false>(cc_geom(a), stage, b2, row0, seg, xw, pe_all[kc], acc);
                    else
                        cc_stage<NSEG, true>(cc_geom(a), stage, b2, row0, seg, xw, pe_all[kc], acc);
                } else {
                    float pe[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) pe[t] = pe_all[t * a.C + kc];
                    if (!MIXED || fl[kc] == 0)
                        cc_stage_mt<NSEG, false, MT>(cc_geom(a), stage, b2, row0, seg, xc, x_tok, pe, acc);
                    else
                        cc_stage_mt<NSEG, true, MT>(cc_geom(a), stage, b2, row0, seg, xc, x_tok, pe, acc);
                }
            }
            // every compute thread arrives: its own reads of the slot are done
            mbar_arrive(&empty[slot]);
            if (++slot == a.n_stages) {
                slot = 0;
                ++lap;
            }
        }

        // ---------------- fixed-order reduction over segments (a butterfly
        // across the segment lanes of the warp) and phases, epilogue
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i)
#pragma unroll
            for (int off = NSEG / 2; off >= 1; off >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
        if (active && seg == 0) {
#pragma unroll
            for (int i = 0; i < kCcRows; ++i)
#pragma unroll
                for (int t = 0; t < MT; ++t) red[(b2 * a.R8 + row0 + i) * MT + t] = acc[i * MT + t];
        }
        named_barrier_sync(1, kCcThreads);
        if (!aborted) {
            const int r0 = u * a.R;
            for (int r = threadIdx.x; r < a.R; r += kCcThreads) {
                if (r0 + r >= a.n_out) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    float v[NGU];
#pragma unroll
                    for (int gg = 0; gg < NGU; ++gg) {
                        float s = 0.f;
                        for (int pp = 0; pp < a.P; ++pp) s += red[((pp * NGU + gg) * a.R8 + r) * MT + t];
                        v[gg] = s * a.g;
                    }
                    float val = v[0];
                    if (EPI == EPI_SWIGLU) val = (val / (1.0f + expf(-val))) * v[NGU - 1];
                    const int o = t * a.n_out + r0 + r;
                    if (EPI == EPI_RESID)
                        val += u == static_cast<int>(blockIdx.x) && r == static_cast<int>(threadIdx.x)
                                   ? res_first[t]
                                   : bf16_bits_to_f32(a.residual[o]);
                    if (a.out_f32)
                        reinterpret_cast<float*>(a.y)[o] = val;
                    else
                        reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(val);
                }
            }
        }
        named_barrier_sync(1, kCcThreads);  // red is rewritten by the next unit
    }
}

template <int EPI, int NSEG, int MT>
__global__ void __launch_bounds__(kCcAllThreads, 1)
    cc_gemv_kernel(const __grid_constant__ CcArgs a, const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCcMaxStages);
    volatile int* any_bf = abort_flag + 1;  // some chunk of x kept raw bf16

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
        // ------------------------------------------------------------ producer
        if (elect_one()) {
            prefetch_tensormap(&tm_codes);
            prefetch_tensormap(&tm_scales);
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
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(live * NGU) * a.box_tx);
                    for (int pp = 0; pp < a.P; ++pp) {
                        const int kc = c * a.P + pp;
                        if (kc >= a.C) continue;
#pragma unroll
                        for (int gg = 0; gg < NGU; ++gg) {
                            const int b2 = pp * NGU + gg;
                            const int row = row0 + gg * a.up_row_offset;
                            tma_load_2d(sb + b2 * a.R8 * 128, &tm_codes, kc * (kChunkK / 2), row, &full[slot]);
                            tma_load_2d(sb + a.scales_off + b2 * a.R8 * 16, &tm_scales, kc * (kChunkK / 16), row,
                                        &full[slot]);
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
        const uint32_t roff[4] = {0u, a.scales_off, 0u, 0u}, rbytes[4] = {128u, 16u, 0u, 0u};
        cc_zero_padding(a, smem, a.P * NGU, roff, rbytes, 2);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (MT == 1)
        cc_convert<NSEG>(a, smem, warp, lane, any_bf);
    else
        cc_convert_q45<NSEG, XSRC_NC, kCcWarps, MT, false>(a, smem, warp, lane, any_bf);
    named_barrier_sync(1, kCcThreads);
    if (*any_bf)
        cc_units<EPI, NSEG, true, MT>(a, smem, full, empty, abort_flag);
    else
        cc_units<EPI, NSEG, false, MT>(a, smem, full, empty, abort_flag);
}

// The compute warps' unit loop of the groupwise-int kernel (MIXED as in
// cc_units).
// SwiGLU (a separate up matrix of BITS_U-bit codes): each phase holds a gate
// box (BITS) and an up box (BITS_U). MT tokens (1 or 2) share every decoded
// code: their activations, factors and sums are kept per token, their
// outputs and residuals are rows of n_out values.
template <int BITS, int EPI, int NSEG, bool MIXED, int BITS_U = BITS, int MT = 1>
__device__ __forceinline__ void cc_q45_units(const CcArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             volatile int* abort_flag)
{
    constexpr int KS = kChunkK / NSEG;
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    // item = (box, row group, segment); the row groups cover rows 0 .. R
    // rounded up to 4
    const int rg_per_box = (a.R + kCcRows - 1) / kCcRows;
    const int item = threadIdx.x;
    const int seg = item % NSEG;
    const int bg = item / NSEG;
    const int b2 = bg / rg_per_box;
    const int row0 = (bg % rg_per_box) * kCcRows;
    const bool active = b2 < a.P * NGU;
    const int p = active ? b2 / NGU : 0;
    const bool up_box = NGU == 2 && (b2 & 1);
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(smem + a.smem_x);
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const float* gx = reinterpret_cast<const float*>(smem + a.smem_gx);
    const uint8_t* fl = smem + a.smem_fl;
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const uint32_t ring = smem_u32(smem + a.smem_ring);
    // phase p takes chunks p, p + P, p + 2P, ... (the P boxes of a stage are
    // adjacent in k): n_mine of them in every unit
    const int n_mine = active ? max(0, (a.C - p + a.P - 1) / a.P) : 0;
    const uint32_t x0 = smem_u32(xs + p * (kChunkK / 2) + seg * 4);
    const uint32_t x_step = static_cast<uint32_t>(a.P) * (kChunkK * 2u);
    const uint32_t x_tok = static_cast<uint32_t>(a.C) * (kChunkK * 2u);  // bytes per token's activations

    // residual of the first unit's rows, read now rather than in the epilogue
    float res_first[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        res_first[t] = 0.f;
        if (EPI == EPI_RESID && threadIdx.x < a.R && blockIdx.x * a.R + static_cast<int>(threadIdx.x) < a.n_out)
            res_first[t] = bf16_bits_to_f32(a.residual[t * a.n_out + blockIdx.x * a.R + threadIdx.x]);
    }

    bool aborted = false;
    int slot = 0, lap = 0;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        float acc[kCcRows * MT];
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i) acc[i] = 0.f;
        for (int c = 0; c < a.Cp; ++c) {
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && c < n_mine) {
                const int kc = c * a.P + p;
                const uint32_t stage = ring + slot * a.stage_bytes;
                uint32_t xw[MT * (KS / 2)];
                const uint32_t xc = x0 + static_cast<uint32_t>(c) * x_step;
                float pe[MT], gxs[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
#pragma unroll
                    for (int i = 0; i < KS / 8; ++i) {
                        const uint4 v = lds128(xc + t * x_tok + i * NSEG * 16);
                        uint32_t* d = xw + t * (KS / 2) + 4 * i;
                        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
                    }
                    pe[t] = pe_all[t * a.C + kc];
                    gxs[t] = gx[(t * a.C + kc) * NSEG + seg];
                }
                if (up_box) {
                    if (!MIXED || fl[kc] == 0)
                        cc_stage_q45<NSEG, BITS_U, false, MT>(cc_geom(a), stage, b2, row0, seg, xw, pe, gxs, acc);
                    else
                        cc_stage_q45<NSEG, BITS_U, true, MT>(cc_geom(a), stage, b2, row0, seg, xw, pe, gxs, acc);
                } else {
                    if (!MIXED || fl[kc] == 0)
                        cc_stage_q45<NSEG, BITS, false, MT>(cc_geom(a), stage, b2, row0, seg, xw, pe, gxs, acc);
                    else
                        cc_stage_q45<NSEG, BITS, true, MT>(cc_geom(a), stage, b2, row0, seg, xw, pe, gxs, acc);
                }
            }
            // every compute thread arrives: its own reads of the slot are done
            mbar_arrive(&empty[slot]);
            if (++slot == a.n_stages) {
                slot = 0;
                ++lap;
            }
        }

        // ---------------- fixed-order reduction over segments (a butterfly
        // across the segment lanes of the warp) and phases, epilogue
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i)
#pragma unroll
            for (int off = NSEG / 2; off >= 1; off >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
        if (active && seg == 0) {
#pragma unroll
            for (int i = 0; i < kCcRows; ++i)
#pragma unroll
                for (int t = 0; t < MT; ++t) red[(b2 * a.R8 + row0 + i) * MT + t] = acc[i * MT + t];
        }
        named_barrier_sync(1, kCcThreads);
        if (!aborted) {
            const int r0 = u * a.R;
            for (int r = threadIdx.x; r < a.R; r += kCcThreads) {
                if (r0 + r >= a.n_out) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    float v[NGU];
#pragma unroll
                    for (int gg = 0; gg < NGU; ++gg) {
                        float s = 0.f;
                        for (int pp = 0; pp < a.P; ++pp) s += red[((pp * NGU + gg) * a.R8 + r) * MT + t];
                        v[gg] = s;
                    }
                    float val = v[0];
                    if (EPI == EPI_SWIGLU) val = (val / (1.0f + expf(-val))) * v[NGU - 1];
                    const int o = t * a.n_out + r0 + r;
                    if (EPI == EPI_RESID)
                        val += u == static_cast<int>(blockIdx.x) && r == static_cast<int>(threadIdx.x)
                                   ? res_first[t]
                                   : bf16_bits_to_f32(a.residual[o]);
                    if (a.out_f32)
                        reinterpret_cast<float*>(a.y)[o] = val;
                    else
                        reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(val);
                }
            }
        }
        named_barrier_sync(1, kCcThreads);
    }
}

// The groupwise-int maps of one matrix: codes (q_lo), scales, mins, Q5 plane.
struct Q45Maps {
    CUtensorMap m[2][4];  // [gate or only matrix, SwiGLU up matrix][codes, scales, mins, hi]
};

template <int BITS, int EPI, int NSEG, int BITS_U, int MT>
__global__ void __launch_bounds__(kCcAllThreads, 1)
    cc_q45_kernel(const __grid_constant__ CcArgs a, const __grid_constant__ Q45Maps maps)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCcMaxStages);
    volatile int* any_bf = abort_flag + 1;  // some chunk of x kept raw bf16

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
        // ------------------------------------------------------------ producer
        if (elect_one()) {
            for (int gg = 0; gg < NGU; ++gg) {
                prefetch_tensormap(&maps.m[gg][0]);
                prefetch_tensormap(&maps.m[gg][1]);
                prefetch_tensormap(&maps.m[gg][2]);
                if ((gg ? BITS_U : BITS) == 5) prefetch_tensormap(&maps.m[gg][3]);
            }
        }
        __syncwarp();
        int slot = 0, lap = 0, issued = 0;
        bool stop = false;
        for (int u = blockIdx.x; u < a.n_units && !stop; u += gridDim.x) {
            const int row = u * a.R;
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
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(live) * a.box_tx);
                    for (int pp = 0; pp < a.P; ++pp) {
                        const int kc = c * a.P + pp;
                        if (kc >= a.C) continue;
#pragma unroll
                        for (int gg = 0; gg < NGU; ++gg) {
                            const uint32_t bx = static_cast<uint32_t>(pp * NGU + gg) * a.R8;
                            tma_load_2d(sb + bx * 128, &maps.m[gg][0], kc * (kChunkK / 2), row, &full[slot]);
                            tma_load_2d(sb + a.scales_off + bx * 16, &maps.m[gg][1], kc * (kChunkK / 32), row,
                                        &full[slot]);
                            tma_load_2d(sb + a.mins_off + bx * 16, &maps.m[gg][2], kc * (kChunkK / 32), row,
                                        &full[slot]);
                            if ((gg ? BITS_U : BITS) == 5)
                                tma_load_2d(sb + a.hi_off + bx * 32, &maps.m[gg][3], kc * (kChunkK / 8), row,
                                            &full[slot]);
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
        cc_zero_padding(a, smem, a.P * NGU, roff, rbytes, (BITS == 5 || BITS_U == 5) ? 4 : 3);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    cc_convert_q45<NSEG, XSRC_NC, kCcWarps, MT>(a, smem, warp, lane, any_bf);
    named_barrier_sync(1, kCcThreads);
    if (*any_bf)
        cc_q45_units<BITS, EPI, NSEG, true, BITS_U, MT>(a, smem, full, empty, abort_flag);
    else
        cc_q45_units<BITS, EPI, NSEG, false, BITS_U, MT>(a, smem, full, empty, abort_flag);
}


constexpr uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

template <int EPI, int NSEG, int MT>
qg_status cc_launch(CcArgs a, const CUtensorMap& tmc, const CUtensorMap& tms, int grid, cudaStream_t stream)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;

    const uint32_t nbox = static_cast<uint32_t>(a.P * NGU);
    a.scales_off = nbox * a.R8 * 128u;
    a.stage_bytes = align_up(a.scales_off + nbox * a.R8 * 16u, 1024);
    a.box_tx = static_cast<uint32_t>(a.R) * (128u + 16u);
    const uint32_t x_bytes = static_cast<uint32_t>(MT * a.C) * kChunkK * 2u;
    const uint32_t pe_bytes = align_up(static_cast<uint32_t>(MT * a.C) * 4u, 16);
    const uint32_t fl_bytes = align_up(static_cast<uint32_t>(a.C), 16);
    const uint32_t ss_bytes = a.norm_w ? align_up(static_cast<uint32_t>(MT * a.C) * 4u, 16) : 0u;
    const uint32_t red_bytes = align_up(nbox * a.R8 * 4u * MT, 128);
    const uint32_t bar_bytes = 2 * kCcMaxStages * 8 + 16;
    const uint32_t fixed = x_bytes + pe_bytes + fl_bytes + ss_bytes + red_bytes + bar_bytes;
    if (fixed + 3 * a.stage_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
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
    a.smem_ss = so;
    so += ss_bytes;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;

    auto kern = cc_gemv_kernel<EPI, NSEG, MT>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[dev] = true;
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
    if (cudaLaunchKernelEx(&cfg, kern, a, tmc, tms) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <int EPI>
qg_status cc_dispatch(const CcArgs& a, const CUtensorMap& tmc, const CUtensorMap& tms, int grid,
                      cudaStream_t stream, int M)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    // 8 segments of 32 k when the rows fill 16 warps that way, else 16 of 16 k
    const int items8 = a.P * NGU * ((a.R + kCcRows - 1) / kCcRows) * 8;
    if (M == 2) {
        if (items8 > kCcThreads / 2) return cc_launch<EPI, 8, 2>(a, tmc, tms, grid, stream);
        return cc_launch<EPI, 16, 2>(a, tmc, tms, grid, stream);
    }
    if (items8 > kCcThreads / 2) return cc_launch<EPI, 8, 1>(a, tmc, tms, grid, stream);
    return cc_launch<EPI, 16, 1>(a, tmc, tms, grid, stream);
}

template <int BITS, int EPI, int NSEG, int BITS_U, int MT>
qg_status cc_q45_launch(CcArgs a, const Q45Maps& maps, int grid, cudaStream_t stream)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    constexpr bool any5 = BITS == 5 || BITS_U == 5;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;

    const uint32_t nbox = static_cast<uint32_t>(a.P * NGU);
    a.scales_off = nbox * a.R8 * 128u;
    a.mins_off = a.scales_off + nbox * a.R8 * 16u;
    a.hi_off = a.mins_off + nbox * a.R8 * 16u;
    a.stage_bytes = align_up(a.hi_off + (any5 ? nbox * a.R8 * 32u : 0u), 1024);
    // bytes one phase brings in (its gate box and, for SwiGLU, its up box)
    a.box_tx = static_cast<uint32_t>(a.R) * (128u + 16u + 16u + (BITS == 5 ? 32u : 0u));
    if (NGU == 2) a.box_tx += static_cast<uint32_t>(a.R) * (128u + 16u + 16u + (BITS_U == 5 ? 32u : 0u));
    const uint32_t x_bytes = static_cast<uint32_t>(MT * a.C) * kChunkK * 2u;
    const uint32_t pe_bytes = align_up(static_cast<uint32_t>(MT * a.C) * 4u, 16);
    const uint32_t gx_bytes = align_up(static_cast<uint32_t>(MT * a.C * NSEG) * 4u, 16);
    const uint32_t fl_bytes = align_up(static_cast<uint32_t>(a.C), 16);
    const uint32_t ss_bytes = a.norm_w ? align_up(static_cast<uint32_t>(MT * a.C) * 4u, 16) : 0u;
    const uint32_t red_bytes = align_up(nbox * a.R8 * 4u * MT, 128);
    const uint32_t bar_bytes = 2 * kCcMaxStages * 8 + 16;
    const uint32_t fixed = x_bytes + pe_bytes + gx_bytes + fl_bytes + ss_bytes + red_bytes + bar_bytes;
    if (fixed + 3 * a.stage_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    a.n_stages = std::min<int>(kCcMaxStages, static_cast<int>((kCcSmemMax - fixed) / a.stage_bytes));

    uint32_t so = 0;
    a.smem_ring = so;
    so += a.n_stages * a.stage_bytes;
    a.smem_x = so;
    so += x_bytes;
    a.smem_pe = so;
    so += pe_bytes;
    a.smem_gx = so;
    so += gx_bytes;
    a.smem_fl = so;
    so += fl_bytes;
    a.smem_ss = so;
    so += ss_bytes;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;

    auto kern = cc_q45_kernel<BITS, EPI, NSEG, BITS_U, MT>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[dev] = true;
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
    if (cudaLaunchKernelEx(&cfg, kern, a, maps) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

template <int BITS, int EPI, int BITS_U = BITS>
qg_status cc_q45_dispatch(const CcArgs& a, const Q45Maps& maps, int grid, cudaStream_t stream, int M)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    const int items8 = a.P * NGU * ((a.R + kCcRows - 1) / kCcRows) * 8;
    if (M == 2) {
        if (items8 > kCcThreads / 2) return cc_q45_launch<BITS, EPI, 8, BITS_U, 2>(a, maps, grid, stream);
        return cc_q45_launch<BITS, EPI, 16, BITS_U, 2>(a, maps, grid, stream);
    }
    if (items8 > kCcThreads / 2) return cc_q45_launch<BITS, EPI, 8, BITS_U, 1>(a, maps, grid, stream);
    return cc_q45_launch<BITS, EPI, 16, BITS_U, 1>(a, maps, grid, stream);
}

}  // namespace

// One-token NVFP4 GEMV on the CUDA cores; QG_ERR_UNSUPPORTED for other M,
// for K not a multiple of 256 or when x does not fit in shared memory.
qg_status launch_cc_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > 2 || K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
    const int ngu = swiglu ? 2 : 1;
    const int n_out = swiglu ? N / 2 : N;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    // Smallest number of units per CTA whose rows fit the 256-row budget of
    // one stage; R = ceil(n_out / (SMs * units)) gives every SM the same
    // byte count.
    int R = 1;
    for (int U = 1;; ++U) {
        R = (n_out + sms * U - 1) / (sms * U);
        if (ngu * ((R + 7) / 8 * 8) <= 256) break;
    }
    R = std::max(R, 1);
    CcArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.residual = static_cast<const uint16_t*>(residual);
    a.norm_w = static_cast<const uint16_t*>(norm_w);
    a.norm_eps = norm_eps;
    a.K = K;
    a.C = K / kChunkK;
    a.n_out = n_out;
    a.R = R;
    a.R8 = (R + 7) / 8 * 8;
    a.P = std::max(1, std::min(256 / (ngu * a.R8), a.C));
    a.Cp = (a.C + a.P - 1) / a.P;
    a.up_row_offset = swiglu ? n_out : 0;
    a.out_f32 = swiglu ? 0 : out_f32;
    a.g = g;
    a.n_units = (n_out + R - 1) / R;
    const int grid = std::min(sms, a.n_units);
    CUtensorMap tmc, tms;
    memset(&tmc, 0, sizeof(tmc));
    memset(&tms, 0, sizeof(tms));
    if (!encode_tmap_2d(&tmc, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, R, true) ||
        !encode_tmap_2d(&tms, scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, N, 16, R, false))
        return QG_ERR_CUDA;
    if (swiglu) return cc_dispatch<EPI_SWIGLU>(a, tmc, tms, grid, stream, M);
    if (residual) return cc_dispatch<EPI_RESID>(a, tmc, tms, grid, stream, M);
    return cc_dispatch<EPI_NONE>(a, tmc, tms, grid, stream, M);
}

namespace {

// The groupwise-int plan for one token: units of R rows (per matrix) over all
// of K, P phases so that P * ngu boxes of R8 rows fill at most 256 rows.
CcArgs q45_plan(const void* x, void* y, int out_f32, const void* residual, int n_out, int ngu, int K,
                const void* norm_w, float norm_eps)
{
    const int sms = sm_count(-1);
    int R = 1;
    for (int U = 1;; ++U) {
        R = (n_out + sms * U - 1) / (sms * U);
        if (ngu * ((R + 7) / 8 * 8) <= 256) break;
    }
    R = std::max(R, 1);
    CcArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.residual = static_cast<const uint16_t*>(residual);
    a.norm_w = static_cast<const uint16_t*>(norm_w);
    a.norm_eps = norm_eps;
    a.K = K;
    a.C = K / kChunkK;
    a.n_out = n_out;
    a.R = R;
    a.R8 = (R + 7) / 8 * 8;
    a.P = std::max(1, std::min(256 / (ngu * a.R8), a.C));
    a.Cp = (a.C + a.P - 1) / a.P;
    a.out_f32 = out_f32;
    a.g = 1.f;
    a.n_units = (n_out + R - 1) / R;
    return a;
}

bool q45_maps(CUtensorMap (&m)[4], const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min,
              int bits, int N, int K, int R)
{
    memset(m, 0, sizeof(m));
    if (!encode_tmap_2d(&m[0], q_lo, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, R, true) ||
        !encode_tmap_2d(&m[1], scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false) ||
        !encode_tmap_2d(&m[2], min, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false))
        return false;
    if (bits == 5) return encode_tmap_2d(&m[3], q_hi, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, N, 32, R, false);
    m[3] = m[2];
    return true;
}

}  // namespace

// One-token Q4/Q5 GEMV on the CUDA cores; QG_ERR_UNSUPPORTED for other M,
// for K not a multiple of 256 or when x does not fit in shared memory.
qg_status launch_cc_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                              const void* x, void* y, int out_f32, const void* residual, int M, int N, int K,
                              cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > 2 || K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
    if (sm_count(-1) <= 0) return QG_ERR_CUDA;
    const CcArgs a = q45_plan(x, y, out_f32, residual, N, 1, K, norm_w, norm_eps);
    const int grid = std::min(sm_count(-1), a.n_units);
    Q45Maps maps;
    if (!q45_maps(maps.m[0], q_lo, q_hi, scale, min, bits, N, K, a.R)) return QG_ERR_CUDA;
    maps.m[1][0] = maps.m[1][1] = maps.m[1][2] = maps.m[1][3] = maps.m[0][0];
    if (bits == 5) {
        if (residual) return cc_q45_dispatch<5, EPI_RESID>(a, maps, grid, stream, M);
        return cc_q45_dispatch<5, EPI_NONE>(a, maps, grid, stream, M);
    }
    if (residual) return cc_q45_dispatch<4, EPI_RESID>(a, maps, grid, stream, M);
    return cc_q45_dispatch<4, EPI_NONE>(a, maps, grid, stream, M);
}

// One-token SwiGLU over separate groupwise-int gate and up matrices (I rows
// each, gate_bits / up_bits wide), y bf16 [I]; QG_ERR_UNSUPPORTED as above.
qg_status launch_cc_swiglu_q45(const Q45Matrix& gate, const Q45Matrix& up, const void* x, void* y, int M, int I,
                               int K, cudaStream_t stream, const void* norm_w, float norm_eps)
{
    if (M < 1 || M > 2 || K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
    if (sm_count(-1) <= 0) return QG_ERR_CUDA;
    const CcArgs a = q45_plan(x, y, 0, nullptr, I, 2, K, norm_w, norm_eps);
    const int grid = std::min(sm_count(-1), a.n_units);
    Q45Maps maps;
    if (!q45_maps(maps.m[0], gate.q_lo, gate.q_hi, gate.scale, gate.min, gate.bits, I, K, a.R) ||
        !q45_maps(maps.m[1], up.q_lo, up.q_hi, up.scale, up.min, up.bits, I, K, a.R))
        return QG_ERR_CUDA;
    if (gate.bits == 5 && up.bits == 4) return cc_q45_dispatch<5, EPI_SWIGLU, 4>(a, maps, grid, stream, M);
    if (gate.bits == 5 && up.bits == 5) return cc_q45_dispatch<5, EPI_SWIGLU, 5>(a, maps, grid, stream, M);
    if (gate.bits == 4 && up.bits == 5) return cc_q45_dispatch<4, EPI_SWIGLU, 5>(a, maps, grid, stream, M);
    return cc_q45_dispatch<4, EPI_SWIGLU, 4>(a, maps, grid, stream, M);
}

}  // namespace qg
