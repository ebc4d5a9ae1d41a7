// qgemv_chain.cu -- the one- or two-token projections of a decode layer in
// one persistent launch.
//
// Decode engines replay one fixed sequence of projections per layer (NInfer
// article, section 1: one CUDA graph per batch size; Decapybara README,
// "Blackwell CUDA 内核套件": a persistent single-launch decode loop,
// megakernel.cu). Launched one by one, every projection pays its own start
// (launch, barrier set-up, the first weight stage's latency, the wait for the
// previous kernel) and its own tail (the slowest CTA, the epilogue), and on
// one GB300 those fixed costs were about a fifth of a 27B-class layer.
//
// Here one CTA per SM walks the whole list. Its TMA warp streams the weights
// of op after op into one shared-memory ring without stopping at an op
// boundary (weights never depend on earlier outputs), so the next op's first
// stages are already in flight while the compute warps finish the current op.
// The compute warps run each op exactly as the one- and two-token kernels of
// qgemv_cc.cu do (same units, phases, exact activation conversion and
// fixed-order reductions, so results are identical to separate calls): they
// convert the op's activations into shared memory, stream its units and
// write its outputs. An op that reads an earlier op's output first waits at a
// grid-wide barrier (bounded, sense-reversing, on two caller-owned words),
// and then reads activations and residuals through L2 only.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "mt_core.cuh"

namespace qg {

namespace {

constexpr int kChainMaxOps = 8;
constexpr int kChainNseg = 8;   // 32-k segments (always valid: at most 256 rows per stage)

struct ChainOp {
    CcArgs a;   // the op's plan, as the standalone kernel would use it
    int fmt;    // FMT_NVFP4, FMT_Q4, FMT_Q5 (the gate matrix of a SwiGLU)
    int epi;    // EPI_NONE, EPI_RESID, EPI_SWIGLU
    int dep;    // grid-wide barrier before the op reads its inputs
    int ufmt;   // groupwise-int SwiGLU: the up matrix's format
    // 3..8 tokens (the warp-MMA stage): 16-row blocks per box, activation
    // window in chunks, bytes between tokens' activations
    int NRB;
    int W;
    uint32_t x_tok;
};

struct ChainParams {
    // codes, scales, mins, Q5 high plane; then the same for a separate
    // groupwise-int SwiGLU up matrix
    CUtensorMap map[kChainMaxOps][8];
    ChainOp op[kChainMaxOps];
    int n_ops;
    int M;                             // tokens (3..8 in the warp-MMA kernel)
    int n_stages;
    uint32_t slot_bytes;               // ring slot stride (the largest op's stage)
    uint32_t smem_bar;
    uint32_t* sync;                    // [0] arrivals, [1] generation; nullptr without barriers
    uint64_t wait_ns;
    int starve;
    int* status;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier among the compute warps of all CTAs. Thread 0 of each CTA
// arrives once all of its CTA's compute threads are here (their earlier
// global writes ordered before the arrival); the last arrival resets the
// count and advances the generation the others wait on. Bounded: on expiry
// it records QG_ERR_DEVICE_TIMEOUT and sets the CTA's abort flag.
__device__ void chain_grid_barrier(const ChainParams& p, volatile int* abort_flag)
{
    named_barrier_sync(1, kCcThreads);
    if (threadIdx.x == 0 && !*abort_flag) {
        uint32_t* count = p.sync;
        uint32_t* gen = p.sync + 1;
        __threadfence();
        const uint32_t g0 = ld_acquire_u32(gen);
        if (atomicAdd(count, 1u) == gridDim.x - 1) {
            atomicExch(count, 0u);
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_u32(gen) == g0) {
                __nanosleep(64);
                if (global_timer_ns() - t0 > p.wait_ns) {
                    set_device_status(p.status, QG_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
        }
        __threadfence();
    }
    named_barrier_sync(1, kCcThreads);
}

__device__ __forceinline__ void chain_store(const CcArgs& a, int idx, float val)
{
    if (a.out_f32)
        reinterpret_cast<float*>(a.y)[idx] = val;
    else
        reinterpret_cast<uint16_t*>(a.y)[idx] = f32_to_bf16_bits_rn(val);
}

// The compute warps' unit loop of one NVFP4 op (cc_units of qgemv_cc.cu with
// the ring position carried across ops, coherent residual loads, and the
// epilogue chosen at run time: it only runs after a unit's stage loop, and one
// loop copy for all epilogues keeps the kernel's code small).
template <bool MIXED, int MT>
__device__ __forceinline__ void chain_units_nvfp4(const CcArgs& a, int epi, uint8_t* smem, uint32_t ring,
                                                  uint32_t slot_bytes, int n_stages, uint64_t* full,
                                                  uint64_t* empty, volatile int* abort_flag, bool& aborted,
                                                  int& slot, int& lap)
{
    constexpr int NSEG = kChainNseg;
    constexpr int KS = kChunkK / NSEG;
    const bool swiglu = epi == EPI_SWIGLU, resid = epi == EPI_RESID;
    const int gsh = swiglu ? 1 : 0;   // log2 of the boxes per phase (gate and up rows)
    // the op's plan in registers (the parameter block is indexed by op)
    const CcGeom geom = cc_geom_chunked(a, gsh);
    const int R = a.R, P = a.P, C = a.C, Cp = a.Cp, n_units = a.n_units, n_out = a.n_out;
    const float gscale = a.g;
    const int rg_per_box = (R + kCcRows - 1) / kCcRows;
    const int item = threadIdx.x;
    const int seg = item % NSEG;
    const int bg = item / NSEG;
    const int b2 = bg / rg_per_box;
    const int row0 = (bg % rg_per_box) * kCcRows;
    const bool active = b2 < (P << gsh);
    const int p = active ? b2 >> gsh : 0;
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(smem + a.smem_x);
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const uint8_t* fl = smem + a.smem_fl;
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const int n_mine = active ? max(0, (C - p + P - 1) / P) : 0;
    const uint32_t x0 = smem_u32(xs + p * (kChunkK / 2) + seg * 4);
    const uint32_t x_step = static_cast<uint32_t>(P) * (kChunkK * 2u);
    const uint32_t x_tok = static_cast<uint32_t>(C) * (kChunkK * 2u);
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        float acc[kCcRows * MT];
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i) acc[i] = 0.f;
        // the unit's residuals, read while its stages stream
        float res[MT];
        const int r0 = u * R;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            res[t] = 0.f;
            if (resid && threadIdx.x < R && r0 + static_cast<int>(threadIdx.x) < n_out)
                res[t] = bf16_bits_to_f32(ldg_cg_u16(a.residual + t * n_out + r0 + threadIdx.x));
        }
        for (int c = 0; c < Cp; ++c) {
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && c < n_mine) {
                const uint32_t stage = ring + slot * slot_bytes;
                const uint32_t xc = x0 + static_cast<uint32_t>(c) * x_step;
                const int kc = c * P + p;
                if constexpr (MT == 1) {
                    uint32_t xw[KS / 2];
#pragma unroll
                    for (int i = 0; i < KS / 8; ++i) {
                        const uint4 v = lds128(xc + i * NSEG * 16);
                        xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
                    }
                    if (!MIXED || fl[kc] == 0)
                        cc_stage<NSEG, false>(geom, stage, b2, row0, seg, xw, pe_all[kc], acc);
                    else
                        cc_stage<NSEG, true>(geom, stage, b2, row0, seg, xw, pe_all[kc], acc);
                } else {
                    float pe[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) pe[t] = pe_all[t * C + kc];
                    if (!MIXED || fl[kc] == 0)
                        cc_stage_mt<NSEG, false, MT>(geom, stage, b2, row0, seg, xc, x_tok, pe, acc);
                    else
                        cc_stage_mt<NSEG, true, MT>(geom, stage, b2, row0, seg, xc, x_tok, pe, acc);
                }
            }
            mbar_arrive(&empty[slot]);
            if (++slot == n_stages) {
                slot = 0;
                ++lap;
            }
        }
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
            for (int r = threadIdx.x; r < R; r += kCcThreads) {
                if (r0 + r >= n_out) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    float v0 = 0.f, v1 = 0.f;
                    for (int pp = 0; pp < P; ++pp) v0 += red[((pp << gsh) * a.R8 + r) * MT + t];
                    v0 *= gscale;
                    float val = v0;
                    if (swiglu) {
                        for (int pp = 0; pp < P; ++pp) v1 += red[(((pp << gsh) + 1) * a.R8 + r) * MT + t];
                        v1 *= gscale;
                        val = (v0 / (1.0f + expf(-v0))) * v1;
                    }
                    const int o = t * n_out + r0 + r;
                    if (resid)
                        val += r == static_cast<int>(threadIdx.x) ? res[t]
                                                                  : bf16_bits_to_f32(ldg_cg_u16(a.residual + o));
                    chain_store(a, o, val);
                }
            }
        }
        named_barrier_sync(1, kCcThreads);
    }
}

// The unit loop of one groupwise-int op (cc_q45_units of qgemv_cc.cu, as
// above): the epilogue at run time; SwiGLU reads a gate box (BITS) and an up
// box (BITS_U) per phase.
template <int BITS, int BITS_U, bool MIXED, int MT>
__device__ __forceinline__ void chain_units_q45(const CcArgs& a, int epi, uint8_t* smem, uint32_t ring,
                                                uint32_t slot_bytes, int n_stages, uint64_t* full, uint64_t* empty,
                                                volatile int* abort_flag, bool& aborted, int& slot, int& lap)
{
    constexpr int NSEG = kChainNseg;
    constexpr int KS = kChunkK / NSEG;
    const bool swiglu = epi == EPI_SWIGLU, resid = epi == EPI_RESID;
    const int gsh = swiglu ? 1 : 0;
    const CcGeom geom = cc_geom_chunked(a, gsh);
    const int R = a.R, P = a.P, C = a.C, Cp = a.Cp, n_units = a.n_units, n_out = a.n_out;
    const int rg_per_box = (R + kCcRows - 1) / kCcRows;
    const int item = threadIdx.x;
    const int seg = item % NSEG;
    const int bg = item / NSEG;
    const int b2 = bg / rg_per_box;
    const int row0 = (bg % rg_per_box) * kCcRows;
    const bool active = b2 < (P << gsh);
    const int p = active ? b2 >> gsh : 0;
    const bool up_box = swiglu && (b2 & 1);
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(smem + a.smem_x);
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const float* gx = reinterpret_cast<const float*>(smem + a.smem_gx);
    const uint8_t* fl = smem + a.smem_fl;
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const int n_mine = active ? max(0, (C - p + P - 1) / P) : 0;
    const uint32_t x0 = smem_u32(xs + p * (kChunkK / 2) + seg * 4);
    const uint32_t x_step = static_cast<uint32_t>(P) * (kChunkK * 2u);
    const uint32_t x_tok = static_cast<uint32_t>(C) * (kChunkK * 2u);
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        float acc[kCcRows * MT];
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i) acc[i] = 0.f;
        // the unit's residuals, read while its stages stream
        float res[MT];
        const int r0 = u * R;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            res[t] = 0.f;
            if (resid && threadIdx.x < R && r0 + static_cast<int>(threadIdx.x) < n_out)
                res[t] = bf16_bits_to_f32(ldg_cg_u16(a.residual + t * n_out + r0 + threadIdx.x));
        }
        for (int c = 0; c < Cp; ++c) {
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && c < n_mine) {
                const int kc = c * P + p;
                const uint32_t stage = ring + slot * slot_bytes;
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
                    gxs[t] = gx[(t * C + kc) * NSEG + seg];
                    pe[t] = pe_all[t * C + kc];
                }
                const bool bf = MIXED && fl[kc] != 0;
                if (up_box) {
                    if (bf)
                        cc_stage_q45<NSEG, BITS_U, true, MT>(geom, stage, b2, row0, seg, xw, pe, gxs, acc);
                    else
                        cc_stage_q45<NSEG, BITS_U, false, MT>(geom, stage, b2, row0, seg, xw, pe, gxs, acc);
                } else {
                    if (bf)
                        cc_stage_q45<NSEG, BITS, true, MT>(geom, stage, b2, row0, seg, xw, pe, gxs, acc);
                    else
                        cc_stage_q45<NSEG, BITS, false, MT>(geom, stage, b2, row0, seg, xw, pe, gxs, acc);
                }
            }
            mbar_arrive(&empty[slot]);
            if (++slot == n_stages) {
                slot = 0;
                ++lap;
            }
        }
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
            for (int r = threadIdx.x; r < R; r += kCcThreads) {
                if (r0 + r >= n_out) break;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    float val = 0.f;
                    for (int pp = 0; pp < P; ++pp) val += red[((pp << gsh) * a.R8 + r) * MT + t];
                    if (swiglu) {
                        float v1 = 0.f;
                        for (int pp = 0; pp < P; ++pp) v1 += red[(((pp << gsh) + 1) * a.R8 + r) * MT + t];
                        val = (val / (1.0f + expf(-val))) * v1;
                    }
                    const int o = t * n_out + r0 + r;
                    if (resid)
                        val += r == static_cast<int>(threadIdx.x) ? res[t]
                                                                  : bf16_bits_to_f32(ldg_cg_u16(a.residual + o));
                    chain_store(a, o, val);
                }
            }
        }
        named_barrier_sync(1, kCcThreads);
    }
}

template <int MT>
__device__ __forceinline__ void chain_nvfp4(const CcArgs& a, int epi, bool mixed, uint8_t* smem, uint32_t ring,
                                            uint32_t slot_bytes, int n_stages, uint64_t* full, uint64_t* empty,
                                            volatile int* abort_flag, bool& aborted, int& slot, int& lap)
{
    if (mixed)
        chain_units_nvfp4<true, MT>(a, epi, smem, ring, slot_bytes, n_stages, full, empty, abort_flag, aborted, slot,
                                lap);
    else
        chain_units_nvfp4<false, MT>(a, epi, smem, ring, slot_bytes, n_stages, full, empty, abort_flag, aborted, slot,
                                 lap);
}

template <int BITS, int BITS_U, int MT>
__device__ __forceinline__ void chain_q45(const CcArgs& a, int epi, bool mixed, uint8_t* smem, uint32_t ring,
                                          uint32_t slot_bytes, int n_stages, uint64_t* full, uint64_t* empty,
                                          volatile int* abort_flag, bool& aborted, int& slot, int& lap)
{
    if (mixed)
        chain_units_q45<BITS, BITS_U, true, MT>(a, epi, smem, ring, slot_bytes, n_stages, full, empty, abort_flag,
                                            aborted, slot, lap);
    else
        chain_units_q45<BITS, BITS_U, false, MT>(a, epi, smem, ring, slot_bytes, n_stages, full, empty, abort_flag,
                                             aborted, slot, lap);
}

// The TMA warp of a chained launch: the weight stages of op after op into one
// ring, without a stop at an op boundary (weights never depend on outputs).
__device__ __forceinline__ void chain_producer(const ChainParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                               volatile int* abort_flag, int lane)
{
    // ------------------------------------------------------------ producer
    if (elect_one()) {
        for (int o = 0; o < p.n_ops; ++o) {
            prefetch_tensormap(&p.map[o][0]);
            prefetch_tensormap(&p.map[o][1]);
            if (p.op[o].fmt != FMT_NVFP4) prefetch_tensormap(&p.map[o][2]);
            if (p.op[o].fmt == FMT_Q5) prefetch_tensormap(&p.map[o][3]);
            if (p.op[o].fmt != FMT_NVFP4 && p.op[o].epi == EPI_SWIGLU)
                for (int i = 4; i < 8; ++i) prefetch_tensormap(&p.map[o][i]);
        }
    }
    __syncwarp();
    int slot = 0, lap = 0, issued = 0;
    bool stop = false;
    for (int o = 0; o < p.n_ops && !stop; ++o) {
        const CcArgs& a = p.op[o].a;
        const int fmt = p.op[o].fmt;
        const int ngu = p.op[o].epi == EPI_SWIGLU ? 2 : 1;
        const int P = a.P, Cp = a.Cp, R = a.R, n_units = a.n_units, up_off = a.up_row_offset;
        const uint32_t cpitch = a.code_pitch, spitch = a.sc_pitch;
        const uint32_t scales_off = a.scales_off, mins_off = a.mins_off, hi_off = a.hi_off, box_tx = a.box_tx;
        for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
            const int row0 = u * R;
            for (int c = 0; c < Cp; ++c) {
                if (lap > 0 && !cc_wait_warp(&empty[slot], (lap - 1) & 1, a, abort_flag)) {
                    stop = true;
                    break;
                }
                if (*abort_flag || p.starve) {
                    stop = true;
                    break;
                }
                uint8_t* sb = smem + a.smem_ring + slot * p.slot_bytes;
                if (elect_one()) {
                    // per matrix one box of the stage's P chunks x R rows
                    // (chunks past K are filled with zeros and still counted)
                    mbar_arrive_expect_tx(&full[slot], box_tx);
                    const int kc0 = c * P;
                    for (int gg = 0; gg < ngu; ++gg) {
                        if (fmt == FMT_NVFP4) {
                            const int row = row0 + gg * up_off;
                            tma_load_3d(sb + gg * cpitch, &p.map[o][0], 0, row, kc0, &full[slot]);
                            tma_load_3d(sb + scales_off + gg * spitch, &p.map[o][1], 0, row, kc0, &full[slot]);
                        } else {
                            // gate (or only) box, then a SwiGLU's up box: same rows of two matrices
                            const CUtensorMap* mp = &p.map[o][4 * gg];
                            tma_load_3d(sb + gg * cpitch, mp, 0, row0, kc0, &full[slot]);
                            tma_load_3d(sb + scales_off + gg * spitch, mp + 1, 0, row0, kc0, &full[slot]);
                            tma_load_3d(sb + mins_off + gg * spitch, mp + 2, 0, row0, kc0, &full[slot]);
                            if ((gg ? p.op[o].ufmt : fmt) == FMT_Q5)
                                tma_load_3d(sb + hi_off + gg * 2u * spitch, mp + 3, 0, row0, kc0, &full[slot]);
                        }
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == p.n_stages) {
                    slot = 0;
                    ++lap;
                }
            }
        }
    }
    // No copy may still be landing in shared memory when the CTA exits.
    if (lane == 0)
        for (int g = max(0, issued - p.n_stages); g < issued; ++g)
            mbar_wait_bounded(&full[g % p.n_stages], (g / p.n_stages) & 1, p.wait_ns, p.status);
    __syncwarp();
}

// MT tokens (1 or 2) per op: every op's activations, residuals and outputs
// are MT rows (K, N or n_out apart), as in the one- and two-token kernels.
template <int MT>
__global__ void __launch_bounds__(kCcAllThreads, 1) chain_kernel(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCcMaxStages);
    volatile int* any_bf = abort_flag + 1;

    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCcThreads);
        }
        *abort_flag = 0;
        *any_bf = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const uint32_t ring = smem_u32(smem + p.op[0].a.smem_ring);

    if (warp == kCcTmaWarp) {
        chain_producer(p, smem, full, empty, abort_flag, lane);
        return;
    }

    // ---------------------------------------------------------------- compute warps
    // The first op's inputs may come from the previous kernel on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool aborted = false;
    int slot = 0, lap = 0;
    for (int o = 0; o < p.n_ops; ++o) {
        const ChainOp& op = p.op[o];
        const CcArgs& a = op.a;
        if (op.dep) chain_grid_barrier(p, abort_flag);
        if (*abort_flag) aborted = true;
        if (threadIdx.x == 0) *any_bf = 0;
        named_barrier_sync(1, kCcThreads);
        // x through L2 only: an earlier op of this launch may have written it
        if (op.fmt == FMT_NVFP4) {
            if constexpr (MT == 1)
                cc_convert<kChainNseg, XSRC_CG>(a, smem, warp, lane, any_bf);
            else
                cc_convert_q45<kChainNseg, XSRC_CG, kCcWarps, MT, false>(a, smem, warp, lane, any_bf);
        } else {
            cc_convert_q45<kChainNseg, XSRC_CG, kCcWarps, MT>(a, smem, warp, lane, any_bf);
        }
        named_barrier_sync(1, kCcThreads);
        const bool mixed = *any_bf != 0;
        if (op.fmt == FMT_NVFP4) {
            chain_nvfp4<MT>(a, op.epi, mixed, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag, aborted,
                        slot, lap);
        } else {
            const bool b5 = op.fmt == FMT_Q5;
            const bool u5 = op.epi == EPI_SWIGLU ? op.ufmt == FMT_Q5 : b5;
            if (b5 && u5)
                chain_q45<5, 5, MT>(a, op.epi, mixed, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag,
                                aborted, slot, lap);
            else if (b5)
                chain_q45<5, 4, MT>(a, op.epi, mixed, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag,
                                aborted, slot, lap);
            else if (u5)
                chain_q45<4, 5, MT>(a, op.epi, mixed, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag,
                                aborted, slot, lap);
            else
                chain_q45<4, 4, MT>(a, op.epi, mixed, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag,
                                aborted, slot, lap);
        }
    }
}

// 3..8 tokens: the unit loop of one op on the warp-MMA stage (mt_units of
// qgemv_mt.cu with the ring position carried across ops, the epilogue chosen
// at run time, activations and residuals read through L2, and the op's plan
// in registers).
template <int BITS, bool MIXED, int BITS_U, bool NORM_OK>
__device__ __forceinline__ void chain_units_mt(const MtArgs& m, int epi, uint8_t* smem, uint32_t ring,
                                               uint32_t slot_bytes, int n_stages, uint64_t* full, uint64_t* empty,
                                               volatile int* abort_flag, volatile int* any_bf, bool& aborted,
                                               int& slot, int& lap, int warp, int lane)
{
    const CcArgs& a = m.a;
    const bool swiglu = epi == EPI_SWIGLU, resid = epi == EPI_RESID;
    const int ngu = swiglu ? 2 : 1;
    const int M = m.M, W = m.W, NRB = m.NRB;
    const int R = a.R, R8 = a.R8, P = a.P, C = a.C, Cp = a.Cp, n_units = a.n_units, n_out = a.n_out;
    const float gscale = a.g;
    const int b2 = warp / NRB;
    const int rb = warp % NRB;
    const bool active = b2 < P * ngu;
    const int p = active ? b2 / ngu : 0;
    const int n_mine = active ? max(0, (C - p + P - 1) / P) : 0;
    const int g = lane >> 2, c = lane & 3;
    const int t0 = 2 * c, t1 = 2 * c + 1;
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const uint8_t* fl = smem + a.smem_fl;
    const float* gx_all = reinterpret_cast<const float*>(smem + a.smem_gx);
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    // the chunked stage layout: matrix gm's box holds [chunk][row], R rows per
    // chunk (rows past R read the next chunk's rows or the slot's tail)
    const uint32_t gm = active ? static_cast<uint32_t>(b2 % ngu) : 0u;
    const uint32_t r0 = static_cast<uint32_t>(p * R + 16 * rb);
    const uint32_t sw = r0 & 7u;
    const uint32_t box_off = gm * a.code_pitch + r0 * 128u;
    const uint32_t sbox_off = a.scales_off + gm * a.sc_pitch + r0 * 16u;
    const uint32_t mbox_off = a.mins_off + gm * a.sc_pitch + r0 * 16u;
    const uint32_t hbox_off = a.hi_off + gm * 2u * a.sc_pitch + r0 * 32u;
    const uint32_t x0 = smem_u32(smem + a.smem_x) + static_cast<uint32_t>(g) * m.x_tok;

    int cur_win = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cc = 0; cc < Cp; ++cc) {
            const int win = (cc * P) / W;
            if (win != cur_win) {
                named_barrier_sync(1, kCcThreads);
                mt_convert_any<BITS != 0, true, NORM_OK>(m, smem, warp, lane, any_bf, win * W);
                named_barrier_sync(1, kCcThreads);
                cur_win = win;
            }
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && cc < n_mine) {
                const int kc = cc * P + p;
                const int j = kc - win * W;
                const uint32_t stage = ring + slot * slot_bytes;
                const uint32_t xc = x0 + static_cast<uint32_t>(j) * (kChunkK * 2u);
                const float pe0 = t0 < M ? pe_all[t0 * W + j] : 0.f;
                const float pe1 = t1 < M ? pe_all[t1 * W + j] : 0.f;
                const bool bf = MIXED && fl[j] != 0;
                if constexpr (BITS == 0) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    if (bf)
                        mt_stage<true>(stage + box_off, stage + sbox_off, xc, lane, M, d, sw);
                    else
                        mt_stage<false>(stage + box_off, stage + sbox_off, xc, lane, M, d, sw);
                    acc[0] = fmaf(d[0], pe0, acc[0]);
                    acc[1] = fmaf(d[1], pe1, acc[1]);
                    acc[2] = fmaf(d[2], pe0, acc[2]);
                    acc[3] = fmaf(d[3], pe1, acc[3]);
                } else {
                    float aq[4] = {0.f, 0.f, 0.f, 0.f}, am[4] = {0.f, 0.f, 0.f, 0.f};
                    const float* gx0 = gx_all + ((t0 < M ? t0 : 0) * W + j) * 8;
                    const float* gx1 = gx_all + ((t1 < M ? t1 : 0) * W + j) * 8;
                    if (swiglu && (b2 & 1)) {  // the up matrix's box
                        if (bf)
                            mtq_stage<BITS_U, true>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                    stage + hbox_off, xc, gx0, gx1, lane, M, aq, am, sw);
                        else
                            mtq_stage<BITS_U, false>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                     stage + hbox_off, xc, gx0, gx1, lane, M, aq, am, sw);
                    } else if (bf) {
                        mtq_stage<BITS, true>(stage + box_off, stage + sbox_off, stage + mbox_off, stage + hbox_off,
                                              xc, gx0, gx1, lane, M, aq, am, sw);
                    } else {
                        mtq_stage<BITS, false>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                               stage + hbox_off, xc, gx0, gx1, lane, M, aq, am, sw);
                    }
                    const float f0 = bf ? 1.0f : 16777216.0f * pe0, f1 = bf ? 1.0f : 16777216.0f * pe1;
                    acc[0] = fmaf(aq[0], f0, acc[0]) + am[0];
                    acc[1] = fmaf(aq[1], f1, acc[1]) + am[1];
                    acc[2] = fmaf(aq[2], f0, acc[2]) + am[2];
                    acc[3] = fmaf(aq[3], f1, acc[3]) + am[3];
                }
            }
            mbar_arrive(&empty[slot]);
            if (++slot == n_stages) {
                slot = 0;
                ++lap;
            }
        }
        if (active) {
            float* rw = red + static_cast<size_t>(b2 * R8 + 16 * rb + g) * 8;
            rw[t0] = acc[0];
            rw[t1] = acc[1];
            rw[64 + t0] = acc[2];
            rw[64 + t1] = acc[3];
        }
        named_barrier_sync(1, kCcThreads);
        if (!aborted) {
            const int r0 = u * R;
            for (int it = threadIdx.x; it < R * M; it += kCcThreads) {
                const int r = it % R, t = it / R;
                if (r0 + r >= n_out) continue;
                float v0 = 0.f;
                for (int pp = 0; pp < P; ++pp) v0 += red[static_cast<size_t>((pp * ngu) * R8 + r) * 8 + t];
                v0 *= gscale;
                float val = v0;
                if (swiglu) {
                    float v1 = 0.f;
                    for (int pp = 0; pp < P; ++pp) v1 += red[static_cast<size_t>((pp * ngu + 1) * R8 + r) * 8 + t];
                    v1 *= gscale;
                    val = (v0 / (1.0f + expf(-v0))) * v1;
                }
                const int o = t * n_out + r0 + r;
                if (resid) val += bf16_bits_to_f32(ldg_cg_u16(a.residual + o));
                chain_store(a, o, val);
            }
        }
        named_barrier_sync(1, kCcThreads);
    }
}

// 3..8 tokens per op (the warp-MMA stage): every op kind (NVFP4 or Q4/Q5,
// any epilogue, with or without the RMSNorm prologue). HAS_NORM: some op has
// the prologue (a list without compiles the plain conversion alone).
template <bool HAS_NORM>
__global__ void __launch_bounds__(kCcAllThreads, 1) chain_mt_kernel(const __grid_constant__ ChainParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCcMaxStages);
    volatile int* any_bf = abort_flag + 1;

    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCcThreads);
        }
        *abort_flag = 0;
        *any_bf = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const uint32_t ring = smem_u32(smem + p.op[0].a.smem_ring);

    if (warp == kCcTmaWarp) {
        chain_producer(p, smem, full, empty, abort_flag, lane);
        return;
    }

    // ---------------------------------------------------------------- compute warps
    // Rows past an op's R in its 16-row blocks hold whatever an earlier op's
    // boxes left in the ring: each D row depends on its own weight row only,
    // and those rows are never written out.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool aborted = false;
    int slot = 0, lap = 0;
    for (int o = 0; o < p.n_ops; ++o) {
        const ChainOp& op = p.op[o];
        MtArgs m;
        m.a = op.a;
        m.M = p.M;
        m.NRB = op.NRB;
        m.W = op.W;
        m.x_tok = op.x_tok;
        if (op.dep) chain_grid_barrier(p, abort_flag);
        if (*abort_flag) aborted = true;
        if (threadIdx.x == 0) *any_bf = 0;
        named_barrier_sync(1, kCcThreads);
        if (HAS_NORM && m.a.norm_w != nullptr) mt_norm_factors<true>(m, smem, warp, lane);
        if (op.fmt == FMT_NVFP4)
            mt_convert_any<false, true, HAS_NORM>(m, smem, warp, lane, any_bf, 0);
        else
            mt_convert_any<true, true, HAS_NORM>(m, smem, warp, lane, any_bf, 0);
        named_barrier_sync(1, kCcThreads);
        const bool mixed = *any_bf != 0 || m.W < m.a.C;
        if (op.fmt == FMT_NVFP4) {
            if (mixed)
                chain_units_mt<0, true, 0, HAS_NORM>(m, op.epi, smem, ring, p.slot_bytes, p.n_stages, full, empty,
                                                     abort_flag, any_bf, aborted, slot, lap, warp, lane);
            else
                chain_units_mt<0, false, 0, HAS_NORM>(m, op.epi, smem, ring, p.slot_bytes, p.n_stages, full, empty,
                                                      abort_flag, any_bf, aborted, slot, lap, warp, lane);
        } else {
            // the gate (or only) matrix's width, and a SwiGLU's up matrix's
            const bool b5 = op.fmt == FMT_Q5;
            const bool u5 = op.epi == EPI_SWIGLU ? op.ufmt == FMT_Q5 : b5;
            // one loop per width pair (the mixed one: its per-stage flag test is
            // cheap, and fewer inlined copies keep the kernel's registers from
            // spilling)
#define QG_CHAIN_MT_Q(B, BU)                                                                                     \
    chain_units_mt<B, true, BU, HAS_NORM>(m, op.epi, smem, ring, p.slot_bytes, p.n_stages, full, empty, abort_flag, \
                                          any_bf, aborted, slot, lap, warp, lane)
            if (b5 && u5)
                QG_CHAIN_MT_Q(5, 5);
            else if (b5)
                QG_CHAIN_MT_Q(5, 4);
            else if (u5)
                QG_CHAIN_MT_Q(4, 5);
            else
                QG_CHAIN_MT_Q(4, 4);
#undef QG_CHAIN_MT_Q
        }
    }
}

constexpr uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

// Units of R rows with the one-token kernels' rule: the smallest number of
// units per CTA whose rows fit 256 per stage, R = ceil(rows / (SMs * units)).
void cc_plan(CcArgs& a, int n_out, int ngu, int K, int sms)
{
    int R = 1;
    for (int U = 1;; ++U) {
        R = (n_out + sms * U - 1) / (sms * U);
        if (ngu * ((R + 7) / 8 * 8) <= 256) break;
    }
    R = std::max(R, 1);
    a.K = K;
    a.C = K / kChunkK;
    a.n_out = n_out;
    a.R = R;
    a.R8 = (R + 7) / 8 * 8;
    a.P = std::max(1, std::min(256 / (ngu * a.R8), a.C));
    a.Cp = (a.C + a.P - 1) / a.P;
    a.n_units = (n_out + R - 1) / R;
}

}  // namespace

// One persistent launch for a list of one- or two-token projections;
// QG_ERR_UNSUPPORTED when the list does not fit its plan (M > 2, K not a
// multiple of 256, too many ops, or shared memory), so that the caller runs
// the ops one by one instead.
namespace {

// The chunked stage layout of op g in both chained plans: per matrix (gate,
// up) one box of the stage's P chunks x R rows for the codes ([chunk][row],
// 128-byte swizzled lines, 1024-aligned), then the scales (then the mins and
// the Q5 plane), and the 3-D tensor maps that load them. box_tx is a whole
// stage; st the bytes the layout uses.
qg_status chain_layout(CcArgs& a, const qg_gemv_op& g, int fmt, int ufmt, int ngu, bool sep_up, CUtensorMap* maps,
                       uint32_t& st)
{
    const uint32_t PR = static_cast<uint32_t>(a.P * a.R), nm = static_cast<uint32_t>(ngu);
    a.code_pitch = align_up(PR * 128u, 1024);
    a.sc_pitch = align_up(PR * 16u, 128);
    a.scales_off = nm * a.code_pitch;
    if (fmt == FMT_NVFP4) {
        st = a.scales_off + nm * a.sc_pitch;
        a.box_tx = nm * PR * (128u + 16u);
    } else {
        const bool any5 = fmt == FMT_Q5 || ufmt == FMT_Q5;
        a.mins_off = align_up(a.scales_off + nm * a.sc_pitch, 1024);
        a.hi_off = align_up(a.mins_off + nm * a.sc_pitch, 1024);
        st = a.hi_off + (any5 ? nm * 2u * a.sc_pitch : 0u);
        a.box_tx = PR * (128u + 16u + 16u + (fmt == FMT_Q5 ? 32u : 0u));
        if (ngu == 2) a.box_tx += PR * (128u + 16u + 16u + (ufmt == FMT_Q5 ? 32u : 0u));
    }
    const uint64_t rows = static_cast<uint64_t>(g.N), C = static_cast<uint64_t>(a.C);
    const uint32_t Rb = static_cast<uint32_t>(a.R), Pb = static_cast<uint32_t>(a.P);
    if (!encode_tmap_chunks(&maps[0], g.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, rows, C, Rb, Pb, true))
        return QG_ERR_CUDA;
    if (fmt == FMT_NVFP4)
        return encode_tmap_chunks(&maps[1], g.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 16, rows, C, Rb, Pb, false)
                   ? QG_OK
                   : QG_ERR_CUDA;
    const void* srcs[2][4] = {{g.codes, g.scales, g.mins, g.q_hi}, {g.up_codes, g.up_scales, g.up_mins, g.up_q_hi}};
    const int fm[2] = {fmt, ufmt};
    for (int gg = 0; gg < (sep_up ? 2 : 1); ++gg) {
        CUtensorMap* mm = &maps[4 * gg];
        if ((gg == 1 &&
             !encode_tmap_chunks(&mm[0], srcs[gg][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, rows, C, Rb, Pb, true)) ||
            !encode_tmap_chunks(&mm[1], srcs[gg][1], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, 8, rows, C, Rb, Pb, false) ||
            !encode_tmap_chunks(&mm[2], srcs[gg][2], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, 8, rows, C, Rb, Pb, false))
            return QG_ERR_CUDA;
        if (fm[gg] == FMT_Q5 &&
            !encode_tmap_chunks(&mm[3], srcs[gg][3], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 32, rows, C, Rb, Pb, false))
            return QG_ERR_CUDA;
    }
    return QG_OK;
}

// 3..8 tokens: every op on the warp-MMA stage (its plan: R for equal bytes per
// SM, boxes padded to 16-row blocks, at most 16 blocks per stage), the
// activations of each op held a window of chunks at a time.
qg_status launch_chain_mt(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, cudaStream_t stream)
{
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    static ChainParams p;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    memset(&p, 0, sizeof(p));
    p.n_ops = n_ops;
    p.M = M;
    bool any_dep = false, any_q = false, any_norm = false;
    uint32_t slot_bytes = 0, red_max = 0;
    int c_max = 0;
    for (int o = 0; o < n_ops; ++o) {
        const qg_gemv_op& g = ops[o];
        if (g.K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
        ChainOp& op = p.op[o];
        op.fmt = g.format == QG_FMT_NVFP4 ? FMT_NVFP4 : g.format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4;
        op.epi = g.epilogue == QG_EPI_SWIGLU ? EPI_SWIGLU : g.epilogue == QG_EPI_RESIDUAL ? EPI_RESID : EPI_NONE;
        op.dep = o > 0 && g.after_previous ? 1 : 0;
        const bool sep_up = g.up_codes != nullptr;
        op.ufmt = sep_up ? (g.up_format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4) : op.fmt;
        any_dep = any_dep || op.dep;
        any_q = any_q || op.fmt != FMT_NVFP4;
        const int ngu = op.epi == EPI_SWIGLU ? 2 : 1;
        const int n_out = op.epi == EPI_SWIGLU && !sep_up ? g.N / 2 : g.N;
        int R = 1;
        for (int U = 1;; ++U) {
            R = (n_out + sms * U - 1) / (sms * U);
            if (ngu * ((R + 15) / 16) <= kCcWarps) break;
        }
        R = std::max(R, 1);
        CcArgs& a = op.a;
        a.x = static_cast<const uint16_t*>(g.x);
        a.y = g.y;
        a.residual = static_cast<const uint16_t*>(g.residual);
        a.norm_w = static_cast<const uint16_t*>(g.norm_weight);
        a.norm_eps = g.norm_eps;
        any_norm = any_norm || g.norm_weight != nullptr;
        c_max = std::max(c_max, g.K / kChunkK);
        a.K = g.K;
        a.C = g.K / kChunkK;
        a.n_out = n_out;
        a.R = R;
        a.R8 = (R + 15) / 16 * 16;
        op.NRB = a.R8 / 16;
        a.P = std::max(1, std::min(kCcWarps / (ngu * op.NRB), a.C));
        a.Cp = (a.C + a.P - 1) / a.P;
        a.n_units = (n_out + R - 1) / R;
        a.up_row_offset = op.epi == EPI_SWIGLU && !sep_up ? n_out : 0;
        a.out_f32 = op.epi == EPI_SWIGLU ? 0 : (g.y_dtype == QG_OUT_F32 ? 1 : 0);
        a.g = op.fmt == FMT_NVFP4 ? g.global_scale : 1.f;
        const uint32_t nbox = static_cast<uint32_t>(a.P * ngu);
        (void)nbox;
        uint32_t st = 0;
        const qg_status ls = chain_layout(a, g, op.fmt, op.ufmt, ngu, g.up_codes != nullptr, p.map[o], st);
        if (ls != QG_OK) return ls;
        // + 2 KB: a thread's or warp's last rows read up to 15 lines past its box
        slot_bytes = std::max(slot_bytes, align_up(st + 2048u, 1024));
        red_max = std::max(red_max, nbox * a.R8 * 8u);
    }
    if (any_dep && !sync) return QG_ERR_INVALID_ARG;
    // shared memory: ring | activation window | 2^-prescale | flags | sums of
    // x per group | partial sums | barriers; each op's window W (a multiple of
    // its P chunks, all of K when it fits) leaves at least three ring slots
    const uint32_t red_bytes = align_up(red_max * 4u, 128);
    const uint32_t bar_bytes = 2 * kCcMaxStages * 8 + 16;
    const uint32_t ss_bytes = any_norm ? align_up(static_cast<uint32_t>(M * (c_max + 1)) * 4u, 16) : 0u;
    auto win_bytes = [&](int W) {
        const uint32_t xt = static_cast<uint32_t>(W) * kChunkK * 2u + 16u;
        return align_up(static_cast<uint32_t>(M) * xt, 128) + align_up(static_cast<uint32_t>(M * W) * 4u, 16) +
               align_up(static_cast<uint32_t>(W), 16) +
               (any_q ? align_up(static_cast<uint32_t>(M * W) * 32u, 16) : 0u);
    };
    const uint32_t other = red_bytes + bar_bytes + ss_bytes;
    if (other + 3 * slot_bytes >= kCcSmemMax) return QG_ERR_UNSUPPORTED;
    const uint32_t budget = kCcSmemMax - other - 4 * slot_bytes > kCcSmemMax
                                ? 0u
                                : kCcSmemMax - other - 4 * slot_bytes;  // all of K beside four slots
    const uint32_t budget3 = kCcSmemMax - other - 3 * slot_bytes;
    uint32_t win_max = 0;
    int w_max = 1;
    for (int o = 0; o < n_ops; ++o) {
        CcArgs& a = p.op[o].a;
        int W = a.C;
        if (win_bytes(W) > budget) {
            W = (a.C / a.P) * a.P;
            while (W > a.P && win_bytes(W) > budget3) W -= a.P;
        }
        if (win_bytes(W) > budget3) return QG_ERR_UNSUPPORTED;
        p.op[o].W = W;
        p.op[o].x_tok = static_cast<uint32_t>(W) * kChunkK * 2u + 16u;
        win_max = std::max(win_max, win_bytes(W));
        w_max = std::max(w_max, W);
    }
    const uint32_t x_bytes = align_up(static_cast<uint32_t>(M) * (static_cast<uint32_t>(w_max) * kChunkK * 2u + 16u),
                                      128);
    const uint32_t pe_bytes = align_up(static_cast<uint32_t>(M * w_max) * 4u, 16);
    const uint32_t fl_bytes = align_up(static_cast<uint32_t>(w_max), 16);
    const uint32_t gx_bytes = any_q ? align_up(static_cast<uint32_t>(M * w_max) * 32u, 16) : 0u;
    const uint32_t fixed = x_bytes + pe_bytes + fl_bytes + gx_bytes + ss_bytes + red_bytes + bar_bytes;
    if (fixed + 3 * slot_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    const int n_stages = std::min<int>(kCcMaxStages, static_cast<int>((kCcSmemMax - fixed) / slot_bytes));
    uint32_t so = 0;
    const uint32_t smem_ring = so;
    so += n_stages * slot_bytes;
    const uint32_t smem_x = so;
    so += x_bytes;
    const uint32_t smem_pe = so;
    so += pe_bytes;
    const uint32_t smem_fl = so;
    so += fl_bytes;
    const uint32_t smem_gx = so;
    so += gx_bytes;
    const uint32_t smem_ss = so;
    so += ss_bytes;
    const uint32_t smem_red = so;
    so += red_bytes;
    const uint32_t smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    (void)win_max;

    int* status = device_status_ptr();
    if (!status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    p.n_stages = n_stages;
    p.slot_bytes = slot_bytes;
    p.smem_bar = smem_bar;
    p.sync = sync;
    p.wait_ns = dbg.wait_ns;
    p.starve = dbg.starve;
    p.status = status;
    for (int o = 0; o < n_ops; ++o) {
        CcArgs& a = p.op[o].a;
        a.n_stages = n_stages;
        a.stage_bytes = slot_bytes;
        a.smem_ring = smem_ring;
        a.smem_x = smem_x;
        a.smem_pe = smem_pe;
        a.smem_fl = smem_fl;
        a.smem_gx = smem_gx;
        a.smem_ss = smem_ss;
        a.smem_red = smem_red;
        a.smem_bar = smem_bar;
        a.wait_ns = dbg.wait_ns;
        a.starve = dbg.starve;
        a.status = status;
    }
    const int kv = any_norm ? 1 : 0;
    auto kern = any_norm ? chain_mt_kernel<true> : chain_mt_kernel<false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[kv][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[kv][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kCcAllThreads);
    cfg.dynamicSmemBytes = so;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (any_dep) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace

qg_status launch_chain(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, cudaStream_t stream)
{
    if (n_ops < 1 || n_ops > kChainMaxOps) return QG_ERR_UNSUPPORTED;
    if (M >= 3 && M <= kMtTokens) return launch_chain_mt(ops, n_ops, M, sync, stream);
    if (M < 1 || M > 2) return QG_ERR_UNSUPPORTED;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    static ChainParams p;  // large: built here, copied into the launch's parameters
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    memset(&p, 0, sizeof(p));
    p.n_ops = n_ops;
    bool any_dep = false;
    uint32_t slot_bytes = 0;
    int c_max = 0, red_max = 0;
    for (int o = 0; o < n_ops; ++o) {
        const qg_gemv_op& g = ops[o];
        if (g.K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
        ChainOp& op = p.op[o];
        op.fmt = g.format == QG_FMT_NVFP4 ? FMT_NVFP4 : g.format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4;
        op.epi = g.epilogue == QG_EPI_SWIGLU ? EPI_SWIGLU : g.epilogue == QG_EPI_RESIDUAL ? EPI_RESID : EPI_NONE;
        op.dep = o > 0 && g.after_previous ? 1 : 0;
        any_dep = any_dep || op.dep;
        const bool sep_up = g.up_codes != nullptr;
        op.ufmt = sep_up ? (g.up_format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4) : op.fmt;
        const int ngu = op.epi == EPI_SWIGLU ? 2 : 1;
        const int n_out = op.epi == EPI_SWIGLU && !sep_up ? g.N / 2 : g.N;
        CcArgs& a = op.a;
        cc_plan(a, n_out, ngu, g.K, sms);
        a.x = static_cast<const uint16_t*>(g.x);
        a.y = g.y;
        a.residual = static_cast<const uint16_t*>(g.residual);
        a.norm_w = static_cast<const uint16_t*>(g.norm_weight);
        a.norm_eps = g.norm_eps;
        a.up_row_offset = op.epi == EPI_SWIGLU ? n_out : 0;
        a.out_f32 = op.epi == EPI_SWIGLU ? 0 : (g.y_dtype == QG_OUT_F32 ? 1 : 0);
        a.g = op.fmt == FMT_NVFP4 ? g.global_scale : 1.f;
        const uint32_t nbox = static_cast<uint32_t>(a.P * ngu);
        (void)nbox;
        uint32_t st = 0;
        const qg_status ls = chain_layout(a, g, op.fmt, op.ufmt, ngu, g.up_codes != nullptr, p.map[o], st);
        if (ls != QG_OK) return ls;
        // + 2 KB: a thread's or warp's last rows read up to 15 lines past its box
        slot_bytes = std::max(slot_bytes, align_up(st + 2048u, 1024));
        c_max = std::max(c_max, a.C);
        red_max = std::max(red_max, static_cast<int>(nbox) * a.R8);
    }
    if (any_dep && !sync) return QG_ERR_INVALID_ARG;
    // shared memory: ring | activations | 2^-prescale | flags | sums of x |
    // sums of squares | partial sums | barriers
    const uint32_t x_bytes = static_cast<uint32_t>(M * c_max) * kChunkK * 2u;
    const uint32_t pe_bytes = align_up(static_cast<uint32_t>(M * c_max) * 4u, 16);
    const uint32_t fl_bytes = align_up(static_cast<uint32_t>(c_max), 16);
    bool any_q = false;
    for (int o = 0; o < n_ops; ++o) any_q = any_q || p.op[o].fmt != FMT_NVFP4;
    const uint32_t gx_bytes = any_q ? align_up(static_cast<uint32_t>(M * c_max * kChainNseg) * 4u, 16) : 0u;
    const uint32_t ss_bytes = align_up(static_cast<uint32_t>(M * c_max) * 4u, 16);
    const uint32_t red_bytes = align_up(static_cast<uint32_t>(M * red_max) * 4u, 128);
    const uint32_t bar_bytes = 2 * kCcMaxStages * 8 + 16;
    const uint32_t fixed = x_bytes + pe_bytes + fl_bytes + gx_bytes + ss_bytes + red_bytes + bar_bytes;
    if (fixed + 3 * slot_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    const int n_stages = std::min<int>(kCcMaxStages, static_cast<int>((kCcSmemMax - fixed) / slot_bytes));
    uint32_t so = 0;
    const uint32_t smem_ring = so;
    so += n_stages * slot_bytes;
    const uint32_t smem_x = so;
    so += x_bytes;
    const uint32_t smem_pe = so;
    so += pe_bytes;
    const uint32_t smem_fl = so;
    so += fl_bytes;
    const uint32_t smem_gx = so;
    so += gx_bytes;
    const uint32_t smem_ss = so;
    so += ss_bytes;
    const uint32_t smem_red = so;
    so += red_bytes;
    const uint32_t smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;

    int* status = device_status_ptr();
    if (!status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    p.n_stages = n_stages;
    p.slot_bytes = slot_bytes;
    p.smem_bar = smem_bar;
    p.sync = sync;
    p.wait_ns = dbg.wait_ns;
    p.starve = dbg.starve;
    p.status = status;
    for (int o = 0; o < n_ops; ++o) {
        CcArgs& a = p.op[o].a;
        a.n_stages = n_stages;
        a.stage_bytes = slot_bytes;
        a.smem_ring = smem_ring;
        a.smem_x = smem_x;
        a.smem_ss = smem_ss;
        a.smem_pe = smem_pe;
        a.smem_fl = smem_fl;
        a.smem_gx = smem_gx;
        a.smem_red = smem_red;
        a.smem_bar = smem_bar;
        a.wait_ns = dbg.wait_ns;
        a.starve = dbg.starve;
        a.status = status;
    }

    auto kern = M == 2 ? chain_kernel<2> : chain_kernel<1>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[M - 1][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[M - 1][dev] = true;
    }
    // Every CTA must be resident for the grid-wide barrier: one CTA per SM
    // (the shared memory allows no more), launched cooperatively when an op
    // waits at the barrier; otherwise with programmatic dependent launch.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kCcAllThreads);
    cfg.dynamicSmemBytes = so;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (any_dep) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
