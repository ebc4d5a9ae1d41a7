// moe_cc.cu -- the MoE expert FFN's two grouped projections (gate/up with
// SwiGLU, then down) on the CUDA cores.
//
// What is computed is moe_qgemv_nvfp4's definition (NInfer article, section
// 2: the fused NVFP4 GEMV with SwiGLU; Decapybara README, "Blackwell CUDA
// 内核套件": moe.cu). With top-8 routing over ~128 experts, eight decode
// tokens give about 1.2 tokens per active expert: a tensor-core tile with 8
// token columns would be mostly padding, and each weight feeds one or two dot
// products. So each active expert's rows stream through the one- and
// two-token CUDA-core stage code of qgemv_cc.cu (exact decoded weights,
// exactly prescaled f16 activations, fp32 sums in a fixed order):
//
//   * a pass is a unit of R rows of one expert together with one or two of
//     its tokens; an expert with more tokens gets one pass per token pair,
//     adjacent in the list, so the repeated rows come from L2, not HBM;
//   * one CTA per SM takes passes b, b + G, b + 2G, ... of the list the
//     grouping kernel wrote (G = grid size); its TMA warp streams the passes'
//     weight stages into one shared-memory ring, as in the standalone
//     kernel, without a stop between passes;
//   * before its first pass, the CTA converts only the activation rows its
//     passes read (the M token rows for gate/up, at most two h rows per pass
//     for down) into shared memory, once;
//   * a pass is short (K is 2048 or 768), so its end costs the compute warps
//     no barrier: each 8-lane segment group reduce-scatters its partial sums
//     into one of two buffers, and an epilogue warp sums the phases, applies
//     the expert's global scale and SwiGLU, and writes the tokens' output
//     rows (h for gate/up, fp32 slot rows for down) while the compute warps
//     go on with the next pass.
// A chunk that one token cannot carry exactly in f16 stays raw bf16 for that
// token (a per-row flag); a two-token stage whose tokens disagree runs each
// token on its own arithmetic, so every token gets the exact products either
// way.
#include <algorithm>
#include <cstring>

#include "cc_core.cuh"

namespace qg {

namespace {

constexpr int kMoeNseg = 8;       // 32-k segments
constexpr int kMoeMaxLocal = 32;  // passes one CTA's tables hold
// warps 0-15 compute, warp 16 streams the weights (kCcTmaWarp), warp 17 runs
// the passes' epilogues
constexpr int kMoeEpiWarp = kCcWarps + 1;
constexpr int kMoeThreads = 32 * (kMoeEpiWarp + 1);
constexpr uint32_t kMoeBarBytes = (2 * kCcMaxStages + 4) * 8 + 16;

// One pass: a unit of R rows of one expert with one or two of its tokens.
struct CcPass {
    int w_row0;      // first weight row (gate row for SwiGLU)
    int out_col0;    // first output column
    int e;           // expert id
    int ntok;        // 1 or 2
    int x_row[2];    // activation rows
    int out_row[2];  // output rows
};

struct MoeCcArgs {
    CcArgs a;                 // the unit plan (R, R8, P, Cp, C, K), ring and shared-memory offsets, waits
    const CcPair* pairs;      // pair groups, written by the grouping kernel
    const int* n_pairs;       // their device count
    int blocks;               // row blocks per expert: passes = pairs * blocks
    int expert_rows;          // weight rows per expert (gate and up rows both)
    const float* gscales;     // per-expert global scale
    int out_pitch;            // values per output row
    int max_local;            // passes per CTA the tables were sized for
    int max_rows;             // local activation rows they were sized for
    // CcPass sp[max_local] | float sg[max_local] | int ltab[max_rows] |
    // uint8 lx[2 * max_local] | int n_rows
    uint32_t smem_tab;
};

static_assert(sizeof(CcPass) == 32, "a pass descriptor is eight ints");

// Converts the CTA's local activation rows (global row ltab[j] -> local j)
// into shared memory: chunk kc of local row j at item j * C + kc, laid out as
// cc_convert lays out one token's chunk (f16 after the exact prescale, or raw
// bf16 with its flag set), with the factor pe[item] = 2^-prescale.
__device__ void moe_convert_rows(const MoeCcArgs& m, uint8_t* smem, const int* ltab, int n_rows, int warp, int lane)
{
    const CcArgs& a = m.a;
    constexpr int PPS = kChunkK / kMoeNseg / 8;  // 16-byte pieces per segment
    constexpr int B = 4;                         // chunk loads in flight per warp
    uint32_t* xs = reinterpret_cast<uint32_t*>(smem + a.smem_x);
    float* pe = reinterpret_cast<float*>(smem + a.smem_pe);
    uint8_t* fl = smem + a.smem_fl;
    const int items = n_rows * a.C;
    for (int base = warp; base < items; base += kCcWarps * B) {
        uint4 raw[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = base + u * kCcWarps;
            raw[u] = it < items ? ldg_nc_128(a.x + static_cast<size_t>(ltab[it / a.C]) * a.K +
                                             static_cast<size_t>(it % a.C) * kChunkK + lane * 8)
                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = base + u * kCcWarps;
            if (it >= items) break;
            const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
            uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < 4; ++i) bf16_range_acc(wv[i], mx2, mn2);
            uint32_t emax, emin, magmax;
            bf16_range_fin(mx2, mn2, emax, emin, magmax);
            emax = __reduce_max_sync(0xffffffffu, emax);
            emin = __reduce_min_sync(0xffffffffu, emin);
            if (emax == 0u) magmax = __reduce_max_sync(0xffffffffu, magmax);
            const int e = min(emax != 0u ? 141 - static_cast<int>(emax) : prescale_exponent(magmax), 126);
            const bool inexact = emin != 255u && static_cast<int>(emin) - 127 + e < -17;
            uint32_t o[4];
            if (inexact) {
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] = wv[i];
            } else {
                const float sc = __int_as_float((127 + e) << 23);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = pack_f16x2(__uint_as_float(wv[i] << 16) * sc, __uint_as_float(wv[i] & 0xFFFF0000u) * sc);
            }
            const int off = (lane % PPS) * kMoeNseg * 4 + (lane / PPS) * 4;  // in 4-byte words
            *reinterpret_cast<uint4*>(xs + it * (kChunkK / 2) + off) = make_uint4(o[0], o[1], o[2], o[3]);
            if (lane == 0) {
                pe[it] = inexact ? 1.0f : __int_as_float((127 - e) << 23);
                fl[it] = inexact ? 1 : 0;
            }
        }
    }
}

// Sums v[0..7] over the 8 lanes of a segment group (seg = lane % 8) and
// leaves total j on the lane whose seg is j: three halving exchanges, the
// additions in a fixed order.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int seg)
{
    const bool h4 = (seg & 4) != 0, h2 = (seg & 2) != 0, h1 = (seg & 1) != 0;
    float a4[4], a2[2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = h4 ? v[k] : v[k + 4];
        a4[k] = (h4 ? v[k + 4] : v[k]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = h2 ? a4[k] : a4[k + 2];
        a2[k] = (h2 ? a4[k + 2] : a4[k]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float send = h1 ? a2[0] : a2[1];
    return (h1 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
}

// One token of one stage on its own arithmetic: its sums acc[i * 2 + t].
template <bool BF>
__device__ __forceinline__ void moe_stage_one(const CcGeom& geom, uint32_t stage, int b2, int row0, int seg,
                                              uint32_t xc, float pe, int t, float (&acc)[kCcRows * 2])
{
    constexpr int KS = kChunkK / kMoeNseg;
    uint32_t xw[KS / 2];
#pragma unroll
    for (int i = 0; i < KS / 8; ++i) {
        const uint4 v = lds128(xc + i * kMoeNseg * 16);
        xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
    }
    float a1[kCcRows];
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) a1[i] = acc[i * 2 + t];
    cc_stage<kMoeNseg, BF>(geom, stage, b2, row0, seg, xw, pe, a1);
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) acc[i * 2 + t] = a1[i];
}

template <int EPI>
__global__ void __launch_bounds__(kMoeThreads, 1)
    moe_cc_kernel(const __grid_constant__ MoeCcArgs m, const __grid_constant__ CUtensorMap tm_codes,
                  const __grid_constant__ CUtensorMap tm_scales)
{
    constexpr int NGU = EPI == EPI_SWIGLU ? 2 : 1;
    constexpr int NSEG = kMoeNseg;
    const CcArgs& a = m.a;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kCcMaxStages;
    uint64_t* rfull = empty + kCcMaxStages;  // partial sums of pass i in buffer i % 2 are written
    uint64_t* rempty = rfull + 2;            // ... and have been read by the epilogue warp
    volatile int* abort_flag = reinterpret_cast<volatile int*>(rempty + 2);
    CcPass* sp = reinterpret_cast<CcPass*>(smem + m.smem_tab);
    float* sg = reinterpret_cast<float*>(sp + m.max_local);
    int* ltab = reinterpret_cast<int*>(sg + m.max_local);
    uint8_t* lx = reinterpret_cast<uint8_t*>(ltab + m.max_rows);
    volatile int* n_rows_s = reinterpret_cast<volatile int*>(lx + (2 * m.max_local + 3) / 4 * 4);

    // compute threads that own rows ((phase, gate/up) boxes x row groups x
    // segments), rounded up to whole warps; the others only help convert the
    // activations
    const int n_act = (a.P * NGU * ((a.R + kCcRows - 1) / kCcRows) * NSEG + 31) / 32 * 32;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_act);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&rfull[b], n_act);
            mbar_init(&rempty[b], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // The pass list (and the activations) come from earlier kernels.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int G = gridDim.x;
    const int n_passes = *m.n_pairs * m.blocks;
    const int n_local = n_passes > static_cast<int>(blockIdx.x) ? (n_passes - blockIdx.x + G - 1) / G : 0;
    if (n_local > m.max_local) {  // more passes than the list can hold: not produced by the grouping kernel
        if (threadIdx.x == 0) set_device_status(a.status, QG_ERR_INVALID_ARG);
        return;
    }
    // this CTA's pass descriptors, built once (reading them per pass would
    // stall the producer and the epilogue on global latency)
    for (int k = threadIdx.x; k < n_local; k += blockDim.x) {
        const int v = blockIdx.x + k * G;
        const int gi = v / m.blocks, rb = v - gi * m.blocks;
        const CcPair pr = m.pairs[gi];
        CcPass ps;
        ps.w_row0 = pr.e * m.expert_rows + rb * a.R;
        ps.out_col0 = rb * a.R;
        ps.e = pr.e;
        ps.ntok = pr.ntok;
        ps.x_row[0] = pr.x_row[0];
        ps.x_row[1] = pr.x_row[1];
        ps.out_row[0] = pr.out_row[0];
        ps.out_row[1] = pr.out_row[1];
        sp[k] = ps;
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
        // the plan in registers (a parameter read after each copy's memory
        // clobber would be repeated every stage)
        const int P = a.P, Cp = a.Cp, up_off = a.up_row_offset, n_stages = a.n_stages, starve = a.starve;
        const uint32_t code_pitch = a.code_pitch, sc_pitch = a.sc_pitch, scales_off = a.scales_off;
        const uint32_t box_tx = a.box_tx, stage_bytes = a.stage_bytes, smem_ring = a.smem_ring;
        for (int i = 0; i < n_local && !stop; ++i) {
            const int w_row0 = sp[i].w_row0;
            for (int c = 0; c < Cp; ++c) {
                if (lap > 0 && !cc_wait_warp(&empty[slot], (lap - 1) & 1, a, abort_flag)) {
                    stop = true;
                    break;
                }
                if (*abort_flag || starve) {
                    stop = true;
                    break;
                }
                uint8_t* sb = smem + smem_ring + slot * stage_bytes;
                if (elect_one()) {
                    // per matrix (gate, up) one box of the stage's P chunks x R
                    // rows (chunks past K are filled with zeros and counted)
                    mbar_arrive_expect_tx(&full[slot], box_tx);
#pragma unroll
                    for (int gg = 0; gg < NGU; ++gg) {
                        const int row = w_row0 + gg * up_off;
                        tma_load_3d(sb + gg * code_pitch, &tm_codes, 0, row, c * P, &full[slot]);
                        tma_load_3d(sb + scales_off + gg * sc_pitch, &tm_scales, 0, row, c * P, &full[slot]);
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == n_stages) {
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

    const uint32_t red_stride = static_cast<uint32_t>(a.P * NGU * a.R8 * 2);  // floats per buffer
    float* red = reinterpret_cast<float*>(smem + a.smem_red);

    if (warp == kMoeEpiWarp) {
        // ------------------------------------------------------------ epilogue
        // pass i: sum the phases' partial sums in order, apply the expert's
        // global scale (and SwiGLU), round once, write the tokens' rows
        for (int k = lane; k < n_local; k += 32) sg[k] = m.gscales[sp[k].e];
        __syncwarp();
        bool aborted = false;
        for (int i = 0; i < n_local; ++i) {
            const int buf = i & 1;
            if (!aborted && !cc_wait_warp(&rfull[buf], (i >> 1) & 1, a, abort_flag)) aborted = true;
            if (!aborted && !*abort_flag) {
                const CcPass& ps = sp[i];
                const float g = sg[i];
                const float* rb = red + buf * red_stride;
                for (int r = lane; r < a.R; r += 32) {
                    for (int t = 0; t < ps.ntok; ++t) {
                        float v[NGU];
#pragma unroll
                        for (int gg = 0; gg < NGU; ++gg) {
                            float s = 0.f;
                            for (int pp = 0; pp < a.P; ++pp) s += rb[((pp * NGU + gg) * a.R8 + r) * 2 + t];
                            v[gg] = s * g;
                        }
                        float val = v[0];
                        if (EPI == EPI_SWIGLU) val = (val / (1.0f + expf(-val))) * v[NGU - 1];
                        const size_t o = static_cast<size_t>(ps.out_row[t]) * m.out_pitch + ps.out_col0 + r;
                        if (a.out_f32)
                            reinterpret_cast<float*>(a.y)[o] = val;
                        else
                            reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(val);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[buf]);
        }
        return;
    }

    // ---------------------------------------------------------------- compute warps
    // the distinct activation rows of this CTA's passes, in first-use order
    if (threadIdx.x == 0) {
        int n = 0;
        for (int i = 0; i < n_local; ++i) {
            const CcPass& ps = sp[i];
            for (int t = 0; t < 2; ++t) {
                if (t >= ps.ntok) {
                    lx[2 * i + t] = lx[2 * i];
                    continue;
                }
                const int gr = ps.x_row[t];
                int j = 0;
                while (j < n && ltab[j] != gr) ++j;
                if (j == n) ltab[n++] = gr;
                lx[2 * i + t] = static_cast<uint8_t>(j);
            }
        }
        *n_rows_s = n;
    }
    named_barrier_sync(1, kCcThreads);
    moe_convert_rows(m, smem, ltab, *n_rows_s, warp, lane);
    named_barrier_sync(1, kCcThreads);
    if (static_cast<int>(threadIdx.x) >= n_act) return;  // no rows: not waiting on every stage

    const CcGeom geom = cc_geom_chunked(a, NGU == 2 ? 1 : 0);
    const int rg_per_box = (a.R + kCcRows - 1) / kCcRows;
    const int seg = threadIdx.x % NSEG;
    const int bg = threadIdx.x / NSEG;
    const int b2 = bg / rg_per_box;
    const int row0 = (bg % rg_per_box) * kCcRows;
    const bool active = b2 < a.P * NGU;
    const int p = active ? b2 / NGU : 0;
    const int n_mine = active ? max(0, (a.C - p + a.P - 1) / a.P) : 0;
    const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
    const uint8_t* fl = smem + a.smem_fl;
    const uint32_t ring = smem_u32(smem + a.smem_ring);
    const uint32_t x0 = smem_u32(smem + a.smem_x) + static_cast<uint32_t>(p * (kChunkK / 2) + seg * 4) * 4u;
    const uint32_t x_step = static_cast<uint32_t>(a.P) * (kChunkK * 2u);
    const uint32_t x_row = static_cast<uint32_t>(a.C) * (kChunkK * 2u);  // bytes per local row

    bool aborted = false;
    int slot = 0, lap = 0;
    for (int i = 0; i < n_local; ++i) {
        const CcPass& ps = sp[i];
        const int ntok = ps.ntok;
        const int l0 = lx[2 * i], l1 = lx[2 * i + 1];
        float acc[kCcRows * 2];
#pragma unroll
        for (int k = 0; k < kCcRows * 2; ++k) acc[k] = 0.f;
        for (int c = 0; c < a.Cp; ++c) {
            if (!aborted && !cc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
            if (!aborted && c < n_mine) {
                const int kc = c * a.P + p;
                const uint32_t stage = ring + slot * a.stage_bytes;
                const uint32_t xc0 = x0 + static_cast<uint32_t>(l0) * x_row + static_cast<uint32_t>(c) * x_step;
                const int i0 = l0 * a.C + kc;
                const bool f0 = fl[i0] != 0;
                if (ntok == 1) {
                    if (f0)
                        moe_stage_one<true>(geom, stage, b2, row0, seg, xc0, pe_all[i0], 0, acc);
                    else
                        moe_stage_one<false>(geom, stage, b2, row0, seg, xc0, pe_all[i0], 0, acc);
                } else {
                    const int i1 = l1 * a.C + kc;
                    const bool f1 = fl[i1] != 0;
                    // the second token's pieces sit (l1 - l0) rows away (modulo 2^32)
                    const uint32_t x_tok = static_cast<uint32_t>(l1 - l0) * x_row;
                    if (f0 == f1) {
                        const float pe2[2] = {pe_all[i0], pe_all[i1]};
                        if (f0)
                            cc_stage_mt<NSEG, true, 2>(geom, stage, b2, row0, seg, xc0, x_tok, pe2, acc);
                        else
                            cc_stage_mt<NSEG, false, 2>(geom, stage, b2, row0, seg, xc0, x_tok, pe2, acc);
                    } else {
                        if (f0)
                            moe_stage_one<true>(geom, stage, b2, row0, seg, xc0, pe_all[i0], 0, acc);
                        else
                            moe_stage_one<false>(geom, stage, b2, row0, seg, xc0, pe_all[i0], 0, acc);
                        if (f1)
                            moe_stage_one<true>(geom, stage, b2, row0, seg, xc0 + x_tok, pe_all[i1], 1, acc);
                        else
                            moe_stage_one<false>(geom, stage, b2, row0, seg, xc0 + x_tok, pe_all[i1], 1, acc);
                    }
                }
            }
            mbar_arrive(&empty[slot]);
            if (++slot == a.n_stages) {
                slot = 0;
                ++lap;
            }
        }

        // the sums over the segment lanes (lane seg keeps row seg / 2, token
        // seg % 2) into partial-sum buffer i % 2, once the epilogue warp has
        // read that buffer's previous pass
        const float v = reduce_scatter8(acc, seg);
        const int buf = i & 1;
        if (i >= 2 && !aborted && !cc_wait_warp(&rempty[buf], ((i >> 1) - 1) & 1, a, abort_flag)) aborted = true;
        if (active) red[buf * red_stride + (b2 * a.R8 + row0 + (seg >> 1)) * 2 + (seg & 1)] = v;
        mbar_arrive(&rfull[buf]);
    }
}

constexpr uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

}  // namespace

// The grouped projection over at most max_pairs pair groups, each over
// `blocks` row blocks of R rows; QG_ERR_UNSUPPORTED when the shapes or shared
// memory do not fit the plan (the caller then takes the tcgen05 grouped
// kernel). With launch == false it only answers whether the plan fits.
qg_status launch_cc_moe(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu, int up_offset,
                        int expert_rows, int blocks, const void* x, int n_x_rows, void* y, int out_pitch, int out_f32,
                        const CcPair* pairs, const int* n_pairs, int max_pairs, const float* gscales, int R,
                        cudaStream_t stream, bool launch)
{
    if (K % kChunkK != 0 || R % 8 != 0 || R < 8 || max_pairs < 0 || blocks < 1) return QG_ERR_UNSUPPORTED;
    const int max_passes = max_pairs * blocks;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    const int G = sms;
    const int max_local = std::max(1, (max_passes + G - 1) / G);
    if (max_local > kMoeMaxLocal) return QG_ERR_UNSUPPORTED;
    const int max_rows = std::max(1, std::min(n_x_rows, 2 * max_local));
    const int ngu = swiglu ? 2 : 1;
    if (ngu * R > 256) return QG_ERR_UNSUPPORTED;

    MoeCcArgs m{};
    CcArgs& a = m.a;
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.K = K;
    a.C = K / kChunkK;
    a.R = R;
    a.R8 = R;
    a.P = std::max(1, std::min(256 / (ngu * a.R8), a.C));
    a.Cp = (a.C + a.P - 1) / a.P;
    a.up_row_offset = swiglu ? up_offset : 0;
    a.out_f32 = out_f32;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;
    m.pairs = pairs;
    m.n_pairs = n_pairs;
    m.blocks = blocks;
    m.expert_rows = expert_rows;
    m.gscales = gscales;
    m.out_pitch = out_pitch;
    m.max_local = max_local;
    m.max_rows = max_rows;

    // the chunked stage layout: per matrix one [chunk][row] box of P chunks x
    // R rows (codes: 128-byte swizzled lines), then the scales
    const uint32_t nbox = static_cast<uint32_t>(a.P * ngu);
    const uint32_t PR = static_cast<uint32_t>(a.P * a.R);
    a.code_pitch = align_up(PR * 128u, 1024);
    a.sc_pitch = align_up(PR * 16u, 128);
    a.scales_off = static_cast<uint32_t>(ngu) * a.code_pitch;
    a.stage_bytes = align_up(a.scales_off + static_cast<uint32_t>(ngu) * a.sc_pitch, 1024);
    a.box_tx = static_cast<uint32_t>(ngu) * PR * (128u + 16u);
    const uint32_t items = static_cast<uint32_t>(max_rows * a.C);
    const uint32_t x_bytes = items * kChunkK * 2u;
    const uint32_t pe_bytes = align_up(items * 4u, 16);
    const uint32_t fl_bytes = align_up(items, 16);
    const uint32_t tab_bytes = align_up(static_cast<uint32_t>(max_local) * (32u + 4u) +
                                            static_cast<uint32_t>(max_rows) * 4u +
                                            align_up(2u * static_cast<uint32_t>(max_local), 4) + 4u, 16);
    const uint32_t red_bytes = align_up(2u * nbox * a.R8 * 4u * 2u, 128);  // two buffers, two tokens
    const uint32_t bar_bytes = kMoeBarBytes;
    const uint32_t fixed = x_bytes + pe_bytes + fl_bytes + tab_bytes + red_bytes + bar_bytes;
    if (fixed + 2 * a.stage_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
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
    m.smem_tab = so;
    so += tab_bytes;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    so += bar_bytes;
    if (so > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    if (!launch) return QG_OK;

    CUtensorMap tmc, tms;
    memset(&tmc, 0, sizeof(tmc));
    memset(&tms, 0, sizeof(tms));
    if (!encode_tmap_chunks(&tmc, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, total_rows, a.C, R, a.P, true) ||
        !encode_tmap_chunks(&tms, scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 16, total_rows, a.C, R, a.P, false))
        return QG_ERR_CUDA;

    auto kern = swiglu ? moe_cc_kernel<EPI_SWIGLU> : moe_cc_kernel<EPI_NONE>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[swiglu ? 1 : 0][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[swiglu ? 1 : 0][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kMoeThreads);
    cfg.dynamicSmemBytes = so;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, m, tmc, tms) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
