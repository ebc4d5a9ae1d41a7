// qgemv_chain_ws.cu -- a decode layer's projections at three to eight tokens
// in one persistent launch, with every op's activations converted once per
// call into a caller-provided workspace and streamed into the weight ring.
//
// What is computed is qgemv_chain.cu's (and so the single-projection
// calls'): NVFP4 (NVIDIA NVFP4 blog, "How NVFP4 works") or groupwise-int
// Q4/Q5 (NInfer article, section 2) weights decoded exactly, the warp-level
// MMA stage of qgemv_mt.cu, fixed-order sums and the same epilogues. Only
// where the activations come from differs.
//
// Why: with the activations converted per CTA (qgemv_chain.cu), every one of
// the 152 CTAs repeats the same exact f16 prescale of all M x K activations
// of every op, and an op whose activations do not fit shared memory beside
// the ring converts them again window by window. Timestamps taken inside that
// kernel on a GB300 (a dense 27B-class layer, eight tokens) put about a third
// of the layer in those conversions. Here:
//   * a small kernel converts each op's activations once: one warp per 256-k
//     chunk, all M tokens, into a block of the workspace (the tokens' 256
//     values, f16 after the exact prescale or raw bf16, 576 bytes apart;
//     then the tokens' 2^-prescale, the chunk's bf16 flag and, groupwise
//     int, the sums of each group of 32 values). Launched before the layer
//     kernel with programmatic stream serialisation, so the layer kernel's
//     weight stream starts while it runs.
//   * the layer kernel's TMA warp copies, beside each weight stage, the
//     blocks of the stage's chunks (cp.async.bulk) into a second, shallower
//     ring: no activation window, no per-op conversion, no stop at an op
//     boundary. The weight ring keeps the depth that HBM latency needs (the
//     blocks come from L2 and need less); a stage is ready when both its
//     weights and its blocks have landed.
//   * an op that reads an earlier op's output (after_previous) is converted
//     inside the layer kernel after the grid-wide barrier, one chunk per
//     warp over the whole grid, then a second barrier; the TMA warp copies
//     its blocks once a shared-memory flag says they are written. (With the
//     RMSNorm prologue such an op is left to qgemv_chain.cu.)
// The conversion itself is mt_convert's arithmetic, step for step, so the
// results are identical to the single-projection calls'.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "mt_core.cuh"

namespace qg {

namespace {

constexpr int kWsMaxOps = 8;
constexpr uint32_t kWsTokStride = 576;  // bytes between tokens in a block (512 + 64: no bank conflict)
constexpr uint32_t kWsTrailNv = 48;     // 2^-prescale x 8, bf16 flag, pad
constexpr uint32_t kWsTrailQ = 48 + 256;  // + sums of the 8 groups of 32, x 8 tokens
constexpr int kWsMaxXStages = 4;        // activation ring slots at most
constexpr int kWsMaxPhases = 5;         // chunks per stage (each brings M x 576 bytes of activations)

struct WsOp {
    CcArgs a;         // the op's plan (16-row blocks), as qgemv_chain.cu's 3..8-token path
    int fmt;          // FMT_NVFP4, FMT_Q4, FMT_Q5 (the gate matrix of a SwiGLU)
    int epi;
    int dep;          // converted inside the layer kernel, after a grid-wide barrier
    int ufmt;         // groupwise-int SwiGLU: the up matrix's format
    int NRB;          // 16-row blocks per box
    uint32_t blk;     // bytes of one chunk's block
    uint32_t code_pitch;  // stage bytes between the gate and up matrices' code boxes (1024-aligned)
    uint32_t sc_pitch;    // the same for scales and mins (128-aligned; the Q5 plane: twice)
    size_t ws_off;    // workspace offset of the op's C blocks
};

struct WsParams {
    CUtensorMap map[kWsMaxOps][8];  // as qgemv_chain.cu's
    WsOp op[kWsMaxOps];
    int n_ops;
    int M;
    int n_stages;          // weight ring slots (at offset 0)
    int n_xstages;         // activation ring slots
    uint32_t slot_bytes;
    uint32_t xslot_bytes;
    uint32_t smem_xring;
    uint32_t smem_red;
    uint32_t smem_bar;
    uint8_t* ws;
    uint32_t* sync;
    uint64_t wait_ns;
    int starve;
    int* status;
};

// One warp: chunk kc of an op's activations, all M tokens, into its block
// (layout above). The arithmetic is mt_convert's (exponents from the
// bf16 range, one flag for all tokens when some token's chunk does not fit
// f16 exactly, group sums from the bf16 values, the paired order for the
// groupwise-int MMA). NORM: h = bf16(x * r * gamma) with r per token in rn.
template <bool Q, bool CG, bool NORM>
__device__ __forceinline__ void ws_convert_chunk(const uint16_t* x, int K, int M, int kc, const uint16_t* gamma,
                                                 const float* rn, uint8_t* blk, int lane)
{
    uint4 raw[kMtTokens];
#pragma unroll
    for (int t = 0; t < kMtTokens; ++t)
        raw[t] = t < M ? ldg_128<CG>(x + static_cast<size_t>(t) * K + static_cast<size_t>(kc) * kChunkK + lane * 8)
                       : make_uint4(0, 0, 0, 0);
    if constexpr (NORM) {
        const uint4 gam = ldg_nc_128(gamma + static_cast<size_t>(kc) * kChunkK + lane * 8);
#pragma unroll
        for (int t = 0; t < kMtTokens; ++t)
            if (t < M) raw[t] = rms_apply8(raw[t], gam, rn[t]);
    }
    int e[kMtTokens];
    bool inexact = false;
#pragma unroll
    for (int t = 0; t < kMtTokens; ++t) {
        e[t] = 0;
        if (t >= M) continue;
        const uint32_t wv[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
        uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < 4; ++i) bf16_range_acc(wv[i], mx2, mn2);
        uint32_t emax, emin, magmax;
        bf16_range_fin(mx2, mn2, emax, emin, magmax);
        emax = __reduce_max_sync(0xffffffffu, emax);
        emin = __reduce_min_sync(0xffffffffu, emin);
        if (emax == 0u) magmax = __reduce_max_sync(0xffffffffu, magmax);
        e[t] = min(emax != 0u ? 141 - static_cast<int>(emax) : prescale_exponent(magmax), 126);
        inexact = inexact || (emin != 255u && static_cast<int>(emin) - 127 + e[t] < -17);
    }
    const uint32_t trail = static_cast<uint32_t>(M) * kWsTokStride;
    float* pe = reinterpret_cast<float*>(blk + trail);
    float* gx = reinterpret_cast<float*>(blk + trail + 48);
#pragma unroll
    for (int t = 0; t < kMtTokens; ++t) {
        if (t >= M) continue;
        const uint32_t wv[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
        uint32_t o[4];
        if (inexact) {
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = wv[i];
        } else {
            const float sc = __int_as_float((127 + e[t]) << 23);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = pack_f16x2(__uint_as_float(wv[i] << 16) * sc, __uint_as_float(wv[i] & 0xFFFF0000u) * sc);
        }
        if constexpr (Q) {
            float sx = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                sx += bf16_bits_to_f32((i & 1) ? (wv[i >> 1] >> 16) : (wv[i >> 1] & 0xFFFFu));
            sx += __shfl_xor_sync(0xffffffffu, sx, 1);
            sx += __shfl_xor_sync(0xffffffffu, sx, 2);
            if ((lane & 3) == 0) gx[t * 8 + (lane >> 2)] = sx;
            const uint32_t p0 = __byte_perm(o[0], o[2], 0x5410), p1 = __byte_perm(o[0], o[2], 0x7632);
            const uint32_t p2 = __byte_perm(o[1], o[3], 0x5410), p3 = __byte_perm(o[1], o[3], 0x7632);
            o[0] = p0;
            o[1] = p1;
            o[2] = p2;
            o[3] = p3;
        }
        *reinterpret_cast<uint4*>(blk + t * kWsTokStride + lane * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        if (lane == 0) pe[t] = inexact ? 1.0f : __int_as_float((127 - e[t]) << 23);
    }
    if (lane == 0) *reinterpret_cast<uint32_t*>(blk + trail + 32) = inexact ? 1u : 0u;
}

// The ops without after_previous: blockIdx.y is the op, blockIdx.x the
// chunk, warp t token t (one load round per warp, so the kernel is one
// memory latency long). The tokens agree on the chunk's bf16 flag through
// shared memory; every other step is ws_convert_chunk's, per token, so the
// blocks are the same. With the RMSNorm prologue warp t first takes its
// token's r over all of K in the canonical order (chunk sums of squares,
// added in k order).
__global__ void __launch_bounds__(32 * kMtTokens) chain_ws_convert_kernel(const __grid_constant__ WsParams p)
{
    __shared__ int s_inexact;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const WsOp& op = p.op[blockIdx.y];
    const CcArgs& a = op.a;
    const int t = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kc = blockIdx.x;
    if (op.dep || kc >= a.C) return;
    const int M = p.M, K = a.K;
    const bool tok = t < M;
    if (threadIdx.x == 0) s_inexact = 0;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (tok) raw = ldg_nc_128(a.x + static_cast<size_t>(t) * K + static_cast<size_t>(kc) * kChunkK + lane * 8);
    if (tok && a.norm_w != nullptr) {
        float ss = 0.f;
        constexpr int U = 8;
        for (int c0 = 0; c0 < a.C; c0 += U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                v[u] = c0 + u < a.C ? ldg_nc_128(a.x + static_cast<size_t>(t) * K +
                                                 static_cast<size_t>(c0 + u) * kChunkK + lane * 8)
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + u < a.C) ss += rms_chunk_ss(v[u]);
        }
        const uint4 gam = ldg_nc_128(a.norm_w + static_cast<size_t>(kc) * kChunkK + lane * 8);
        raw = rms_apply8(raw, gam, rms_factor(ss, K, a.norm_eps));
    }
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
    int e = 0;
    bool inexact = false;
    if (tok) {
        uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < 4; ++i) bf16_range_acc(wv[i], mx2, mn2);
        uint32_t emax, emin, magmax;
        bf16_range_fin(mx2, mn2, emax, emin, magmax);
        emax = __reduce_max_sync(0xffffffffu, emax);
        emin = __reduce_min_sync(0xffffffffu, emin);
        if (emax == 0u) magmax = __reduce_max_sync(0xffffffffu, magmax);
        e = min(emax != 0u ? 141 - static_cast<int>(emax) : prescale_exponent(magmax), 126);
        inexact = emin != 255u && static_cast<int>(emin) - 127 + e < -17;
    }
    __syncthreads();
    if (inexact && lane == 0) atomicOr(&s_inexact, 1);
    __syncthreads();
    inexact = s_inexact != 0;
    uint8_t* blk = p.ws + op.ws_off + static_cast<size_t>(kc) * op.blk;
    const uint32_t trail = static_cast<uint32_t>(M) * kWsTokStride;
    if (t == 0 && lane == 0) *reinterpret_cast<uint32_t*>(blk + trail + 32) = inexact ? 1u : 0u;
    if (!tok) return;
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
    if (op.fmt != FMT_NVFP4) {
        float sx = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) sx += bf16_bits_to_f32((i & 1) ? (wv[i >> 1] >> 16) : (wv[i >> 1] & 0xFFFFu));
        sx += __shfl_xor_sync(0xffffffffu, sx, 1);
        sx += __shfl_xor_sync(0xffffffffu, sx, 2);
        if ((lane & 3) == 0) reinterpret_cast<float*>(blk + trail + 48)[t * 8 + (lane >> 2)] = sx;
        const uint32_t p0 = __byte_perm(o[0], o[2], 0x5410), p1 = __byte_perm(o[0], o[2], 0x7632);
        const uint32_t p2 = __byte_perm(o[1], o[3], 0x5410), p3 = __byte_perm(o[1], o[3], 0x7632);
        o[0] = p0;
        o[1] = p1;
        o[2] = p2;
        o[3] = p3;
    }
    *reinterpret_cast<uint4*>(blk + t * kWsTokStride + lane * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    if (lane == 0) reinterpret_cast<float*>(blk + trail)[t] = inexact ? 1.0f : __int_as_float((127 - e) << 23);
}

__device__ __forceinline__ uint32_t ws_ld_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier among the compute warps of all CTAs (qgemv_chain.cu's:
// sense-reversing on the caller's two words, bounded).
__device__ void ws_grid_barrier(const WsParams& p, volatile int* abort_flag)
{
    named_barrier_sync(1, kCcThreads);
    if (threadIdx.x == 0 && !*abort_flag) {
        uint32_t* count = p.sync;
        uint32_t* gen = p.sync + 1;
        __threadfence();
        const uint32_t g0 = ws_ld_acquire(gen);
        if (atomicAdd(count, 1u) == gridDim.x - 1) {
            atomicExch(count, 0u);
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            const uint64_t t0 = global_timer_ns();
            while (ws_ld_acquire(gen) == g0) {
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

// The stages of one CTA in issue order: op o, this CTA's unit u, stage c;
// with the fields of op o that issuing a stage needs, held in registers (a
// load from the kernel's parameters per stage would put the parameter-read
// latency on every issue).
struct WsCursor {
    int o, u, c;
    int P, C, Cp, n_units, R, R8, up_off, fmt, ufmt, ngu, dep;
    uint32_t box_tx, scales_off, mins_off, hi_off, blk, code_pitch, sc_pitch;
    size_t ws_off;
};

__device__ __forceinline__ void ws_cursor_load(const WsParams& p, WsCursor& k)
{
    const WsOp& op = p.op[k.o];
    k.P = op.a.P;
    k.C = op.a.C;
    k.Cp = op.a.Cp;
    k.n_units = op.a.n_units;
    k.R = op.a.R;
    k.R8 = op.a.R8;
    k.up_off = op.a.up_row_offset;
    k.fmt = op.fmt;
    k.ufmt = op.ufmt;
    k.ngu = op.epi == EPI_SWIGLU ? 2 : 1;
    k.dep = op.dep;
    k.box_tx = op.a.box_tx;
    k.scales_off = op.a.scales_off;
    k.mins_off = op.a.mins_off;
    k.hi_off = op.a.hi_off;
    k.blk = op.blk;
    k.code_pitch = op.code_pitch;
    k.sc_pitch = op.sc_pitch;
    k.ws_off = op.ws_off;
}

// Moves k to the first op at or after k.o in which this CTA has a unit.
__device__ __forceinline__ void ws_cursor_settle(const WsParams& p, WsCursor& k)
{
    while (k.o < p.n_ops) {
        ws_cursor_load(p, k);
        if (k.u < k.n_units) return;
        ++k.o;
        k.u = blockIdx.x;
        k.c = 0;
    }
}

__device__ __forceinline__ void ws_cursor_next(const WsParams& p, WsCursor& k)
{
    if (++k.c == k.Cp) {
        k.c = 0;
        k.u += gridDim.x;
        if (k.u >= k.n_units) {
            ++k.o;
            k.u = blockIdx.x;
            ws_cursor_settle(p, k);
        }
    }
}

// The TMA warp. Two rings: weight stages (deep: HBM latency) and the
// stages' activation blocks (shallow: the blocks come from L2). Stage s's
// consumers free both its slots at once, so one event drives the warp: once
// stage s - SX is done it copies stage s's blocks and the weights of stage
// s + SW - SX (the weight ring runs SW - SX stages ahead of the activation
// ring). Between events the warp sleeps in the barrier wait, off the issue
// slots the decoding warps use.
__device__ __forceinline__ void ws_producer(const WsParams& p, uint8_t* smem, uint64_t* full_w, uint64_t* empty_w,
                                           uint64_t* full_x, uint64_t* empty_x, volatile int* abort_flag,
                                           volatile int* xr, int lane)
{
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
    // the parameters the loop reads, in registers (a parameter read after each
    // copy instruction's memory clobber would be repeated every stage)
    const int SW = p.n_stages, SX = p.n_xstages, n_ops = p.n_ops, starve = p.starve;
    const uint32_t slot_bytes = p.slot_bytes, xslot_bytes = p.xslot_bytes, smem_xring = p.smem_xring;
    uint8_t* const ws = p.ws;
    const uint64_t wait_ns = p.wait_ns;
    int* const status = p.status;
    CcArgs wa{};  // cc_wait_warp's limit and status word
    wa.wait_ns = wait_ns;
    wa.status = status;
    WsCursor wc{};
    wc.u = static_cast<int>(blockIdx.x);
    WsCursor xc = wc;
    ws_cursor_settle(p, wc);
    ws_cursor_settle(p, xc);
    int wseq = 0, xseq = 0;
    bool pdl_done = false;

    // the weights of the cursor's stage into its slot (free by now)
    auto issue_w = [&]() {
        const int wsl = wseq % SW, o = wc.o, fmt = wc.fmt, ngu = wc.ngu;
        const int row0 = wc.u * wc.R, kc0 = wc.c * wc.P;
        const uint32_t cpitch = wc.code_pitch, spitch = wc.sc_pitch;
        uint8_t* sb = smem + wsl * slot_bytes;
        if (elect_one()) {
            // per matrix one box of the stage's P chunks x R rows (chunks past
            // K are filled with zeros and still counted)
            mbar_arrive_expect_tx(&full_w[wsl], wc.box_tx);
            for (int gg = 0; gg < ngu; ++gg) {
                if (fmt == FMT_NVFP4) {
                    const int row = row0 + gg * wc.up_off;
                    tma_load_3d(sb + gg * cpitch, &p.map[o][0], 0, row, kc0, &full_w[wsl]);
                    tma_load_3d(sb + wc.scales_off + gg * spitch, &p.map[o][1], 0, row, kc0, &full_w[wsl]);
                } else {
                    const CUtensorMap* mp = &p.map[o][4 * gg];
                    tma_load_3d(sb + gg * cpitch, mp, 0, row0, kc0, &full_w[wsl]);
                    tma_load_3d(sb + wc.scales_off + gg * spitch, mp + 1, 0, row0, kc0, &full_w[wsl]);
                    tma_load_3d(sb + wc.mins_off + gg * spitch, mp + 2, 0, row0, kc0, &full_w[wsl]);
                    if ((gg ? wc.ufmt : fmt) == FMT_Q5)
                        tma_load_3d(sb + wc.hi_off + gg * 2u * spitch, mp + 3, 0, row0, kc0, &full_w[wsl]);
                }
            }
        }
        __syncwarp();
        ws_cursor_next(p, wc);
        ++wseq;
    };
    // the blocks of the cursor's stage, once its op's blocks are written
    auto issue_x = [&]() -> bool {
        if (xc.dep) {
            const uint64_t t0 = global_timer_ns();
            while (__shfl_sync(0xffffffffu, xr[xc.o] != 0 ? 1 : 0, 0) == 0) {
                if (*abort_flag) return false;
                if (global_timer_ns() - t0 > wait_ns) {
                    if (lane == 0) set_device_status(status, QG_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                    return false;
                }
                __nanosleep(128);
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        } else if (!pdl_done) {
            // the conversion kernel's blocks
            asm volatile("griddepcontrol.wait;" ::: "memory");
            pdl_done = true;
        }
        const int xs = xseq % SX;
        const int live = min(xc.P, xc.C - xc.c * xc.P);
        const uint32_t bytes = static_cast<uint32_t>(live) * xc.blk;
        if (elect_one()) {
            mbar_arrive_expect_tx(&full_x[xs], bytes);
            bulk_load(smem + smem_xring + xs * xslot_bytes,
                      ws + xc.ws_off + static_cast<size_t>(xc.c * xc.P) * xc.blk, bytes, &full_x[xs]);
        }
        __syncwarp();
        ws_cursor_next(p, xc);
        ++xseq;
        return true;
    };

    bool stop = starve != 0;
    // the first weight stages go out before the conversion kernel is waited for
    while (!stop && wc.o < n_ops && wseq < SW) issue_w();
    while (!stop && xc.o < n_ops && xseq < SX)
        if (!issue_x()) stop = true;
    while (!stop && xc.o < n_ops) {
        // stage xseq - SX done: its activation slot and the weight slot of
        // stage xseq - SX (= wseq - SW) are free
        if (!cc_wait_warp(&empty_x[xseq % SX], ((xseq / SX) - 1) & 1, wa, abort_flag)) break;
        if (*abort_flag) break;
        if (wc.o < n_ops) issue_w();
        if (!issue_x()) break;
    }
    // No copy may still be landing in shared memory when the CTA exits.
    if (lane == 0) {
        for (int g = max(0, wseq - SW); g < wseq; ++g)
            mbar_wait_bounded(&full_w[g % SW], (g / SW) & 1, wait_ns, status);
        for (int g = max(0, xseq - SX); g < xseq; ++g)
            mbar_wait_bounded(&full_x[g % SX], (g / SX) & 1, wait_ns, status);
    }
    __syncwarp();
}

// The compute warps' unit loop of one op (qgemv_chain.cu's chain_units_mt,
// with each stage's activations, 2^-prescale factors, bf16 flag and group
// sums read from the stage's own ring slot). Tokens at or past M read token
// 0's row: their MMA columns are never stored.
template <int BITS, int BITS_U>
__device__ __forceinline__ void ws_units(const WsParams& pr, const WsOp& op, uint8_t* smem, uint64_t* full_w,
                                         uint64_t* empty_w, uint64_t* full_x, uint64_t* empty_x,
                                         volatile int* abort_flag, bool& aborted, int& seq, int warp, int lane)
{
    const int M = pr.M, SW = pr.n_stages, SX = pr.n_xstages;
    const uint32_t slot_bytes = pr.slot_bytes, xslot_bytes = pr.xslot_bytes;
    const CcArgs& a = op.a;
    const bool swiglu = op.epi == EPI_SWIGLU, resid = op.epi == EPI_RESID;
    const int ngu = swiglu ? 2 : 1;
    const int NRB = op.NRB;
    const int R = a.R, R8 = a.R8, P = a.P, C = a.C, Cp = a.Cp, n_units = a.n_units, n_out = a.n_out;
    const float gscale = a.g;
    // the epilogue's pointers in registers (a parameter read after each
    // store's memory clobber would be repeated per output)
    const uint16_t* const residual = a.residual;
    void* const y = a.y;
    const bool out_f32 = a.out_f32 != 0;
    const int b2 = warp / NRB;
    const int rb = warp % NRB;
    const bool active = b2 < P * ngu;
    const int p = active ? b2 / ngu : 0;
    const int n_mine = active ? max(0, (C - p + P - 1) / P) : 0;
    const int g = lane >> 2, c = lane & 3;
    const int t0 = 2 * c, t1 = 2 * c + 1;
    float* red = reinterpret_cast<float*>(smem + pr.smem_red);
    // the warp's 16 rows in the stage: matrix gg's box holds [chunk][row],
    // R rows per chunk, so the block starts at line L0 (rows past R read the
    // next chunk's rows, or the slot's tail: never stored)
    const uint32_t gm = active ? static_cast<uint32_t>(b2 % ngu) : 0u;
    const uint32_t r0 = static_cast<uint32_t>(p * R + 16 * rb);
    const uint32_t sw = r0 & 7u;
    const uint32_t box_off = gm * op.code_pitch + r0 * 128u;
    const uint32_t sbox_off = a.scales_off + gm * op.sc_pitch + r0 * 16u;
    const uint32_t mbox_off = a.mins_off + gm * op.sc_pitch + r0 * 16u;
    const uint32_t hbox_off = a.hi_off + gm * 2u * op.sc_pitch + r0 * 32u;
    // this warp's phase block in an activation slot, its token row, the block's trailer
    const uint32_t xblk_off = static_cast<uint32_t>(p) * op.blk;
    const uint32_t trow = static_cast<uint32_t>(g < M ? g : 0) * kWsTokStride;
    const uint32_t trail = static_cast<uint32_t>(M) * kWsTokStride;
    const uint32_t ring = smem_u32(smem);
    const uint32_t xring = smem_u32(smem + pr.smem_xring);
    const int tq0 = t0 < M ? t0 : 0, tq1 = t1 < M ? t1 : 0;

    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cc = 0; cc < Cp; ++cc, ++seq) {
            const int ws = seq % SW, xs = seq % SX;
            if (!aborted && !cc_wait_warp(&full_w[ws], (seq / SW) & 1, a, abort_flag)) aborted = true;
            if (!aborted && !cc_wait_warp(&full_x[xs], (seq / SX) & 1, a, abort_flag)) aborted = true;
            if (!aborted && cc < n_mine) {
                const uint32_t stage = ring + ws * slot_bytes;
                const uint32_t xb = xring + xs * xslot_bytes + xblk_off;
                const float pe0 = t0 < M ? __uint_as_float(lds32(xb + trail + 4u * t0)) : 0.f;
                const float pe1 = t1 < M ? __uint_as_float(lds32(xb + trail + 4u * t1)) : 0.f;
                const bool bf = lds32(xb + trail + 32u) != 0u;
                if constexpr (BITS == 0) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    if (bf)
                        mt_stage<true>(stage + box_off, stage + sbox_off, xb + trow, lane, kMtTokens, d, sw);
                    else
                        mt_stage<false>(stage + box_off, stage + sbox_off, xb + trow, lane, kMtTokens, d, sw);
                    acc[0] = fmaf(d[0], pe0, acc[0]);
                    acc[1] = fmaf(d[1], pe1, acc[1]);
                    acc[2] = fmaf(d[2], pe0, acc[2]);
                    acc[3] = fmaf(d[3], pe1, acc[3]);
                } else {
                    float aq[4] = {0.f, 0.f, 0.f, 0.f}, am[4] = {0.f, 0.f, 0.f, 0.f};
                    const float* gxb = reinterpret_cast<const float*>(smem + pr.smem_xring + xs * xslot_bytes +
                                                                      xblk_off + trail + 48u);
                    const float* gx0 = gxb + tq0 * 8;
                    const float* gx1 = gxb + tq1 * 8;
                    if (swiglu && (b2 & 1)) {  // the up matrix's box
                        if (bf)
                            mtq_stage<BITS_U, true>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                    stage + hbox_off, xb + trow, gx0, gx1, lane, kMtTokens, aq, am, sw);
                        else
                            mtq_stage<BITS_U, false>(stage + box_off, stage + sbox_off, stage + mbox_off,
                                                     stage + hbox_off, xb + trow, gx0, gx1, lane, kMtTokens, aq, am, sw);
                    } else if (bf) {
                        mtq_stage<BITS, true>(stage + box_off, stage + sbox_off, stage + mbox_off, stage + hbox_off,
                                              xb + trow, gx0, gx1, lane, kMtTokens, aq, am, sw);
                    } else {
                        mtq_stage<BITS, false>(stage + box_off, stage + sbox_off, stage + mbox_off, stage + hbox_off,
                                               xb + trow, gx0, gx1, lane, kMtTokens, aq, am, sw);
                    }
                    const float f0 = bf ? 1.0f : 16777216.0f * pe0, f1 = bf ? 1.0f : 16777216.0f * pe1;
                    acc[0] = fmaf(aq[0], f0, acc[0]) + am[0];
                    acc[1] = fmaf(aq[1], f1, acc[1]) + am[1];
                    acc[2] = fmaf(aq[2], f0, acc[2]) + am[2];
                    acc[3] = fmaf(aq[3], f1, acc[3]) + am[3];
                }
            }
            mbar_arrive(&empty_w[ws]);
            mbar_arrive(&empty_x[xs]);
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
                if (resid) val += bf16_bits_to_f32(ldg_cg_u16(residual + o));
                if (out_f32)
                    reinterpret_cast<float*>(y)[o] = val;
                else
                    reinterpret_cast<uint16_t*>(y)[o] = f32_to_bf16_bits_rn(val);
            }
        }
        named_barrier_sync(1, kCcThreads);
    }
}

template <bool HAS_Q>
__global__ void __launch_bounds__(kCcAllThreads, 1) chain_ws_kernel(const __grid_constant__ WsParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full_w = reinterpret_cast<uint64_t*>(smem + p.smem_bar);
    uint64_t* empty_w = full_w + kCcMaxStages;
    uint64_t* full_x = empty_w + kCcMaxStages;
    uint64_t* empty_x = full_x + kWsMaxXStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_x + kWsMaxXStages);
    volatile int* xr = abort_flag + 4;  // per op: its blocks are written (ops with after_previous)

    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_stages; ++s) {
            mbar_init(&full_w[s], 1);
            mbar_init(&empty_w[s], kCcThreads);
        }
        for (int s = 0; s < p.n_xstages; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&empty_x[s], kCcThreads);
        }
        *abort_flag = 0;
        for (int o = 0; o < kWsMaxOps; ++o) xr[o] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kCcTmaWarp) {
        ws_producer(p, smem, full_w, empty_w, full_x, empty_x, abort_flag, xr, lane);
        return;
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool aborted = false;
    int seq = 0;
    for (int o = 0; o < p.n_ops; ++o) {
        const WsOp& op = p.op[o];
        if (op.dep) {
            // the op reads an earlier op's output: convert it over the whole grid
            ws_grid_barrier(p, abort_flag);
            const int gw = blockIdx.x * kCcWarps + warp;
            for (int kc = gw; kc < op.a.C && !*abort_flag; kc += gridDim.x * kCcWarps) {
                uint8_t* blk = p.ws + op.ws_off + static_cast<size_t>(kc) * op.blk;
                if (HAS_Q && op.fmt != FMT_NVFP4)
                    ws_convert_chunk<true, true, false>(op.a.x, op.a.K, p.M, kc, nullptr, nullptr, blk, lane);
                else
                    ws_convert_chunk<false, true, false>(op.a.x, op.a.K, p.M, kc, nullptr, nullptr, blk, lane);
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            ws_grid_barrier(p, abort_flag);
            if (threadIdx.x == 0) {
                __threadfence_block();
                xr[o] = 1;
            }
        }
        if (*abort_flag) aborted = true;
        if (!HAS_Q || op.fmt == FMT_NVFP4) {
            ws_units<0, 0>(p, op, smem, full_w, empty_w, full_x, empty_x, abort_flag, aborted, seq, warp, lane);
        } else if constexpr (HAS_Q) {
            const bool b5 = op.fmt == FMT_Q5;
            const bool u5 = op.epi == EPI_SWIGLU ? op.ufmt == FMT_Q5 : b5;
#define QG_WS_Q(B, BU)                                                                                           \
    ws_units<B, BU>(p, op, smem, full_w, empty_w, full_x, empty_x, abort_flag, aborted, seq, warp, lane)
            if (b5 && u5)
                QG_WS_Q(5, 5);
            else if (b5)
                QG_WS_Q(5, 4);
            else if (u5)
                QG_WS_Q(4, 5);
            else
                QG_WS_Q(4, 4);
#undef QG_WS_Q
        }
    }
}

constexpr uint32_t ws_align(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

uint32_t ws_block_bytes(int fmt, int M)
{
    return static_cast<uint32_t>(M) * kWsTokStride + (fmt == FMT_NVFP4 ? kWsTrailNv : kWsTrailQ);
}

int ws_fmt(int format) { return format == QG_FMT_NVFP4 ? FMT_NVFP4 : format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4; }

}  // namespace

size_t chain_workspace_bytes(const qg_gemv_op* ops, int n_ops, int M)
{
    size_t off = 0;
    for (int o = 0; o < n_ops; ++o) {
        const size_t C = static_cast<size_t>(ops[o].K / kChunkK);
        off += (C * ws_block_bytes(ws_fmt(ops[o].format), M) + 255) / 256 * 256;
    }
    return off;
}

// 3..8 tokens with a workspace of chain_workspace_bytes(); QG_ERR_UNSUPPORTED
// when the list does not fit this kernel (K not a multiple of 256, an
// after_previous op with the RMSNorm prologue, shared memory).
qg_status launch_chain_ws(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, void* workspace,
                          cudaStream_t stream)
{
    if (n_ops < 1 || n_ops > kWsMaxOps || M < 3 || M > kMtTokens) return QG_ERR_UNSUPPORTED;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    static WsParams p;  // large: built here, copied into the launches' parameters
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    memset(&p, 0, sizeof(p));
    p.n_ops = n_ops;
    p.M = M;
    bool any_dep = false, any_q = false, any_indep = false;
    uint32_t slot_bytes = 0, xslot_bytes = 0, red_max = 0;
    int c_max = 0;
    size_t ws_off = 0;
    for (int o = 0; o < n_ops; ++o) {
        const qg_gemv_op& g = ops[o];
        if (g.K % kChunkK != 0) return QG_ERR_UNSUPPORTED;
        WsOp& op = p.op[o];
        op.fmt = ws_fmt(g.format);
        op.epi = g.epilogue == QG_EPI_SWIGLU ? EPI_SWIGLU : g.epilogue == QG_EPI_RESIDUAL ? EPI_RESID : EPI_NONE;
        op.dep = o > 0 && g.after_previous ? 1 : 0;
        if (op.dep && g.norm_weight != nullptr) return QG_ERR_UNSUPPORTED;
        const bool sep_up = g.up_codes != nullptr;
        op.ufmt = sep_up ? (g.up_format == QG_FMT_Q5 ? FMT_Q5 : FMT_Q4) : op.fmt;
        any_dep = any_dep || op.dep;
        any_indep = any_indep || !op.dep;
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
        a.K = g.K;
        a.C = g.K / kChunkK;
        c_max = std::max(c_max, a.C);
        a.n_out = n_out;
        a.R = R;
        a.R8 = (R + 15) / 16 * 16;
        op.NRB = a.R8 / 16;
        a.P = std::max(1, std::min(std::min(kCcWarps / (ngu * op.NRB), a.C), kWsMaxPhases));
        a.Cp = (a.C + a.P - 1) / a.P;
        a.n_units = (n_out + R - 1) / R;
        a.up_row_offset = op.epi == EPI_SWIGLU && !sep_up ? n_out : 0;
        a.out_f32 = op.epi == EPI_SWIGLU ? 0 : (g.y_dtype == QG_OUT_F32 ? 1 : 0);
        a.g = op.fmt == FMT_NVFP4 ? g.global_scale : 1.f;
        // stage layout: per matrix (gate, up) one [chunk][row] box of P
        // chunks x R rows for the codes, then the scales (then mins and the
        // Q5 plane); box_tx is the whole stage
        const uint32_t nbox = static_cast<uint32_t>(a.P * ngu);
        const uint32_t PR = static_cast<uint32_t>(a.P * a.R), nm = static_cast<uint32_t>(ngu);
        op.code_pitch = ws_align(PR * 128u, 1024);  // a swizzled box starts a 1024-byte period
        op.sc_pitch = ws_align(PR * 16u, 128);
        a.scales_off = nm * op.code_pitch;
        uint32_t st;
        if (op.fmt == FMT_NVFP4) {
            st = a.scales_off + nm * op.sc_pitch;
            a.box_tx = nm * PR * (128u + 16u);
        } else {
            const bool any5 = op.fmt == FMT_Q5 || op.ufmt == FMT_Q5;
            a.mins_off = ws_align(a.scales_off + nm * op.sc_pitch, 1024);
            a.hi_off = ws_align(a.mins_off + nm * op.sc_pitch, 1024);
            st = a.hi_off + (any5 ? nm * 2u * op.sc_pitch : 0u);
            a.box_tx = PR * (128u + 16u + 16u + (op.fmt == FMT_Q5 ? 32u : 0u));
            if (ngu == 2) a.box_tx += PR * (128u + 16u + 16u + (op.ufmt == FMT_Q5 ? 32u : 0u));
        }
        op.blk = ws_block_bytes(op.fmt, M);
        op.ws_off = ws_off;
        ws_off += (static_cast<size_t>(a.C) * op.blk + 255) / 256 * 256;
        // + 2 KB: a last 16-row block reads up to 15 lines past its box
        slot_bytes = std::max(slot_bytes, ws_align(st + 2048u, 1024));
        xslot_bytes = std::max(xslot_bytes, ws_align(static_cast<uint32_t>(a.P) * op.blk, 128));
        red_max = std::max(red_max, nbox * a.R8 * 8u);
        const uint64_t rows = static_cast<uint64_t>(g.N), C = static_cast<uint64_t>(a.C);
        const uint32_t Rb = static_cast<uint32_t>(a.R), Pb = static_cast<uint32_t>(a.P);
        if (!encode_tmap_chunks(&p.map[o][0], g.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, rows, C, Rb, Pb, true))
            return QG_ERR_CUDA;
        if (op.fmt == FMT_NVFP4) {
            if (!encode_tmap_chunks(&p.map[o][1], g.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 16, rows, C, Rb, Pb,
                                    false))
                return QG_ERR_CUDA;
        } else {
            const void* srcs[2][4] = {{g.codes, g.scales, g.mins, g.q_hi},
                                      {g.up_codes, g.up_scales, g.up_mins, g.up_q_hi}};
            const int fm[2] = {op.fmt, op.ufmt};
            for (int gg = 0; gg < (sep_up ? 2 : 1); ++gg) {
                CUtensorMap* mm = &p.map[o][4 * gg];
                if ((gg == 1 && !encode_tmap_chunks(&mm[0], srcs[gg][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, rows,
                                                    C, Rb, Pb, true)) ||
                    !encode_tmap_chunks(&mm[1], srcs[gg][1], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, 8, rows, C, Rb, Pb,
                                        false) ||
                    !encode_tmap_chunks(&mm[2], srcs[gg][2], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, 8, rows, C, Rb, Pb,
                                        false))
                    return QG_ERR_CUDA;
                if (fm[gg] == FMT_Q5 && !encode_tmap_chunks(&mm[3], srcs[gg][3], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 32,
                                                            rows, C, Rb, Pb, false))
                    return QG_ERR_CUDA;
            }
        }
    }
    if (any_dep && !sync) return QG_ERR_INVALID_ARG;
    // shared memory: weight ring | activation ring | partial sums | barriers and
    // flags. Three activation slots when that leaves four weight slots, else
    // two; at least three weight slots.
    const uint32_t red_bytes = ws_align(red_max * 4u, 128);
    const uint32_t bar_bytes = 2 * (kCcMaxStages + kWsMaxXStages) * 8 + 16 + 4 * kWsMaxOps;
    const uint32_t fixed = red_bytes + ws_align(bar_bytes, 16);
    if (fixed + 2 * xslot_bytes + 3 * slot_bytes > kCcSmemMax) return QG_ERR_UNSUPPORTED;
    const int n_xstages = fixed + 3 * xslot_bytes + 4 * slot_bytes <= kCcSmemMax ? 3 : 2;
    const int n_stages = std::min<int>(
        kCcMaxStages, static_cast<int>((kCcSmemMax - fixed - n_xstages * xslot_bytes) / slot_bytes));
    const uint32_t smem_ring = 0;
    const uint32_t smem_xring = n_stages * slot_bytes;
    const uint32_t smem_red = smem_xring + n_xstages * xslot_bytes;
    const uint32_t smem_bar = smem_red + red_bytes;
    const uint32_t smem_total = smem_bar + ws_align(bar_bytes, 16);
    if (smem_total > kCcSmemMax) return QG_ERR_UNSUPPORTED;

    int* status = device_status_ptr();
    if (!status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    p.n_stages = n_stages;
    p.n_xstages = n_xstages;
    p.slot_bytes = slot_bytes;
    p.xslot_bytes = xslot_bytes;
    p.smem_xring = smem_xring;
    p.smem_red = smem_red;
    p.smem_bar = smem_bar;
    p.ws = static_cast<uint8_t*>(workspace);
    p.sync = sync;
    p.wait_ns = dbg.wait_ns;
    p.starve = dbg.starve;
    p.status = status;
    for (int o = 0; o < n_ops; ++o) {
        CcArgs& a = p.op[o].a;
        a.n_stages = n_stages;
        a.stage_bytes = slot_bytes;
        a.smem_ring = smem_ring;
        a.smem_red = smem_red;
        a.smem_bar = smem_bar;
        a.wait_ns = dbg.wait_ns;
        a.starve = dbg.starve;
        a.status = status;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    // 1. the ops without after_previous: their activation blocks
    if (any_indep) {
        static bool conv_attr[64] = {};
        if (!conv_attr[dev]) {
            // the layer kernel's shared-memory split: an SM that runs a
            // conversion CTA then takes a layer CTA without reconfiguring
            if (cudaFuncSetAttribute(chain_ws_convert_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                return QG_ERR_CUDA;
            conv_attr[dev] = true;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c_max, n_ops);
        cfg.blockDim = dim3(32 * kMtTokens);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, chain_ws_convert_kernel, p) != cudaSuccess) return QG_ERR_CUDA;
    }
    // 2. the layer
    auto kern = any_q ? chain_ws_kernel<true> : chain_ws_kernel<false>;
    static bool attr_set[2][64] = {};
    if (!attr_set[any_q][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[any_q][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kCcAllThreads);
    cfg.dynamicSmemBytes = smem_total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (any_dep) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0] = pdl[0];
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
