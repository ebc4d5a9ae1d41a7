// cc_core.cuh -- the one-token CUDA-core GEMV's shared device code: its
// argument block, bounded waits, the exact activation conversion into
// shared memory and the per-stage dot-product code for NVFP4 and Q4/Q5.
// Included by the standalone one-token kernels (qgemv_cc.cu) and by the
// chained-layer kernel (qgemv_chain.cu); qgemv_cc.cu describes what they
// compute.
#pragma once

#include "common.cuh"

namespace qg {

namespace {

constexpr int kCcWarps = 16;                          // compute warps 0-15
constexpr int kCcThreads = 32 * kCcWarps;
constexpr int kCcTmaWarp = kCcWarps;                  // warp 16: TMA producer
constexpr int kCcAllThreads = 32 * (kCcWarps + 1);
constexpr int kCcMaxStages = 16;
// Stages the producer issues before it waits for the previous kernel to
// complete: CTAs that start early (their SM freed first) then cannot queue a
// whole ring of weight traffic ahead of the CTAs that start late.
constexpr int kCcLeadStages = 1;
constexpr int kCcRows = 4;                            // rows per thread
constexpr uint32_t kCcSmemMax = 227u * 1024u;

struct CcArgs {
    const uint16_t* x;         // bf16 activations, K values
    void* y;
    const uint16_t* residual;  // bf16 [n_out] or nullptr
    int K;
    int C;                     // K / 256
    int n_out;
    int R;                     // output rows per unit
    int R8;                    // R rounded up to 8: row stride of a box in shared memory
    int P;                     // K phases
    int Cp;                    // stages per phase
    int up_row_offset;         // SwiGLU: up row = gate row + this
    int out_f32;
    float g;
    int n_units;
    int n_stages;
    uint32_t stage_bytes;
    uint32_t scales_off;
    uint32_t code_pitch;       // chunked layout (chained kernels): bytes between a stage's matrices' code boxes
    uint32_t sc_pitch;         // the same for scales and mins (the Q5 plane: twice)
    uint32_t box_tx;
    uint32_t smem_ring;
    uint32_t smem_x;           // activations: C chunks of 256 f16 (or raw bf16)
    uint32_t smem_pe;          // C floats: 2^-prescale of each chunk
    uint32_t smem_fl;          // C bytes: 1 = chunk kept as raw bf16
    uint32_t smem_red;         // partial sums: P * NGU * R8 rows
    uint32_t smem_bar;
    // groupwise-int layouts only
    uint32_t mins_off;         // min boxes inside a stage
    uint32_t hi_off;           // Q5 high-bit boxes inside a stage
    uint32_t smem_gx;          // C * NSEG floats: sum of x over each k segment
    // RMSNorm prologue (norm_w == nullptr: none): the projection reads
    // h = bf16(x * r * gamma) with r = 1 / sqrt(mean(x^2) + eps)
    const uint16_t* norm_w;    // gamma, bf16 [K]
    float norm_eps;
    uint32_t smem_ss;          // C floats: each chunk's sum of squares
    uint64_t wait_ns;
    int starve;
    int* status;
};

// Shared-memory geometry of a stage as plain values: a kernel that walks
// several plans (the chained-layer kernel) keeps them in registers instead of
// indexing its parameter block inside the stage loop. Box b2 (phase b2 >>
// gsh, matrix b2 & (2^gsh - 1)) starts at code line (b2 & m) * gl + (b2 >>
// gsh) * pl and scale row (b2 & m) * gls + (b2 >> gsh) * pl: with gsh = 0
// and pl = R8 the per-phase layout (box b2 at b2 * R8); the chunked layout
// of the chained kernel has pl = R (one box per matrix holds a stage's
// chunks, R rows each) and gl, gls its matrices' pitches. Code lines are 128
// bytes, swizzled by (line & 7); scale rows 16 bytes, Q5 plane rows 32.
struct CcGeom {
    int pl;
    int gl;
    int gls;
    int gsh;
    uint32_t scales_off;
    uint32_t mins_off;
    uint32_t hi_off;
};

__device__ __forceinline__ CcGeom cc_geom(const CcArgs& a)
{
    return CcGeom{a.R8, 0, 0, 0, a.scales_off, a.mins_off, a.hi_off};
}

// The chunked layout of a chained kernel's stage (gsh: log2 of the matrices).
__device__ __forceinline__ CcGeom cc_geom_chunked(const CcArgs& a, int gsh)
{
    return CcGeom{a.R, static_cast<int>(a.code_pitch / 128u), static_cast<int>(a.sc_pitch / 16u), gsh, a.scales_off,
                  a.mins_off, a.hi_off};
}

__device__ __forceinline__ uint32_t cc_code_line(const CcGeom& g, int b2)
{
    return static_cast<uint32_t>((b2 & ((1 << g.gsh) - 1)) * g.gl + (b2 >> g.gsh) * g.pl);
}

__device__ __forceinline__ uint32_t cc_scale_row(const CcGeom& g, int b2)
{
    return static_cast<uint32_t>((b2 & ((1 << g.gsh) - 1)) * g.gls + (b2 >> g.gsh) * g.pl);
}

__device__ __forceinline__ bool cc_wait_warp(uint64_t* bar, uint32_t parity, const CcArgs& a,
                                             volatile int* abort_flag)
{
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const uint64_t t0 = global_timer_ns();
        for (;;) {
            if (mbar_try_wait_sleep(bar, parity, 20000u)) {
                ok = true;
                break;
            }
            if (*abort_flag) break;
            if (global_timer_ns() - t0 > a.wait_ns) {
                set_device_status(a.status, QG_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// acc + lo(w) * lo(x) and acc + hi(w) * hi(x): f16 (or bf16) operands, exact
// product, fp32 accumulation.
template <bool BF>
__device__ __forceinline__ float fma2_mixed(uint32_t w, uint32_t x, float acc)
{
    float r;
    if (BF)
        asm("{\n .reg .b16 wl, wh, xl, xh;\n .reg .f32 t;\n mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
            " fma.rn.f32.bf16 t, wl, xl, %3;\n fma.rn.f32.bf16 %0, wh, xh, t;\n}\n"
            : "=f"(r)
            : "r"(w), "r"(x), "f"(acc));
    else
        asm("{\n .reg .b16 wl, wh, xl, xh;\n .reg .f32 t;\n mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
            " fma.rn.f32.f16 t, wl, xl, %3;\n fma.rn.f32.f16 %0, wh, xh, t;\n}\n"
            : "=f"(r)
            : "r"(w), "r"(x), "f"(acc));
    return r;
}

// Where the activation conversion reads x: global memory through the
// read-only path, global memory through L2 only (x written earlier in the
// same kernel by other CTAs), or a raw copy already staged in the very
// shared-memory buffer the conversion writes (chunk kc at byte kc * 512,
// converted in place: each chunk is read whole by its warp before the warp
// writes it).
enum XSrc : int { XSRC_NC = 0, XSRC_CG = 1, XSRC_SMEM = 2 };

template <int SRC>
__device__ __forceinline__ uint4 cc_load_chunk(const CcArgs& a, const uint8_t* smem, int kc, int lane)
{
    if (SRC == XSRC_SMEM)
        return lds128(smem_u32(smem + a.smem_x) + static_cast<uint32_t>(kc) * 512u + static_cast<uint32_t>(lane) * 16u);
    return ldg_128<SRC == XSRC_CG>(a.x + static_cast<size_t>(kc) * kChunkK + lane * 8);
}

// The RMSNorm factor of the token (1 when there is no norm): chunk sums of
// squares in shared memory (one warp per chunk), then added in k order by
// every thread. Ends with a barrier of the compute threads.
// The warps converting: all 16 compute warps (barrier 1), a group of
// converter warps (barrier 2), or one warp alone.
template <int NW>
__device__ __forceinline__ void cc_conv_sync()
{
    if (NW == 1)
        __syncwarp();
    else if (NW == kCcWarps)
        named_barrier_sync(1, kCcThreads);
    else
        named_barrier_sync(2, 32 * NW);
}

template <int SRC, int NW = kCcWarps>
__device__ float cc_norm_factor(const CcArgs& a, const uint8_t* smem, int warp, int lane)
{
    if (a.norm_w == nullptr) return 1.0f;
    float* ss = reinterpret_cast<float*>(const_cast<uint8_t*>(smem) + a.smem_ss);
    for (int kc = warp; kc < a.C; kc += NW) {
        const float part = rms_chunk_ss(cc_load_chunk<SRC>(a, smem, kc, lane));
        if (lane == 0) ss[kc] = part;
    }
    cc_conv_sync<NW>();
    float t = 0.f;
    for (int kc = 0; kc < a.C; ++kc) t += ss[kc];
    return rms_factor(t, a.K, a.norm_eps);
}

// Converts the C chunks of x (h with the RMSNorm prologue) into shared
// memory (one warp per chunk, 8 values per lane): f16 under the chunk's exact
// prescale, or raw bf16 when its smallest nonzero value would fall below
// f16's last bit (a sufficient test of exactness: scaled exponent >= -17
// keeps all 8 significant bits at or above 2^-24). Within a chunk, 16-byte
// piece p of k segment s (NSEG segments of KS values) sits at
// p * NSEG * 16 + s * 16, so the segments' i-th pieces are contiguous and one
// load instruction of 8 threads with 8 segments touches 8 different bank
// groups. A chunk kept raw sets *any_bf. Each warp issues the loads of up to
// kBatch chunks before converting, so K up to 80 chunks costs one round trip
// to memory.
// Loads one batch of this warp's chunks (chunk base + u * NW) and, with the
// RMSNorm prologue, their gamma pieces, all before any use (each load
// followed by its use would serialise the round trips).
template <int SRC, int NW, int B>
__device__ __forceinline__ void cc_load_batch(const CcArgs& a, const uint8_t* smem, int base, int lane, uint4 (&raw)[B],
                                              uint4 (&gam)[B])
{
#pragma unroll
    for (int u = 0; u < B; ++u) {
        const int kc = base + u * NW;
        raw[u] = kc < a.C ? cc_load_chunk<SRC>(a, smem, kc, lane) : make_uint4(0, 0, 0, 0);
    }
    if (a.norm_w != nullptr) {
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int kc = base + u * NW;
            gam[u] = kc < a.C ? ldg_nc_128(a.norm_w + kc * kChunkK + lane * 8) : make_uint4(0, 0, 0, 0);
        }
    }
}

// The RMSNorm factor when every chunk of the warp fits one batch: the chunk
// sums of squares come from the batch already loaded (same order as
// cc_norm_factor), so x is read once.
template <int NW, int B>
__device__ __forceinline__ float cc_norm_factor_batch(const CcArgs& a, uint8_t* smem, int warp, int lane,
                                                      const uint4 (&raw)[B])
{
    float* ss = reinterpret_cast<float*>(smem + a.smem_ss);
#pragma unroll
    for (int u = 0; u < B; ++u) {
        const int kc = warp + u * NW;
        if (kc < a.C) {
            const float part = rms_chunk_ss(raw[u]);
            if (lane == 0) ss[kc] = part;
        }
    }
    cc_conv_sync<NW>();
    float t = 0.f;
    for (int kc = 0; kc < a.C; ++kc) t += ss[kc];
    return rms_factor(t, a.K, a.norm_eps);
}

template <int NSEG, int SRC = XSRC_NC, int NW = kCcWarps>
__device__ void cc_convert(const CcArgs& a, uint8_t* smem, int warp, int lane, volatile int* any_bf)
{
    constexpr int PPS = kChunkK / NSEG / 8;  // 16-byte pieces per segment
    constexpr int kBatch = NW < kCcWarps ? 8 : 5;
    const bool one_batch = a.C <= NW * kBatch;
    float rn = 1.0f;
    if (a.norm_w != nullptr && !one_batch) rn = cc_norm_factor<SRC, NW>(a, smem, warp, lane);
    uint32_t* xs = reinterpret_cast<uint32_t*>(smem + a.smem_x);
    float* pe = reinterpret_cast<float*>(smem + a.smem_pe);
    uint8_t* fl = smem + a.smem_fl;
    for (int base = warp; base < a.C || (a.norm_w != nullptr && one_batch && base == warp); base += NW * kBatch) {
        uint4 raw[kBatch], gam[kBatch];
        cc_load_batch<SRC, NW>(a, smem, base, lane, raw, gam);
        if (a.norm_w != nullptr) {
            // every warp takes part in the factor's barrier, with or without chunks
            if (one_batch) rn = cc_norm_factor_batch<NW>(a, smem, warp, lane, raw);
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (base + u * NW < a.C) raw[u] = rms_apply8(raw[u], gam[u], rn);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int kc = base + u * NW;
            if (kc >= a.C) break;
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
            const int off = (lane % PPS) * NSEG * 4 + (lane / PPS) * 4;  // in 4-byte words
            *reinterpret_cast<uint4*>(xs + kc * (kChunkK / 2) + off) = make_uint4(o[0], o[1], o[2], o[3]);
            if (lane == 0) {
                pe[kc] = inexact ? 1.0f : __int_as_float((127 - e) << 23);
                fl[kc] = inexact ? 1 : 0;
                if (inexact) *any_bf = 1;
            }
        }
    }
}

// Zeroes the padding rows R .. R8 - 1 of every box region in every ring
// slot (a TMA box holds R rows and never writes them), so that they read as
// zero codes and scales; run by the compute threads, concurrently with the
// first copies (which touch other bytes), before their first barrier.
// Regions: (offset of box 0, bytes per row).
__device__ void cc_zero_padding(const CcArgs& a, uint8_t* smem, int nbox, const uint32_t (&roff)[4],
                                const uint32_t (&rbytes)[4], int nreg)
{
    const int pad = a.R8 - a.R;
    if (pad == 0) return;
    for (int reg = 0; reg < nreg; ++reg) {
        const int pieces = static_cast<int>(rbytes[reg] / 16u);  // 16-byte pieces per row
        const int per_slot = nbox * pad * pieces;
        for (int t = threadIdx.x; t < a.n_stages * per_slot; t += kCcThreads) {
            const int slot = t / per_slot;
            const int rem = t % per_slot;
            const int b = rem / (pad * pieces);
            const int rr = a.R + (rem / pieces) % pad;
            const int pc = rem % pieces;
            uint8_t* dst = smem + a.smem_ring + slot * a.stage_bytes + roff[reg] +
                           (static_cast<uint32_t>(b * a.R8 + rr) * rbytes[reg]) + pc * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    }
}

// One thread's share of a stage: rows row0 .. row0 + 3 of box b2 (padding
// rows at or past R hold zero codes and scales), k segment `seg` (KS = 256 /
// NSEG values) of chunk kc. The four rows' blocks are interleaved, one chain
// of pair products per (row, block), so eight independent multiply-add chains
// are in flight.
template <int NSEG, bool BF>
__device__ __forceinline__ void cc_stage(const CcGeom& a, uint32_t stage, int b2, int row0, int seg,
                                         const uint32_t* xw, float pe, float (&acc)[kCcRows])
{
    constexpr int KS = kChunkK / NSEG;  // 32 or 16 k
    constexpr int NW = KS / 8;          // code words per row
    constexpr int NB = NW / 2;          // 16-k blocks per row
    const uint32_t cl = cc_code_line(a, b2) + static_cast<uint32_t>(row0);
    const uint32_t sr = cc_scale_row(a, b2) + static_cast<uint32_t>(row0);
    uint32_t cw[kCcRows][NW];
    float sc[kCcRows][NB];
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) {
        const uint32_t line = cl + static_cast<uint32_t>(i);
        const uint32_t rowb = stage + line * 128u;
        const uint32_t chunk = static_cast<uint32_t>(NW == 4 ? seg : seg >> 1) ^ (line & 7u);
        if constexpr (NW == 4) {
            const uint4 v = lds128(rowb + (chunk << 4));
            cw[i][0] = v.x; cw[i][1] = v.y; cw[i][2] = v.z; cw[i][3] = v.w;
        } else {
            const uint2 v = lds64(rowb + (chunk << 4) + static_cast<uint32_t>(seg & 1) * 8u);
            cw[i][0] = v.x; cw[i][1] = v.y;
        }
        // the NB scale bytes of this segment
        const uint32_t sb = stage + a.scales_off + (sr + static_cast<uint32_t>(i)) * 16u + static_cast<uint32_t>(seg * NB);
        const uint32_t two = NB == 2 ? lds16(sb) : lds8(sb);
        const uint32_t h2 = e4m3x2_to_f16x2(two);
        sc[i][0] = half_bits_to_f32(h2 & 0xFFFFu);
        if constexpr (NB == 2) sc[i][1] = half_bits_to_f32(h2 >> 16);
    }
    float u[kCcRows];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        float s[kCcRows];
#pragma unroll
        for (int i = 0; i < kCcRows; ++i) s[i] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int wd = 2 * blk + h;
            uint32_t w[kCcRows][4];
#pragma unroll
            for (int i = 0; i < kCcRows; ++i) {
                e2m1x8_to_f16x2x4(cw[i][wd], w[i]);
                if (BF) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) w[i][j] = f16x2_to_bf16x2(w[i][j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t xv = xw[wd * 4 + j];
#pragma unroll
                for (int i = 0; i < kCcRows; ++i) s[i] = fma2_mixed<BF>(w[i][j], xv, s[i]);
            }
        }
        // scale the block sums exactly by the E4M3 scale, then by 2^-prescale
#pragma unroll
        for (int i = 0; i < kCcRows; ++i) u[i] = blk == 0 ? s[i] * sc[i][0] : fmaf(s[i], sc[i][blk], u[i]);
    }
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) acc[i] = fmaf(u[i], pe, acc[i]);
}

// cc_stage for MT tokens: each decoded code pair feeds every token; token
// t's activation pieces are read from shared memory at xc + t * x_tok as
// the code words come (the same lds count as cc_stage, fewer live
// registers), its factor is pe[t], its sums acc[i * MT + t].
template <int NSEG, bool BF, int MT>
__device__ __forceinline__ void cc_stage_mt(const CcGeom& a, uint32_t stage, int b2, int row0, int seg,
                                            uint32_t xc, uint32_t x_tok, const float* pe,
                                            float (&acc)[kCcRows * MT])
{
    constexpr int KS = kChunkK / NSEG;
    constexpr int NW = KS / 8;
    constexpr int NB = NW / 2;
    const uint32_t cl = cc_code_line(a, b2) + static_cast<uint32_t>(row0);
    const uint32_t sr = cc_scale_row(a, b2) + static_cast<uint32_t>(row0);
    uint32_t cw[kCcRows][NW];
    float sc[kCcRows][NB];
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) {
        const uint32_t line = cl + static_cast<uint32_t>(i);
        const uint32_t rowb = stage + line * 128u;
        const uint32_t chunk = static_cast<uint32_t>(NW == 4 ? seg : seg >> 1) ^ (line & 7u);
        if constexpr (NW == 4) {
            const uint4 v = lds128(rowb + (chunk << 4));
            cw[i][0] = v.x; cw[i][1] = v.y; cw[i][2] = v.z; cw[i][3] = v.w;
        } else {
            const uint2 v = lds64(rowb + (chunk << 4) + static_cast<uint32_t>(seg & 1) * 8u);
            cw[i][0] = v.x; cw[i][1] = v.y;
        }
        const uint32_t sb = stage + a.scales_off + (sr + static_cast<uint32_t>(i)) * 16u + static_cast<uint32_t>(seg * NB);
        const uint32_t two = NB == 2 ? lds16(sb) : lds8(sb);
        const uint32_t h2 = e4m3x2_to_f16x2(two);
        sc[i][0] = half_bits_to_f32(h2 & 0xFFFFu);
        if constexpr (NB == 2) sc[i][1] = half_bits_to_f32(h2 >> 16);
    }
    float u[kCcRows * MT];
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
        float s[kCcRows * MT];
#pragma unroll
        for (int i = 0; i < kCcRows * MT; ++i) s[i] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int wd = 2 * blk + h;
            uint32_t w[kCcRows][4];
#pragma unroll
            for (int i = 0; i < kCcRows; ++i) {
                e2m1x8_to_f16x2x4(cw[i][wd], w[i]);
                if (BF) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) w[i][j] = f16x2_to_bf16x2(w[i][j]);
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint4 v = lds128(xc + t * x_tok + wd * NSEG * 16);
                const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < kCcRows; ++i) s[i * MT + t] = fma2_mixed<BF>(w[i][j], xv[j], s[i * MT + t]);
            }
        }
#pragma unroll
        for (int i = 0; i < kCcRows; ++i)
#pragma unroll
            for (int t = 0; t < MT; ++t)
                u[i * MT + t] = blk == 0 ? s[i * MT + t] * sc[i][0] : fmaf(s[i * MT + t], sc[i][blk], u[i * MT + t]);
    }
#pragma unroll
    for (int i = 0; i < kCcRows; ++i)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[i * MT + t] = fmaf(u[i * MT + t], pe[t], acc[i * MT + t]);
}

// ---------------------------------------------------------------- groupwise int (Q4 / Q5)
// Same plan for w = scale * q + min per group of 32 (NInfer article, section
// 2: the groupwise-int recipe): per row and group, y += scale * sum(q x) +
// min * sum(x). The codes enter the multiply-add as f16 subnormals: the f16
// with bit pattern q is exactly q * 2^-24 (q < 32), so a masked nibble pair
// is an f16 pair with no conversion at all, and the 2^24 moves into the
// scale. Nibble k and nibble k + 4 of a 32-bit code word form one pair, so
// the activations are stored paired the same way, (x_k, x_{k+4}). The sums
// of x per segment come from the original bf16 values, in a fixed order.

// Converts x as cc_convert does (RMSNorm prologue included), with the
// (k, k+4) pairing, and writes the fp32 sum of each segment's values (the
// values the projection reads: x, or h with the prologue). MT tokens (rows
// of x, K apart): token t's chunks at smem_x + t * C * 512, its factors at
// pe[t * C + kc], its segment sums at gx[(t * C + kc) * NSEG + s]; a chunk
// that one token cannot carry exactly in f16 stays raw bf16 for every token
// (one flag per chunk), so a stage runs one arithmetic for all of them.
// Q45 = false gives the NVFP4 layout of the multi-token NVFP4 kernel:
// natural pairs, no segment sums.
template <int NSEG, int SRC = XSRC_NC, int NW = kCcWarps, int MT = 1, bool Q45 = true>
__device__ void cc_convert_q45(const CcArgs& a, uint8_t* smem, int warp, int lane, volatile int* any_bf)
{
    constexpr int kBatch = MT == 2 ? 3 : (NW < kCcWarps ? 8 : 5);
    constexpr int PPS = kChunkK / NSEG / 8;  // lanes (16-byte pieces) per segment
    const bool one_batch = MT == 1 && a.C <= NW * kBatch;
    float rn[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) rn[t] = 1.0f;
    if (a.norm_w != nullptr && !one_batch) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            CcArgs at = a;
            at.x = a.x + static_cast<size_t>(t) * a.K;
            at.smem_ss = a.smem_ss + static_cast<uint32_t>(t * a.C) * 4u;
            rn[t] = cc_norm_factor<SRC, NW>(at, smem, warp, lane);
        }
    }
    uint32_t* xs = reinterpret_cast<uint32_t*>(smem + a.smem_x);
    float* pe = reinterpret_cast<float*>(smem + a.smem_pe);
    float* gx = reinterpret_cast<float*>(smem + a.smem_gx);
    uint8_t* fl = smem + a.smem_fl;
    for (int base = warp; base < a.C || (a.norm_w != nullptr && one_batch && base == warp); base += NW * kBatch) {
        uint4 raw[MT][kBatch], gam[kBatch];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int kc = base + u * NW;
                raw[t][u] = kc < a.C ? (SRC == XSRC_SMEM && MT == 1
                                            ? cc_load_chunk<SRC>(a, smem, kc, lane)
                                            : ldg_128<SRC == XSRC_CG>(a.x + static_cast<size_t>(t) * a.K +
                                                                      static_cast<size_t>(kc) * kChunkK + lane * 8))
                                     : make_uint4(0, 0, 0, 0);
            }
        }
        if (a.norm_w != nullptr) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int kc = base + u * NW;
                gam[u] = kc < a.C ? ldg_nc_128(a.norm_w + kc * kChunkK + lane * 8) : make_uint4(0, 0, 0, 0);
            }
            if (one_batch) rn[0] = cc_norm_factor_batch<NW>(a, smem, warp, lane, raw[0]);
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (base + u * NW < a.C) raw[t][u] = rms_apply8(raw[t][u], gam[u], rn[t]);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int kc = base + u * NW;
            if (kc >= a.C) break;
            int e[MT];
            bool inexact = false;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint32_t wv[4] = {raw[t][u].x, raw[t][u].y, raw[t][u].z, raw[t][u].w};
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
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint32_t wv[4] = {raw[t][u].x, raw[t][u].y, raw[t][u].z, raw[t][u].w};
                float sx = 0.f;
                if constexpr (Q45) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        sx += bf16_bits_to_f32((i & 1) ? (wv[i >> 1] >> 16) : (wv[i >> 1] & 0xFFFFu));
#pragma unroll
                    for (int sh = 1; sh < PPS; sh <<= 1) sx += __shfl_xor_sync(0xffffffffu, sx, sh);
                }
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
                const int off = (lane % PPS) * NSEG * 4 + (lane / PPS) * 4;
                uint32_t* dst = xs + (t * a.C + kc) * (kChunkK / 2) + off;
                if constexpr (Q45) {
                    // natural pairs (x0,x1)(x2,x3)(x4,x5)(x6,x7) -> (x0,x4)(x1,x5)(x2,x6)(x3,x7)
                    const uint32_t p0 = __byte_perm(o[0], o[2], 0x5410), p1 = __byte_perm(o[0], o[2], 0x7632);
                    const uint32_t p2 = __byte_perm(o[1], o[3], 0x5410), p3 = __byte_perm(o[1], o[3], 0x7632);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(p0, p1, p2, p3);
                    if (lane % PPS == 0) gx[(t * a.C + kc) * NSEG + lane / PPS] = sx;
                } else {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (lane == 0) pe[t * a.C + kc] = inexact ? 1.0f : __int_as_float((127 - e[t]) << 23);
            }
            if (lane == 0) {
                fl[kc] = inexact ? 1 : 0;
                if (inexact) *any_bf = 1;
            }
        }
    }
}

// Code word w (8 unsigned 4-bit codes) -> four f16 pairs of subnormals
// (q_j, q_{j+4}) * 2^-24; Q5 ORs in the fifth bit (bit 4 of each half) from
// hsp, the word's high bits spread as k0..k3 -> bits 4..7 and k4..k7 -> bits
// 20..23.
template <int BITS>
__device__ __forceinline__ void q45_pairs(uint32_t w, uint32_t hsp, uint32_t (&z)[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        z[j] = (w >> (4 * j)) & 0x000F000Fu;
        if (BITS == 5) z[j] |= (hsp >> j) & 0x00100010u;
    }
}

// One thread's share of a stage (see cc_stage); `seg` covers one group
// (NSEG = 8) or half of one (NSEG = 16). The bf16 path (a chunk kept raw)
// widens the codes and activations to fp32.
//
// MT tokens (1 or 2) share each decoded code pair: token t's activation
// words are xw[t * KS / 2 ...], its factors pe[t] and gxs[t], its sums
// acc[i * MT + t].
template <int NSEG, int BITS, bool BF, int MT = 1>
__device__ __forceinline__ void cc_stage_q45(const CcGeom& a, uint32_t stage, int b2, int row0, int seg,
                                             const uint32_t* xw, const float* pe, const float* gxs,
                                             float (&acc)[kCcRows * MT])
{
    constexpr int KS = kChunkK / NSEG;
    constexpr int NW = KS / 8;
    const int grp = NSEG == 8 ? seg : seg >> 1;
    const uint32_t cl = cc_code_line(a, b2) + static_cast<uint32_t>(row0);
    const uint32_t sr = cc_scale_row(a, b2) + static_cast<uint32_t>(row0);
#pragma unroll
    for (int i = 0; i < kCcRows; ++i) {
        // rows at or past R: padding (zeros) or another box's rows; never stored
        const uint32_t line = cl + static_cast<uint32_t>(i);
        const uint32_t rowi = sr + static_cast<uint32_t>(i);
        const uint32_t chunk = static_cast<uint32_t>(NW == 4 ? seg : seg >> 1) ^ (line & 7u);
        uint32_t cw[NW];
        if constexpr (NW == 4) {
            const uint4 v = lds128(stage + line * 128u + (chunk << 4));
            cw[0] = v.x; cw[1] = v.y; cw[2] = v.z; cw[3] = v.w;
        } else {
            const uint2 v = lds64(stage + line * 128u + (chunk << 4) + static_cast<uint32_t>(seg & 1) * 8u);
            cw[0] = v.x; cw[1] = v.y;
        }
        uint32_t hb = 0;
        if (BITS == 5) {
            // 4 (NSEG = 8) or 2 bytes of high bits, one per 8 k
            const uint32_t ha = stage + a.hi_off + rowi * 32u + static_cast<uint32_t>(seg * NW);
            hb = NW == 4 ? lds32(ha) : lds16(ha);
        }
        const float sc = half_bits_to_f32(lds16(stage + a.scales_off + rowi * 16u + static_cast<uint32_t>(grp * 2)));
        const float mn = half_bits_to_f32(lds16(stage + a.mins_off + rowi * 16u + static_cast<uint32_t>(grp * 2)));
        float s0[MT], s1[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) s0[t] = s1[t] = 0.f;
#pragma unroll
        for (int wd = 0; wd < NW; ++wd) {
            uint32_t hsp = 0;
            if (BITS == 5) {
                const uint32_t h8 = (hb >> (8 * wd)) & 0xFFu;
                hsp = ((h8 & 0x0Fu) << 4) | ((h8 & 0xF0u) << 16);
            }
            uint32_t z[4];
            q45_pairs<BITS>(cw[wd], hsp, z);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint32_t xv = xw[t * (KS / 2) + wd * 4 + j];
                    if (BF) {
                        // raw bf16 activations: widen both sides to fp32
                        s0[t] = fmaf(static_cast<float>(z[j] & 0xFFFFu), __uint_as_float(xv << 16), s0[t]);
                        s1[t] = fmaf(static_cast<float>(z[j] >> 16), __uint_as_float(xv & 0xFFFF0000u), s1[t]);
                    } else if (j & 1) {
                        s1[t] = fma2_mixed<false>(z[j], xv, s1[t]);
                    } else {
                        s0[t] = fma2_mixed<false>(z[j], xv, s0[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            // subnormal codes carry 2^-24 (not on the bf16 path)
            const float sq = (s0[t] + s1[t]) * (BF ? 1.0f : 16777216.0f);
            acc[i * MT + t] = fmaf(sq * sc, pe[t], acc[i * MT + t]);
            acc[i * MT + t] = fmaf(mn, gxs[t], acc[i * MT + t]);
        }
    }
}

}  // namespace

}  // namespace qg
