// mt_core.cuh -- the warp-MMA decode GEMV's shared device code: its
// argument block, the activation conversion into shared memory (one window
// of chunks, all tokens) and the per-stage MMA code for NVFP4 and Q4/Q5.
// Included by the standalone kernel (qgemv_mt.cu) and by the chained-layer
// kernel (qgemv_chain.cu); qgemv_mt.cu describes what they compute.
#pragma once

#include "cc_core.cuh"

namespace qg {

namespace {

constexpr int kMtTokens = 8;    // the MMA's n
constexpr int kMtXPad = 16;     // bytes between consecutive tokens' activation rows (bank spread)

struct MtArgs {
    CcArgs a;        // plan; a.R8 is the box pitch here (R rounded up to 16)
    int M;           // tokens
    int NRB;         // 16-row blocks per box
    int W;           // chunks of activations held at a time (a multiple of P; C when all fit)
    uint32_t x_tok;  // bytes between tokens' activations in shared memory
};

// codes, scales, then (groupwise int) mins and the Q5 plane; a groupwise-int
// SwiGLU's up matrix in m[4..7]
struct MtMaps {
    CUtensorMap m[8];
};

__device__ __forceinline__ uint32_t mt_bsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void mt_ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <bool BF>
__device__ __forceinline__ void mt_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if (BF)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Converts window w0, with the RMSNorm prologue if NORM_OK and a.norm_w is
// set (NORM_OK = false compiles the plain conversion alone: a second inlined
// variant slowed the stage loops that hold the window conversion).
template <bool Q45, bool CG, bool NORM_OK>
__device__ __forceinline__ void mt_convert_any(const MtArgs& m, uint8_t* smem, int warp, int lane,
                                               volatile int* any_bf, int w0);

// RMSNorm prologue (a.norm_w set): every token's r = 1 / sqrt(sum(x^2) / K +
// eps) over all of K, in the fixed order of rms_chunk_ss (chunk sums added in
// k order), at a.smem_ss + 4 * (M * C + t); the chunk sums before it. Run by
// all compute warps before the first window is converted.
template <bool CG>
__device__ void mt_norm_factors(const MtArgs& m, uint8_t* smem, int warp, int lane)
{
    const CcArgs& a = m.a;
    float* ss = reinterpret_cast<float*>(smem + a.smem_ss);
    const int items = m.M * a.C;
    constexpr int B = 4;
    for (int base = warp; base < items; base += kCcWarps * B) {
        uint4 raw[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = base + u * kCcWarps;
            raw[u] = it < items ? ldg_128<CG>(a.x + static_cast<size_t>(it / a.C) * a.K +
                                              static_cast<size_t>(it % a.C) * kChunkK + lane * 8)
                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int it = base + u * kCcWarps;
            if (it >= items) break;
            const float v = rms_chunk_ss(raw[u]);
            if (lane == 0) ss[it] = v;
        }
    }
    named_barrier_sync(1, kCcThreads);
    if (static_cast<int>(threadIdx.x) < m.M) {
        float s = 0.f;
        for (int kc = 0; kc < a.C; ++kc) s += ss[threadIdx.x * a.C + kc];
        ss[items + threadIdx.x] = rms_factor(s, a.K, a.norm_eps);
    }
    named_barrier_sync(1, kCcThreads);
}

// Every token's activations of chunks w0 .. w0 + W - 1 (a window) into shared
// memory: chunk kc = w0 + j of token t at smem_x + t * x_tok + j * 512 (k
// order, f16 after the exact prescale, or raw bf16 when some token's chunk
// does not fit f16), 2^-prescale at pe[t * W + j], the chunk's bf16 flag at
// fl[j]. One warp per chunk. Q45: each lane's 8 values stored paired (x0,
// x4)(x1, x5)(x2, x6)(x3, x7), and the sum of each group of 32 values (from
// the bf16 values) at gx[(t * W + j) * 8 + group]. CG: read x through L2
// only (an earlier op of the same launch may have written it). NORM (the
// RMSNorm prologue): the values converted are h = bf16(x * r * gamma), with r
// from mt_norm_factors.
template <bool Q45, bool CG = false, bool NORM = false>
__device__ void mt_convert(const MtArgs& m, uint8_t* smem, int warp, int lane, volatile int* any_bf, int w0)
{
    const CcArgs& a = m.a;
    uint8_t* xs = smem + a.smem_x;
    float* pe = reinterpret_cast<float*>(smem + a.smem_pe);
    uint8_t* fl = smem + a.smem_fl;
    float* gx = reinterpret_cast<float*>(smem + a.smem_gx);
    const int w1 = min(a.C, w0 + m.W);
    for (int kc = w0 + warp; kc < w1; kc += kCcWarps) {
        const int j = kc - w0;
        uint4 raw[kMtTokens];
#pragma unroll
        for (int t = 0; t < kMtTokens; ++t)
            raw[t] = t < m.M ? ldg_128<CG>(a.x + static_cast<size_t>(t) * a.K + static_cast<size_t>(kc) * kChunkK +
                                          lane * 8)
                             : make_uint4(0, 0, 0, 0);
        if constexpr (NORM) {
            const uint4 gam = ldg_nc_128(a.norm_w + static_cast<size_t>(kc) * kChunkK + lane * 8);
            const float* rn = reinterpret_cast<const float*>(smem + a.smem_ss) + m.M * a.C;
#pragma unroll
            for (int t = 0; t < kMtTokens; ++t)
                if (t < m.M) raw[t] = rms_apply8(raw[t], gam, rn[t]);
        }
        int e[kMtTokens];
        bool inexact = false;
#pragma unroll
        for (int t = 0; t < kMtTokens; ++t) {
            e[t] = 0;
            if (t >= m.M) continue;
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
#pragma unroll
        for (int t = 0; t < kMtTokens; ++t) {
            if (t >= m.M) continue;
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
            if constexpr (Q45) {
                float sx = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    sx += bf16_bits_to_f32((i & 1) ? (wv[i >> 1] >> 16) : (wv[i >> 1] & 0xFFFFu));
                sx += __shfl_xor_sync(0xffffffffu, sx, 1);
                sx += __shfl_xor_sync(0xffffffffu, sx, 2);
                if ((lane & 3) == 0) gx[(t * m.W + j) * 8 + (lane >> 2)] = sx;
                const uint32_t p0 = __byte_perm(o[0], o[2], 0x5410), p1 = __byte_perm(o[0], o[2], 0x7632);
                const uint32_t p2 = __byte_perm(o[1], o[3], 0x5410), p3 = __byte_perm(o[1], o[3], 0x7632);
                o[0] = p0;
                o[1] = p1;
                o[2] = p2;
                o[3] = p3;
            }
            *reinterpret_cast<uint4*>(xs + t * m.x_tok + j * (kChunkK * 2) + lane * 16) =
                make_uint4(o[0], o[1], o[2], o[3]);
            if (lane == 0) pe[t * m.W + j] = inexact ? 1.0f : __int_as_float((127 - e[t]) << 23);
        }
        if (lane == 0) {
            fl[j] = inexact ? 1 : 0;
            if (inexact) *any_bf = 1;
        }
    }
    // tokens M..7 of the MMA read zeros: their activation rows are never loaded
}

// One warp, one stage: rows 16 rb .. 16 rb + 15 of box b2 over the stage's
// 256 k; d[] gets the MMA sums (rows g, g + 8; tokens 2c, 2c + 1), built in
// two independent chains (the first and second MMA of each 32-k half) that
// are added at the end.
// sw: the box's first line modulo 8 when the box does not start a 1024-byte
// swizzle period (the 128-byte swizzle follows the line's address).
template <bool BF>
__device__ __forceinline__ void mt_stage(uint32_t box, uint32_t sbox, uint32_t xc, int lane, int M, float (&d)[4],
                                         uint32_t sw = 0)
{
    float d2[4] = {0.f, 0.f, 0.f, 0.f};
    const int g = lane >> 2, c = lane & 3;
    const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);
    const bool tok = g < M;
#pragma unroll
    for (int ti = 0; ti < 4; ++ti) {
        uint32_t cr[4];
        const int lc = 2 * ti + (lane >> 4);
        mt_ldmatrix_x4(cr, box + static_cast<uint32_t>(lr) * 128u +
                               ((static_cast<uint32_t>(lc) ^ ((static_cast<uint32_t>(lr) + sw) & 7u)) << 4));
        const uint32_t sw_g = lds32(sbox + static_cast<uint32_t>(g) * 16u + 4u * ti);
        const uint32_t sw_g8 = lds32(sbox + static_cast<uint32_t>(g + 8) * 16u + 4u * ti);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const uint4 bx = tok ? lds128(xc + static_cast<uint32_t>(64 * ti + 32 * ch + 8 * c) * 2u)
                                 : make_uint4(0, 0, 0, 0);
            // 16-k block 4 ti + 2 ch + c / 2: its E4M3 byte twice, converted,
            // is the scale in both halves
            const uint32_t sel = static_cast<uint32_t>((2 * ch + (c >> 1)) * 0x11);
            const uint32_t s_g = e4m3x2_to_f16x2(__byte_perm(sw_g, 0, sel));
            const uint32_t s_g8 = e4m3x2_to_f16x2(__byte_perm(sw_g8, 0, sel));
            uint32_t pg[4], pg8[4];
            e2m1x8_to_f16x2x4(cr[2 * ch], pg);
            e2m1x8_to_f16x2x4(cr[2 * ch + 1], pg8);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                pg[b] = hmul2(pg[b], s_g);
                pg8[b] = hmul2(pg8[b], s_g8);
                if (BF) {
                    pg[b] = f16x2_to_bf16x2(pg[b]);
                    pg8[b] = f16x2_to_bf16x2(pg8[b]);
                }
            }
            const uint32_t A0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
            const uint32_t A1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
            mt_mma<BF>(d, A0, bx.x, bx.y);
            mt_mma<BF>(d2, A1, bx.z, bx.w);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] += d2[i];
}

// The compute warps' unit loop. Window w0 = 0 is converted on entry; a
// stage in another window first converts it (all compute warps, between two
// barriers; the weight copies keep landing in the ring meanwhile).
// Q4/Q5, one warp, one stage: rows 16 rb .. 16 rb + 15 over the stage's
// 256 k (8 groups of 32). Per group the two MMAs give D = sum(q x) (times
// 2^-24 on the f16 path); aq collects scale * D, am collects min * sum(x),
// per (row g or g + 8, token 2c or 2c + 1).
template <int BITS, bool BF>
__device__ __forceinline__ void mtq_stage(uint32_t box, uint32_t sbox, uint32_t mbox, uint32_t hbox, uint32_t xc,
                                          const float* gxt0, const float* gxt1, int lane, int M, float (&aq)[4],
                                          float (&am)[4], uint32_t sw = 0)
{
    const int g = lane >> 2, c = lane & 3;
    const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);
    const bool tok = g < M;
#pragma unroll
    for (int ti = 0; ti < 4; ++ti) {
        uint32_t cr[4];
        const int lc = 2 * ti + (lane >> 4);
        mt_ldmatrix_x4(cr, box + static_cast<uint32_t>(lr) * 128u +
                               ((static_cast<uint32_t>(lc) ^ ((static_cast<uint32_t>(lr) + sw) & 7u)) << 4));
        // the two groups of this tile: scale and min of rows g and g + 8
        const uint32_t sg = lds32(sbox + static_cast<uint32_t>(g) * 16u + 4u * ti);
        const uint32_t sg8 = lds32(sbox + static_cast<uint32_t>(g + 8) * 16u + 4u * ti);
        const uint32_t mg = lds32(mbox + static_cast<uint32_t>(g) * 16u + 4u * ti);
        const uint32_t mg8 = lds32(mbox + static_cast<uint32_t>(g + 8) * 16u + 4u * ti);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const int grp = 2 * ti + ch;
            uint32_t hs_g = 0, hs_g8 = 0;
            if (BITS == 5) {
                const uint32_t hb = static_cast<uint32_t>(8 * ti + 4 * ch + c);  // plane byte of k .. k + 7
                const uint32_t h8 = lds8(hbox + static_cast<uint32_t>(g) * 32u + hb);
                const uint32_t h88 = lds8(hbox + static_cast<uint32_t>(g + 8) * 32u + hb);
                hs_g = ((h8 & 0x0Fu) << 4) | ((h8 & 0xF0u) << 16);
                hs_g8 = ((h88 & 0x0Fu) << 4) | ((h88 & 0xF0u) << 16);
            }
            uint32_t z[4], z8[4];
            q45_pairs<BITS>(cr[2 * ch], hs_g, z);
            q45_pairs<BITS>(cr[2 * ch + 1], hs_g8, z8);
            if (BF) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    z[b] = mt_bsub2(z[b] | 0x43004300u, 0x43004300u);
                    z8[b] = mt_bsub2(z8[b] | 0x43004300u, 0x43004300u);
                }
            }
            const uint4 bx = tok ? lds128(xc + static_cast<uint32_t>(64 * ti + 32 * ch + 8 * c) * 2u)
                                 : make_uint4(0, 0, 0, 0);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t A0[4] = {z[0], z8[0], z[1], z8[1]};
            const uint32_t A1[4] = {z[2], z8[2], z[3], z8[3]};
            mt_mma<BF>(d, A0, bx.x, bx.y);
            mt_mma<BF>(d, A1, bx.z, bx.w);
            const float s_g = half_bits_to_f32(ch ? (sg >> 16) : (sg & 0xFFFFu));
            const float s_g8 = half_bits_to_f32(ch ? (sg8 >> 16) : (sg8 & 0xFFFFu));
            const float m_g = half_bits_to_f32(ch ? (mg >> 16) : (mg & 0xFFFFu));
            const float m_g8 = half_bits_to_f32(ch ? (mg8 >> 16) : (mg8 & 0xFFFFu));
            const float x0 = gxt0[grp], x1 = gxt1[grp];
            aq[0] = fmaf(s_g, d[0], aq[0]);
            aq[1] = fmaf(s_g, d[1], aq[1]);
            aq[2] = fmaf(s_g8, d[2], aq[2]);
            aq[3] = fmaf(s_g8, d[3], aq[3]);
            am[0] = fmaf(m_g, x0, am[0]);
            am[1] = fmaf(m_g, x1, am[1]);
            am[2] = fmaf(m_g8, x0, am[2]);
            am[3] = fmaf(m_g8, x1, am[3]);
        }
    }
}

template <bool Q45, bool CG, bool NORM_OK>
__device__ __forceinline__ void mt_convert_any(const MtArgs& m, uint8_t* smem, int warp, int lane,
                                               volatile int* any_bf, int w0)
{
    if (NORM_OK && m.a.norm_w != nullptr)
        mt_convert<Q45, CG, NORM_OK>(m, smem, warp, lane, any_bf, w0);
    else
        mt_convert<Q45, CG, false>(m, smem, warp, lane, any_bf, w0);
}

}  // namespace

}  // namespace qg
