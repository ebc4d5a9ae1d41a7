// qgemv_dense.cu -- TMA-fed tensor-core GEMV for NVFP4 and Q4/Q5 weights,
// M = 1..8 tokens, with fused residual-add and SwiGLU epilogues.
//
// Prior art on the pages: NInfer writes one fused matmul (+ residual add /
// SwiGLU) kernel per weight format because decode is memory-bandwidth bound
// (NInfer article, section 2 "自研 CUDA 算子 混合量化权重"); Decapybara's
// mx_gemv.cu is an NVFP4 block mat-vec (Decapybara README, "Blackwell CUDA 内核
// 套件"). Both target sm_120a; this kernel is designed for sm_103a:
//
//   * Each CTA owns a contiguous range of R output rows (R = ceil(N / #SMs),
//     so every SM streams the same number of bytes) and walks K in 256-wide
//     chunks. One warp issues 2-D TMA loads of the chunk's codes and scales
//     into a ring of shared-memory stages (mbarrier full/empty pairs); eight
//     consumer warps decode and multiply. Every weight byte crosses HBM once.
//   * Codes arrive 128B-swizzled, so ldmatrix reads a 16-row x 64-k tile of
//     4-bit codes per instruction without bank conflicts.
//   * NVFP4 decode: cvt.rn.f16x2.e2m1x2 turns two codes into f16 exactly, and
//     an f16 multiply by the E4M3 block scale (also converted exactly) is exact
//     too: e2m1 * e4m3 has at most 6 significant bits and lies in
//     [2^-10, 2688]. Q4/Q5 decode: q is placed in an f16 mantissa
//     (1024 + q) and 1024 subtracted, exactly.
//   * The products run on the tensor cores (mma.m16n8k16, f16 in, fp32
//     accumulate), 16 weight rows x 8 token columns per MMA. Tokens beyond M
//     are zero columns.
//   * Activations are bf16; they enter the MMA as f16 after an exact
//     power-of-two prescale chosen per (token, 256-k chunk) so that the chunk
//     maximum lands in [2^14, 2^15). Every bf16 value within 2^31 of that
//     maximum is then exact in f16. A chunk holding a smaller nonzero value is
//     flagged and gets extra passes over residual terms (x - f16(x)) * 2^24, so
//     the result is exact-product fp32 accumulation for every finite input.
//   * Accumulation: each chunk's MMA partial (at most 16 chained MMAs) is
//     scaled back by 2^-p and added to an fp32 accumulator; Q groups add
//     scale * sum(q x) + min * sum(x) per group of 32.
#include "common.cuh"

#include <cuda_bf16.h>

namespace qg {

namespace {

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr)
{
    uint32_t v;
    asm volatile("{\n .reg .u8 b;\n ld.shared.u8 b, [%1];\n cvt.u32.u8 %0, b;\n}\n" : "=r"(v) : "r"(addr));
    return v;
}

// Pack 8 16-bit values in the format's pair order: natural k order for
// NVFP4 ({k, k+1} pairs, matching the e2m1x2 decode), {k, k+4} pairs for Q
// (matching the 1024 + q mantissa decode).
template <int FMT>
__device__ __forceinline__ uint4 pack_pairs(const uint32_t (&h)[8])
{
    if (FMT == FMT_NVFP4)
        return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    return make_uint4(h[0] | (h[4] << 16), h[1] | (h[5] << 16), h[2] | (h[6] << 16), h[3] | (h[7] << 16));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

struct TileAcc {
    float v[2][4];  // [gate/up][element]
};

// One consumer warp's work on one pipeline stage (256 k) for one 16-row tile
// of NVFP4 weights. BF = false: f16 MMA on the prescaled activations (every value of the chunk
// exact in f16). BF = true: bf16 MMA on the raw bf16 activations, used for a
// chunk whose values do not all fit one f16 exponent window; the decoded
// weights are exact in bf16 as well, so the products stay exact.
template <int EPI, bool BF>
__device__ __forceinline__ void tile_stage(const DenseArgs& a, uint32_t sb, uint32_t xb, uint32_t sm_base, int jsub,
                                           int kk0, int ti, int lane, const int* xexp, int ntok, TileAcc& acc)
{
    constexpr int NGU = (EPI == EPI_SWIGLU) ? 2 : 1;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int p0 = xexp[jsub * 8 + 2 * t];
    const int p1 = xexp[jsub * 8 + 2 * t + 1];

    // four independent accumulator chains per gate/up tile (chunk x MMA half)
    float d[2][2][4];
    float d2[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[i][j][e] = d2[i][j][e] = 0.f;

    const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ms = 0; ms < 4; ++ms) {
        uint4 bx[2];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const int kk = kk0 + 64 * ms + 32 * ch + 8 * t;
            bx[ch] = g < ntok ? lds128(xb + (g * a.x_pitch + kk) * 2) : make_uint4(0, 0, 0, 0);
        }
        // ldmatrix: lane l supplies row (l & 7) + 8 * ((l >> 3) & 1) of the tile and
        // 16-byte chunk 2 * ms + (l >> 4); chunk c of row r sits at c ^ (r & 7).
        const int lc = 2 * ms + (lane >> 4);
        const uint32_t lofs = (16 * ti + lr) * 128 + ((lc ^ (lr & 7)) << 4);
#pragma unroll
        for (int gu = 0; gu < NGU; ++gu) {
            uint32_t cr[4];
            ldmatrix_x4(cr, sb + (gu ? a.st.codes2 : a.st.codes) + lofs);
            // cr[0]: row g chunk 2ms; cr[1]: row g+8 chunk 2ms; cr[2], cr[3]: chunk 2ms+1.
            // Each register holds the 8 codes of k = 32 * chunk + 8t .. 8t+7.
            {
                const uint32_t sbase = sb + (gu ? a.st.scales2 : a.st.scales);
                const uint32_t sw_g = lds32(sbase + (16 * ti + g) * 16 + 4 * ms);
                const uint32_t sw_g8 = lds32(sbase + (16 * ti + g + 8) * 16 + 4 * ms);
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    // 16-k block 4ms + 2ch + (t>>1): its E4M3 byte duplicated, then
                    // converted, gives the scale already broadcast to both halves.
                    const uint32_t sel = static_cast<uint32_t>((2 * ch + (t >> 1)) * 0x11);
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
                    const uint4 bb = bx[ch];
                    const uint32_t A0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
                    const uint32_t A1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
                    if (BF) {
                        mma_bf16_16816(d[gu][ch], A0, bb.x, bb.y);
                        mma_bf16_16816(d2[gu][ch], A1, bb.z, bb.w);
                    } else {
                        mma_f16_16816(d[gu][ch], A0, bb.x, bb.y);
                        mma_f16_16816(d2[gu][ch], A1, bb.z, bb.w);
                    }
                }
            }
        }
    }
    // fold the chunk partial into the accumulator: value = d * 2^-p per token column
    const int e0 = BF ? 0 : p0, e1 = BF ? 0 : p1;
#pragma unroll
    for (int gu = 0; gu < NGU; ++gu) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float part = (d[gu][0][e] + d2[gu][0][e]) + (d[gu][1][e] + d2[gu][1][e]);
            acc.v[gu][e] += ldexp_exact(part, (e & 1) ? -e1 : -e0);
        }
    }
}

// One consumer warp's work on one pipeline stage (256 k) for one 16-row tile
// of Q4/Q5 weights. The codes are small integers, exact in bf16, so the MMAs
// run in bf16 on the raw bf16 activations the stage carries (no prescale):
// per 32-k group, sum(q x) from the codes and sum(x) from an MMA of all-ones
// rows, which lands in the same fragment layout; then
// y += scale * sum(q x) + min * sum(x).
template <int FMT>
__device__ __forceinline__ void tile_stage_q(const DenseArgs& a, uint32_t sb, int ti, int lane, int ntok,
                                             TileAcc& acc)
{
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint4 qs_g = lds128(sb + a.st.scales + (16 * ti + g) * 16);
    const uint4 qs_g8 = lds128(sb + a.st.scales + (16 * ti + g + 8) * 16);
    const uint4 qm_g = lds128(sb + a.st.mins + (16 * ti + g) * 16);
    const uint4 qm_g8 = lds128(sb + a.st.mins + (16 * ti + g + 8) * 16);
    constexpr uint32_t kOnes = 0x3F803F80u;  // bf16 pair (1, 1)
    const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
    float d[2][4];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[ch][e] = 0.f;

    const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ms = 0; ms < 4; ++ms) {
        // token g's 8 activations at k = 64 ms + 32 ch + 8 t, as the pairs
        // (k, k+4) (k+1, k+5) (k+2, k+6) (k+3, k+7) the code decode produces
        uint4 bx[2];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const uint4 v = g < ntok ? lds128(sb + a.st.x + g * 512 + (64 * ms + 32 * ch + 8 * t) * 2)
                                     : make_uint4(0, 0, 0, 0);
            bx[ch] = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
        }
        const int lc = 2 * ms + (lane >> 4);
        const uint32_t lofs = (16 * ti + lr) * 128 + ((lc ^ (lr & 7)) << 4);
        uint32_t cr[4];
        ldmatrix_x4(cr, sb + a.st.codes + lofs);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            const int grp = 2 * ms + ch;  // 32-k group inside the chunk
            const uint32_t rg = cr[2 * ch], rg8 = cr[2 * ch + 1];
            uint32_t hg = 0, hg8 = 0;
            if (FMT == FMT_Q5) {
                const uint32_t h0 = lds8(sb + a.st.hi + (16 * ti + g) * 32 + 4 * grp + t);
                const uint32_t h1 = lds8(sb + a.st.hi + (16 * ti + g + 8) * 32 + 4 * grp + t);
                hg = (h0 << 4) | (h0 << 16);
                hg8 = (h1 << 4) | (h1 << 16);
            }
            // pair {q(8t+i), q(8t+i+4)}: bf16 128 + q, minus 128
            constexpr uint32_t kMagic = 0x43004300u;
            uint32_t q0[4], q8[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t u = ((rg >> (4 * i)) & 0x000F000Fu) | kMagic;
                uint32_t u8 = ((rg8 >> (4 * i)) & 0x000F000Fu) | kMagic;
                if (FMT == FMT_Q5) {
                    u |= (hg >> i) & 0x00100010u;
                    u8 |= (hg8 >> i) & 0x00100010u;
                }
                q0[i] = bsub2(u, kMagic);
                q8[i] = bsub2(u8, kMagic);
            }
            const uint4 bb = bx[ch];
            const uint32_t A0[4] = {q0[0], q8[0], q0[1], q8[1]};
            const uint32_t A1[4] = {q0[2], q8[2], q0[3], q8[3]};
            float dg[4] = {0.f, 0.f, 0.f, 0.f};
            float ds[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16_16816(dg, A0, bb.x, bb.y);
            mma_bf16_16816(dg, A1, bb.z, bb.w);
            mma_bf16_16816(ds, ones, bb.x, bb.y);
            mma_bf16_16816(ds, ones, bb.z, bb.w);
            const uint32_t sv_g = (&qs_g.x)[grp >> 1], sv_g8 = (&qs_g8.x)[grp >> 1];
            const uint32_t mv_g = (&qm_g.x)[grp >> 1], mv_g8 = (&qm_g8.x)[grp >> 1];
            const int sh = (grp & 1) * 16;
            const float s0 = half_bits_to_f32((sv_g >> sh) & 0xFFFFu);
            const float s8 = half_bits_to_f32((sv_g8 >> sh) & 0xFFFFu);
            const float m0 = half_bits_to_f32((mv_g >> sh) & 0xFFFFu);
            const float m8 = half_bits_to_f32((mv_g8 >> sh) & 0xFFFFu);
            // ds[e]: sum of x over the group for token column 2t + (e & 1)
            float* dd = d[ch];
            dd[0] = fmaf(m0, ds[0], fmaf(s0, dg[0], dd[0]));
            dd[1] = fmaf(m0, ds[1], fmaf(s0, dg[1], dd[1]));
            dd[2] = fmaf(m8, ds[2], fmaf(s8, dg[2], dd[2]));
            dd[3] = fmaf(m8, ds[3], fmaf(s8, dg[3], dd[3]));
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc.v[0][e] += d[0][e] + d[1][e];
}

// Unit of work: rows [w_row0, w_row0 + rows) of the weight tensor (gate rows
// for SwiGLU; the up rows follow at + up_row_offset) against one group of
// activation rows, written to output columns out_col0 + r.
struct Unit {
    int w_row0;
    int rows;
    int out_col0;
    int grp;
};

__device__ __forceinline__ Unit load_unit(const DenseArgs& a, int u)
{
    Unit un;
    if (a.units == nullptr) {
        un.w_row0 = u * a.rows_per_cta;
        un.rows = min(a.rows_per_cta, a.n_out - un.w_row0);
        un.out_col0 = un.w_row0;
        un.grp = 0;
    } else {
        const UnitDesc d = a.units[u];
        un.w_row0 = d.w_row0;
        un.rows = d.rows;
        un.out_col0 = d.out_col0;
        un.grp = d.grp;
    }
    return un;
}

// Units of this CTA: dense launches own exactly one (blockIdx.x); grouped
// launches split the device-side unit list into contiguous ranges so that
// consecutive units mostly share their group (and its converted activations).
__device__ __forceinline__ void unit_range(const DenseArgs& a, int& u_begin, int& u_end)
{
    if (a.units == nullptr) {
        u_begin = blockIdx.x;
        u_end = blockIdx.x + 1;
    } else {
        const int n = *a.n_units;
        u_begin = static_cast<int>((static_cast<long long>(n) * blockIdx.x) / gridDim.x);
        u_end = static_cast<int>((static_cast<long long>(n) * (blockIdx.x + 1)) / gridDim.x);
    }
}

template <int FMT, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ DenseArgs a, const __grid_constant__ CUtensorMap tm0,
                const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm2,
                const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tmx)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int NGU = (EPI == EPI_SWIGLU) ? 2 : 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_chunks = a.K / kChunkK;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMaxStages);

    // Let the next kernel on the stream be scheduled as soon as SMs free up
    // (programmatic dependent launch); it waits for this grid before it reads
    // anything this grid writes.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Every stage is consumed by one warp per 16-row tile of a full unit.
    const int T = (a.rows_per_cta + 15) >> 4;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], T);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // Grouped launches read their unit list from the previous kernel's output.
    if (a.units != nullptr) asm volatile("griddepcontrol.wait;" ::: "memory");
    int u_begin, u_end;
    unit_range(a, u_begin, u_end);

    // ------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            prefetch_tensormap(&tm0);
            prefetch_tensormap(&tm1);
            if (FMT != FMT_NVFP4) prefetch_tensormap(&tm2);
            if (FMT == FMT_Q5) prefetch_tensormap(&tm3);
            if (FMT != FMT_NVFP4) prefetch_tensormap(&tmx);
            int gc = 0;  // global stage counter across units
            bool stop = false;
            // Q4/Q5 stages carry their activations, which may come from the
            // previous kernel: weight copies start at once, the activation
            // copies of the stages issued so far follow the dependency wait
            // (before the first wait for a free slot, so no stage is left
            // without its activations).
            bool x_ready = FMT == FMT_NVFP4;
            auto x_backfill = [&]() {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                for (int s = max(0, gc - a.n_stages); s < gc; ++s)
                    tma_load_2d(smem + a.smem_ring + (s % a.n_stages) * a.st.bytes + a.st.x, &tmx,
                                (s % n_chunks) * kChunkK, 0, &full[s % a.n_stages]);
                x_ready = true;
            };
            for (int u = u_begin; u < u_end && !stop; ++u) {
                const Unit un = load_unit(a, u);
                for (int c = 0; c < n_chunks; ++c, ++gc) {
                    const int slot = gc % a.n_stages;
                    if (gc >= a.n_stages && !x_ready) x_backfill();
                    if (gc >= a.n_stages) {
                        if (!mbar_wait_bounded(&empty[slot], ((gc / a.n_stages) - 1) & 1, a.wait_ns, a.status)) {
                            *abort_flag = 1;
                            stop = true;
                            break;
                        }
                    }
                    if (*abort_flag || a.starve) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[slot], a.st.tx_bytes);
                    uint8_t* sb = smem + a.smem_ring + slot * a.st.bytes;
                    const int kb = c * kChunkK;
                    tma_load_2d(sb + a.st.codes, &tm0, kb / 2, un.w_row0, &full[slot]);
                    if (FMT == FMT_NVFP4) {
                        tma_load_2d(sb + a.st.scales, &tm1, kb / 16, un.w_row0, &full[slot]);
                        if (EPI == EPI_SWIGLU) {
                            tma_load_2d(sb + a.st.codes2, &tm0, kb / 2, un.w_row0 + a.up_row_offset, &full[slot]);
                            tma_load_2d(sb + a.st.scales2, &tm1, kb / 16, un.w_row0 + a.up_row_offset, &full[slot]);
                        }
                    } else {
                        tma_load_2d(sb + a.st.scales, &tm1, kb / 32, un.w_row0, &full[slot]);
                        tma_load_2d(sb + a.st.mins, &tm2, kb / 32, un.w_row0, &full[slot]);
                        if (FMT == FMT_Q5) tma_load_2d(sb + a.st.hi, &tm3, kb / 8, un.w_row0, &full[slot]);
                        if (x_ready) tma_load_2d(sb + a.st.x, &tmx, kb, 0, &full[slot]);
                    }
                }
            }
            if (!x_ready) x_backfill();
            // No copy may still be landing in shared memory when the CTA exits.
            for (int c = max(0, gc - a.n_stages); c < gc; ++c)
                mbar_wait_bounded(&full[c % a.n_stages], (c / a.n_stages) & 1, a.wait_ns, a.status);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    // Warps w = S * tile + slice: the S slices of a tile take the stages
    // c with c % S == slice (consecutive warps sit on different schedulers);
    // slices are summed in a fixed order at the end of each unit.
    const int Tp = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
    const int S = kConsumerWarps / Tp;
    const int slice = warp % S;
    const int my_tile = (warp / S) < T ? (warp / S) : -1;

    const uint32_t sm_base = smem_u32(smem);
    const uint32_t x_base = sm_base + a.smem_x;
    const uint32_t xraw_base = sm_base + a.smem_xraw;
    int* xexp = reinterpret_cast<int*>(smem + a.smem_exp);            // [nsub][8]
    uint8_t* xflag = smem + a.smem_flag;                                // [nsub][8]
    float* xsum = reinterpret_cast<float*>(smem + a.smem_sum);        // [nsub * 8 groups][8]
    float* red = reinterpret_cast<float*>(smem + a.smem_red);
    const int ctid = threadIdx.x;                                       // 0 .. 511 among consumers

    // Activations (and residuals) may come from the previous kernel on the
    // stream: wait for it before touching them. Weight streaming above does
    // not depend on it and is already running.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    bool aborted = false;
    int gc = 0;
    int conv_key = -1;     // activation rows (group xkey) the buffer holds
    int conv_ks0 = -1;     // and the super-chunk start
    for (int u = u_begin; u < u_end; ++u) {
        const Unit un = load_unit(a, u);
        // ---------------- group info of this unit
        int ntok, xkey;
        float gsc;
        if (a.units == nullptr) {
            ntok = a.M;
            gsc = a.g;
            xkey = 0;
        } else {
            ntok = a.groups[un.grp].ntok;
            gsc = a.gscales[a.groups[un.grp].e];
            xkey = a.groups[un.grp].xkey;
        }
        TileAcc acc;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc.v[j][e] = 0.f;

        for (int c = 0; c < n_chunks; ++c, ++gc) {
            const int kglob = c * kChunkK;
            const int ks0 = (kglob / a.ksc) * a.ksc;
            // ---------------- activation super-chunk: prescale, convert, flag
            if (FMT == FMT_NVFP4 && (ks0 != conv_ks0 || xkey != conv_key)) {
                const int len = min(a.ksc, a.K - ks0);
                const int nsub = len / kChunkK;
                const int n_items = nsub * ntok;
                named_barrier_sync(1, 32 * kConsumerWarps);
                // columns >= ntok read zero exponents / flags / sums
                for (int i = ctid; i < nsub * 8; i += 32 * kConsumerWarps) {
                    if ((i & 7) >= ntok) {
                        xexp[i] = 0;
                        xflag[i] = 0;
                    }
                }
                if (FMT != FMT_NVFP4)
                    for (int i = ctid; i < nsub * 64; i += 32 * kConsumerWarps)
                        if ((i & 7) >= ntok) xsum[i] = 0.f;
                for (int base = warp; base < n_items; base += 2 * kConsumerWarps) {
                    uint4 raw[2];
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        const int it = base + uu * kConsumerWarps;
                        raw[uu] = make_uint4(0, 0, 0, 0);
                        if (it < n_items) {
                            const int m = it % ntok, j = it / ntok;
                            const int xr = a.units == nullptr ? m : a.groups[un.grp].x_row[m];
                            raw[uu] = ldg_nc_128(a.x + static_cast<size_t>(xr) * a.K + ks0 + j * kChunkK + lane * 8);
                        }
                    }
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        const int it = base + uu * kConsumerWarps;
                        if (it >= n_items) break;
                        const int m = it % ntok, j = it / ntok;
                        const uint32_t wv[4] = {raw[uu].x, raw[uu].y, raw[uu].z, raw[uu].w};
                        uint32_t hbits[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) hbits[i] = (i & 1) ? (wv[i >> 1] >> 16) : (wv[i >> 1] & 0xFFFFu);
                        // prescale from the largest magnitude (at most 126, so 2^p
                        // is a normal float); exact in f16 if the smallest
                        // nonzero value keeps its 8 bits at or above 2^-24
                        uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu, emax, emin, mag;
#pragma unroll
                        for (int i = 0; i < 4; ++i) bf16_range_acc(wv[i], mx2, mn2);
                        bf16_range_fin(mx2, mn2, emax, emin, mag);
                        mag = __reduce_max_sync(0xffffffffu, mag);
                        emin = __reduce_min_sync(0xffffffffu, emin);
                        const int p = min(prescale_exponent(mag), 126);
                        const bool exact = emin == 255u || static_cast<int>(emin) - 127 + p >= -17;
                        const float sp = __int_as_float((127 + p) << 23);
                        uint32_t h[8];
                        float ls = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float v = bf16_bits_to_f32(hbits[i]) * sp;
                            h[i] = __half_as_ushort(__float2half_rn(v));
                            ls += v;
                        }
                        const uint32_t off = (static_cast<uint32_t>(m) * a.x_pitch + j * kChunkK + lane * 8) * 2;
                        const uint4 hv = pack_pairs<FMT>(h);
                        const uint4 rv = pack_pairs<FMT>(hbits);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(x_base + off), "r"(hv.x),
                                     "r"(hv.y), "r"(hv.z), "r"(hv.w));
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xraw_base + off), "r"(rv.x),
                                     "r"(rv.y), "r"(rv.z), "r"(rv.w));
                        const bool any_inexact = __any_sync(0xffffffffu, !exact);
                        if (lane == 0) {
                            xexp[j * 8 + m] = p;
                            xflag[j * 8 + m] = any_inexact ? 1 : 0;
                        }
                        if (FMT != FMT_NVFP4) {
                            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
                            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
                            if ((lane & 3) == 0) xsum[(j * 8 + (lane >> 2)) * 8 + m] = ls;
                        }
                    }
                }
                named_barrier_sync(1, 32 * kConsumerWarps);
                conv_ks0 = ks0;
                conv_key = xkey;
            }

            const int slot = gc % a.n_stages;
            if ((c % S) != slice || my_tile < 0) continue;
            if (!aborted && *abort_flag) aborted = true;
            if (!aborted) {
                if (!mbar_wait_bounded(&full[slot], (gc / a.n_stages) & 1, a.wait_ns, a.status)) {
                    aborted = true;
                    *abort_flag = 1;
                }
            }
            if (!aborted && 16 * my_tile < un.rows) {
                const uint32_t sb = sm_base + a.smem_ring + slot * a.st.bytes;
                if constexpr (FMT == FMT_NVFP4) {
                    const int jsub = (kglob - ks0) / kChunkK;
                    const uint64_t flags8 = *reinterpret_cast<const uint64_t*>(xflag + jsub * 8);
                    const int kk0 = kglob - ks0;
                    if (flags8)
                        tile_stage<EPI, true>(a, sb, xraw_base, sm_base, jsub, kk0, my_tile, lane, xexp, ntok, acc);
                    else
                        tile_stage<EPI, false>(a, sb, x_base, sm_base, jsub, kk0, my_tile, lane, xexp, ntok, acc);
                } else {
                    tile_stage_q<FMT>(a, sb, my_tile, lane, ntok, acc);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---------------- cross-slice reduction (fixed order) and epilogue
        if (S > 1) {
            named_barrier_sync(1, 32 * kConsumerWarps);
            if (slice > 0 && my_tile >= 0) {
#pragma unroll
                for (int gu = 0; gu < NGU; ++gu)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        red[(((slice * Tp + my_tile) * 2 + gu) * 32 + lane) * 4 + e] = acc.v[gu][e];
            }
            named_barrier_sync(1, 32 * kConsumerWarps);
            if (slice == 0 && my_tile >= 0) {
                for (int s = 1; s < S; ++s)
#pragma unroll
                    for (int gu = 0; gu < NGU; ++gu)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc.v[gu][e] += red[(((s * Tp + my_tile) * 2 + gu) * 32 + lane) * 4 + e];
            }
        }
        if (slice == 0 && !aborted && my_tile >= 0) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * my_tile + g + ((e & 2) ? 8 : 0);
                const int col = 2 * t + (e & 1);
                if (r >= un.rows || col >= ntok) continue;
                const int orow = a.units == nullptr ? col : a.groups[un.grp].out_row[col];
                if (orow < 0) continue;
                const size_t o = static_cast<size_t>(orow) * a.out_pitch + un.out_col0 + r;
                float v = acc.v[0][e] * gsc;
                if (EPI == EPI_SWIGLU) {
                    const float uv = acc.v[1][e] * gsc;
                    v = (v / (1.0f + expf(-v))) * uv;
                }
                if (EPI == EPI_RESID) v += bf16_bits_to_f32(a.residual[o]);
                if (a.out_f32)
                    reinterpret_cast<float*>(a.y)[o] = v;
                else
                    reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(v);
            }
        }
    }
}

constexpr uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Fills in the launch-time fields of `a` (status word, debug limits, shared
// memory plan) and launches `grid` CTAs with programmatic dependent launch.
template <int FMT, int EPI>
qg_status launch_gemv_impl(const CUtensorMap* maps, DenseArgs a, int grid, cudaStream_t stream)
{
    const int M = a.M;
    const int K = a.K;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;

    // NVFP4: activation super-chunk, f16 (prescaled) and raw bf16 copies of M
    // token rows of (ksc + 32) values. Q4/Q5: the activations travel with
    // each stage instead.
    constexpr uint32_t kXBudget = 80 * 1024;
    int ksc = (static_cast<int>(kXBudget / (4u * M)) - 32) / kChunkK * kChunkK;
    ksc = min(ksc, K);
    a.ksc = ksc;
    a.x_pitch = FMT == FMT_NVFP4 ? ksc + 32 : 0;
    const int nsub = FMT == FMT_NVFP4 ? ksc / kChunkK : 0;

    const int R = a.rows_per_cta;
    const int R16 = (R + 15) / 16 * 16;  // regions cover whole 16-row tiles
    StageLayout st{};
    uint32_t off = 0;
    st.codes = off;
    off = align_up(off + R16 * 128, 1024);
    if (EPI == EPI_SWIGLU) {
        st.codes2 = off;
        off = align_up(off + R16 * 128, 1024);
    }
    st.scales = off;
    off = align_up(off + R16 * 16, 128);
    if (EPI == EPI_SWIGLU) {
        st.scales2 = off;
        off = align_up(off + R16 * 16, 128);
    }
    if (FMT != FMT_NVFP4) {
        st.mins = off;
        off = align_up(off + R16 * 16, 128);
    }
    if (FMT == FMT_Q5) {
        st.hi = off;
        off = align_up(off + R16 * 32, 128);
    }
    if (FMT != FMT_NVFP4) {
        st.x = off;
        off = align_up(off + static_cast<uint32_t>(M) * kChunkK * 2, 128);
    }
    st.bytes = align_up(off, 1024);
    uint32_t tx = R * 128 + R * 16;
    if (EPI == EPI_SWIGLU) tx *= 2;
    if (FMT != FMT_NVFP4) tx += R * 16 + M * kChunkK * 2;
    if (FMT == FMT_Q5) tx += R * 32;
    st.tx_bytes = tx;
    a.st = st;

    // shared memory plan
    uint32_t so = 0;
    const uint32_t x_bytes = align_up(static_cast<uint32_t>(M) * a.x_pitch * 2, 128);
    const uint32_t exp_bytes = align_up(nsub * 8 * 4, 128);
    const uint32_t flag_bytes = align_up(nsub * 8, 128);
    const uint32_t sum_bytes = 0;
    const uint32_t red_bytes = kConsumerWarps * 2 * 32 * 4 * 4;
    const uint32_t bar_bytes = 2 * kMaxStages * 8 + 16;
    const uint32_t fixed = 2 * x_bytes + exp_bytes + flag_bytes + sum_bytes + red_bytes + bar_bytes;
    const uint32_t smem_max = 227 * 1024;
    if (fixed + st.bytes > smem_max) return QG_ERR_UNSUPPORTED;
    int n_stages = static_cast<int>((smem_max - fixed) / st.bytes);
    n_stages = min(n_stages, kMaxStages);
    n_stages = min(n_stages, K / kChunkK);
    if (n_stages < 2 && K / kChunkK >= 2) return QG_ERR_UNSUPPORTED;
    a.n_stages = max(n_stages, 1);
    a.smem_ring = so;
    so += a.n_stages * st.bytes;
    a.smem_x = so;
    so += x_bytes;
    a.smem_xraw = so;
    so += x_bytes;
    a.smem_exp = so;
    so += exp_bytes;
    a.smem_flag = so;
    so += flag_bytes;
    a.smem_sum = so;
    so += sum_bytes;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    so += bar_bytes;

    auto kern = gemv_kernel<FMT, EPI>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = so;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, a, maps[0], maps[1], maps[2], maps[3], maps[4]) != cudaSuccess)
        return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

int choose_rows_per_cta(int n_out, int factor)
{
    const int sms = sm_count(-1);
    int R = (n_out + sms - 1) / sms;
    R = max(R, 16);
    R = min(R, kMaxRowsPerCta / factor);
    return R;
}

DenseArgs dense_args(const void* x, void* y, int out_f32, const void* residual, int M, int n_out, int up_offset,
                     int K, float g, int R)
{
    DenseArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.residual = static_cast<const uint16_t*>(residual);
    a.M = M;
    a.K = K;
    a.n_out = n_out;
    a.out_pitch = n_out;
    a.rows_per_cta = R;
    a.up_row_offset = up_offset;
    a.out_f32 = out_f32;
    a.g = g;
    return a;
}

}  // namespace

qg_status launch_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                             int out_f32, const void* residual, int M, int N, int K, int swiglu,
                             cudaStream_t stream)
{
    const int n_out = swiglu ? N / 2 : N;
    const int R = choose_rows_per_cta(n_out, 1);
    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (!encode_tmap_2d(&maps[0], codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, R, true)) return QG_ERR_CUDA;
    if (!encode_tmap_2d(&maps[1], scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, N, 16, R, false))
        return QG_ERR_CUDA;
    maps[2] = maps[1];
    maps[3] = maps[1];
    maps[4] = maps[1];
    const int grid = (n_out + R - 1) / R;
    if (swiglu)
        return launch_gemv_impl<FMT_NVFP4, EPI_SWIGLU>(maps, dense_args(x, y, 0, nullptr, M, n_out, n_out, K, g, R),
                                                       grid, stream);
    if (residual)
        return launch_gemv_impl<FMT_NVFP4, EPI_RESID>(maps, dense_args(x, y, out_f32, residual, M, n_out, 0, K, g, R),
                                                      grid, stream);
    return launch_gemv_impl<FMT_NVFP4, EPI_NONE>(maps, dense_args(x, y, out_f32, nullptr, M, n_out, 0, K, g, R), grid,
                                                 stream);
}

qg_status launch_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min,
                           int bits, const void* x, void* y, int out_f32, const void* residual, int M,
                           int N, int K, cudaStream_t stream)
{
    const int R = choose_rows_per_cta(N, 1);
    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (!encode_tmap_2d(&maps[0], q_lo, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, N, 128, R, true)) return QG_ERR_CUDA;
    if (!encode_tmap_2d(&maps[1], scale, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false))
        return QG_ERR_CUDA;
    if (!encode_tmap_2d(&maps[2], min, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K / 32, N, 8, R, false))
        return QG_ERR_CUDA;
    if (bits == 5) {
        if (!encode_tmap_2d(&maps[3], q_hi, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, N, 32, R, false))
            return QG_ERR_CUDA;
    } else {
        maps[3] = maps[2];
    }
    // the M activation rows, one 256-k chunk per stage
    if (!encode_tmap_2d(&maps[4], x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, K, M, kChunkK, M, false)) return QG_ERR_CUDA;
    const int grid = (N + R - 1) / R;
    const DenseArgs a = dense_args(x, y, out_f32, residual, M, N, 0, K, 1.f, R);
    if (bits == 5) {
        if (residual) return launch_gemv_impl<FMT_Q5, EPI_RESID>(maps, a, grid, stream);
        return launch_gemv_impl<FMT_Q5, EPI_NONE>(maps, a, grid, stream);
    }
    if (residual) return launch_gemv_impl<FMT_Q4, EPI_RESID>(maps, a, grid, stream);
    return launch_gemv_impl<FMT_Q4, EPI_NONE>(maps, a, grid, stream);
}

qg_status launch_grouped_nvfp4(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu,
                               int up_offset, const void* x, int max_cols, void* y, int out_pitch, int out_f32,
                               const GroupDesc* groups, const UnitDesc* units, const int* n_units,
                               const float* gscales, int rows_per_unit, cudaStream_t stream)
{
    const int R = rows_per_unit;
    CUtensorMap maps[5];
    memset(maps, 0, sizeof(maps));
    if (!encode_tmap_2d(&maps[0], codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, total_rows, 128, R, true))
        return QG_ERR_CUDA;
    if (!encode_tmap_2d(&maps[1], scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, total_rows, 16, R, false))
        return QG_ERR_CUDA;
    maps[2] = maps[1];
    maps[3] = maps[1];
    maps[4] = maps[1];
    DenseArgs a = dense_args(x, y, out_f32, nullptr, max_cols, 0, up_offset, K, 1.f, R);
    a.out_pitch = out_pitch;
    a.groups = groups;
    a.units = units;
    a.n_units = n_units;
    a.gscales = gscales;
    const int grid = sm_count(-1);
    if (swiglu) return launch_gemv_impl<FMT_NVFP4, EPI_SWIGLU>(maps, a, grid, stream);
    return launch_gemv_impl<FMT_NVFP4, EPI_NONE>(maps, a, grid, stream);
}

}  // namespace qg
