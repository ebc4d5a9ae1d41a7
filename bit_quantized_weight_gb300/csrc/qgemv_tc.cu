// qgemv_tc.cu -- NVFP4 decode GEMV / skinny GEMM (M = 1..8 tokens) on the
// 5th-generation tensor cores (tcgen05), with fused residual-add and SwiGLU
// epilogues, for dense layers and for expert-gathered MoE units.
//
// The pages' NVFP4 format (NVIDIA NVFP4 blog, "How NVFP4 works": E2M1 codes,
// one E4M3 scale per 16 values, one FP32 tensor scale) and the decode-GEMV
// fusions (NInfer article, section 2: one fused matmul + residual / SwiGLU
// kernel per weight format, decode being bandwidth bound) fix what is
// computed; the layout below is designed for sm_103a.
//
// Work split. A CTA owns units of R output rows (the gate rows and up rows of
// a SwiGLU pair count as two rows each) and streams all of K for them. The
// 128 TMEM lanes hold (row, gate/up, K-phase) triples: the K range is cut into
// P contiguous phases, so that even a CTA with 34 rows keeps ~100 lanes -- and
// all four SM sub-partitions -- busy. Every weight byte crosses HBM once.
//
// Pipeline. One warp streams, per 256-k chunk of every phase (a stage), the
// codes (128B-swizzled) and scales of each (phase, gate/up) box into a ring of
// shared-memory stages with 2-D TMA loads. A stage is worked on in two 128-k
// granules; granule g belongs to decode set g % 4 and passes through three
// roles:
//   * the set's four decode warps (one per TMEM lane quadrant) turn codes
//     into f16 with cvt.rn.f16x2.e2m1x2 (exact) and store them to the set's
//     TMEM buffer with tcgen05.st: TMEM lane = the triple, 32-bit column =
//     two consecutive k;
//   * the set's MMA warp (one per set, each on its own SM sub-partition)
//     issues eight tcgen05.mma (M = 128, K = 16) with the activations as the
//     shared-memory B operand;
//   * four fold warps (one per quadrant, every granule in order) read D back
//     with tcgen05.ld, free the buffer and accumulate in fp32; they own the
//     per-unit reduction and epilogue, which thus overlaps the next unit.
// The roles meet only at per-buffer mbarriers ("A written", "MMA done", "D
// read"), and every synchronisation covers a whole 128-k granule: an mbarrier
// round trip costs about as much as decoding 32 k. Before the first stage
// (and whenever the activations no longer fit in shared memory, per
// super-chunk) the decode warps convert the activations into the B layout.
//
// The E4M3 block scale is applied in one of two exact ways:
//   * one token (M = 1): after the MMA, in fp32. Four 16-k blocks share one
//     16-column D region: block j's B operand holds the P phase rows in rows
//     4j .. 4j+3 and zeros elsewhere, so the four chained MMAs leave block j's
//     sums in columns 4j + phase. The lane folds scale * D for all four phase
//     columns and keeps its own phase's sum at the end, so the per-weight work
//     is the code conversion alone;
//   * 2..8 tokens: before the MMA, on the f16 weights (e2m1 * e4m3 has at
//     most 6 significant bits and lies in [2^-10, 2688], so the f16 product
//     is exact), the eight blocks of a granule chained into one D region --
//     cheaper than one fp32 multiply-add per block and token.
// Activations enter the MMA as f16 after an exact power-of-two prescale per
// (token, 256-k chunk) that puts the chunk maximum in [2^14, 2^15); a stage
// where some chunk's smallest nonzero value lies too far below its maximum
// for f16 to hold it exactly under that scale runs in bf16 on the raw
// activations instead (weights are exact in both). Products are therefore
// exact and the accumulation is fp32.
//
// Determinism: every sum runs in a fixed order (MMA chains, granules in k
// order per fold warp, then fold warps and phases in index order). Results for
// a token do not depend on how many other tokens share the call, from 2 to 8
// tokens; a single-token call differs from those only by fp32 rounding.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace qg {

namespace {

constexpr int kTcDecodeSets = 4;                    // decode warp sets; set s takes granules g % 4 == s
constexpr int kTcDecodeWarps = 4 * kTcDecodeSets;   // warps 0-15: quadrant w % 4, set w / 4
constexpr int kTcDecodeThreads = 32 * kTcDecodeWarps;
constexpr int kTcFoldWarps = 4;                     // warps 16-19: quadrant w % 4, every granule
constexpr int kTcFoldThreads = 32 * kTcFoldWarps;
constexpr int kTcMmaWarp0 = kTcDecodeWarps + kTcFoldWarps;  // warps 20-23: MMA issue for decode set w - 20
constexpr int kTcTmaWarp = kTcMmaWarp0 + kTcDecodeSets;
constexpr int kTcThreads = 32 * (kTcTmaWarp + 1);
constexpr int kTcMaxStages = 24;
constexpr int kTcCols = 512;                        // TMEM columns allocated (all of them)
constexpr int kTcMaxBufs = 4;                       // TMEM buffers in rotation, one per decode set
constexpr int kTcGran = 2;                          // 128-k granules per 256-k stage
constexpr uint32_t kTcZeroPad = 256;                // zero bytes before and after the one-token B layout
constexpr uint32_t kTcSmemMax = 227u * 1024u;
constexpr uint32_t kTcSmemMin = 120u * 1024u;       // keeps one CTA per SM (TMEM is not shared)

struct TcArgs {
    const uint16_t* x;         // bf16 activations, rows of K values
    void* y;                   // output rows of out_pitch values
    const uint16_t* residual;  // bf16, same layout as y, or nullptr
    int M;                     // dense: tokens; grouped: max columns per group
    int K;
    int C;                     // K / 256
    int n_out;                 // dense: output columns
    int out_pitch;
    int R;                     // rows per unit
    int R8;                    // R rounded up to 8: row stride of a box in shared memory
    int P;                     // K phases
    int Cp;                    // 256-k stages per phase
    int SC;                    // stages per activation super-chunk
    int PES;                   // prescale factors per stage (P * MT, or 4 for one token)
    int up_row_offset;         // SwiGLU: up row = gate row + this
    int out_f32;
    float g;
    int n_units;               // dense launches
    const GroupDesc* groups;   // grouped launches (nullptr for dense)
    const UnitDesc* units;
    const int* n_units_dev;
    const float* gscales;
    int n_stages;
    uint32_t stage_bytes;
    uint32_t scales_off;       // scales boxes inside a stage
    uint32_t box_tx;           // bytes one (phase, gate/up) box pair brings in
    uint32_t smem_ring;
    uint32_t smem_z;           // activations as MMA B operand
    uint32_t z_bytes;
    uint32_t smem_ex;          // prescale exponent per (stage, phase, token), int
    uint32_t smem_fl;          // inexact flag per (stage, phase, token)
    uint32_t smem_fs;          // bf16 stage flag per stage
    uint32_t smem_pe;          // 2^-exponent per (stage, phase, token), fp32, PES per stage
    uint32_t smem_red;
    uint32_t smem_bar;
    // RMSNorm prologue (dense launches; norm_w == nullptr: none): the MMA
    // reads h = bf16(x * r_m * gamma) with r_m = 1 / sqrt(mean(x_m^2) + eps)
    const uint16_t* norm_w;
    float norm_eps;
    uint32_t smem_rms;         // M * C chunk sums of squares, then r_m [8]
    uint64_t wait_ns;
    int starve;
    int* status;
};

template <int MT, int EPI>
struct TcCfg {
    static constexpr int NGU = (EPI == EPI_SWIGLU) ? 2 : 1;
    static constexpr bool DEF = (MT == 1);             // block scale applied after the MMA
    static constexpr int W = 4 * MT;                   // D columns of all phases (P <= 4)
    static constexpr int N = W < 16 ? 16 : W;          // MMA n
    static constexpr int STEPS = 8;                    // MMAs (16-k blocks) per granule
    static constexpr int ACOLS = 64;                   // A columns per granule
    static constexpr int DREG = DEF ? 2 : 1;           // D regions per granule
    static constexpr int BUFC = ACOLS + DREG * N;      // TMEM columns per buffer
    // One buffer per decode set: buffer b = granule % 4 then always belongs to
    // the same decode set, fold parity and MMA warp, so each mbarrier of a
    // buffer has one waiting warp per role, which consumes its phases in order
    // (a parity wait for phase k is only sound once phase k - 1 has completed).
    static constexpr int NB = kTcMaxBufs;
    static_assert(NB * BUFC <= kTcCols && NB % kTcDecodeSets == 0, "buffers per decode set");
    static_assert(kTcGran == 2, "granule parity = granule index within the stage");
    static_assert(kTcGran * STEPS * 16 == kChunkK, "granules tile a stage");
};

struct TcUnit {
    int w_row0;
    int rows;
    int out_col0;
    int grp;
};

__device__ __forceinline__ TcUnit tc_unit(const TcArgs& a, int u)
{
    TcUnit un;
    if (a.units == nullptr) {
        un.w_row0 = u * a.R;
        un.rows = min(a.R, a.n_out - un.w_row0);
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

// Dense launches deal units round-robin; grouped launches give each CTA a
// contiguous range, so that consecutive units mostly share a group and its
// converted activations.
__device__ __forceinline__ void tc_unit_range(const TcArgs& a, int& begin, int& end, int& stride)
{
    if (a.units == nullptr) {
        begin = blockIdx.x;
        end = a.n_units;
        stride = gridDim.x;
    } else {
        const int n = *a.n_units_dev;
        begin = static_cast<int>((static_cast<long long>(n) * blockIdx.x) / gridDim.x);
        end = static_cast<int>((static_cast<long long>(n) * (blockIdx.x + 1)) / gridDim.x);
        stride = 1;
    }
}

// Bounded mbarrier wait that also gives up as soon as another role of the CTA
// has aborted. Each try sleeps until the phase completes or ~20 us pass, so a
// waiting role takes no issue slots from the others on its sub-partition.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const TcArgs& a, volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > a.wait_ns) {
            set_device_status(a.status, QG_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// The same wait for all 32 lanes of a warp with one outcome for all of them
// (the tcgen05 instructions that follow are warp-collective).
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, const TcArgs& a,
                                             volatile int* abort_flag)
{
    return __all_sync(0xffffffffu, tc_wait(bar, parity, a, abort_flag));
}

// ---------------------------------------------------------------- B layouts
// Rows of 16 bytes, 8 consecutive k each. s = MMA step (16-k block) within the
// super-chunk, kg = which 8 k of the block; the conversion's lane L of stage
// cr covers step 16 cr + L / 2, kg = L % 2, i.e. "piece" 32 cr + L.
//
// Several tokens: B row n = phase * MT + token of piece (s, kg) is Z row
// (2 s + kg) * P * MT + n; one K-major core matrix (8 rows, 16 bytes apart)
// is 8 consecutive Z rows: leading byte offset (k direction) P*MT*16, stride
// byte offset (n direction) 128. Rows n >= P*MT read neighbouring data and
// only produce D columns whose sums are never kept.
//
// One token: piece (s, kg) is an 8-row pattern [0, 0, 0, 0, x_p0, x_p1, x_p2,
// x_p3] (phases >= P zero), patterns back to back after kTcZeroPad zero bytes
// and followed by kTcZeroPad more. Block j of a four-block group reads B rows
// 4j .. 4j+3 = the four phase rows, all other rows zero: core matrices are 8
// rows, so rows 0-7 come from (start) and rows 8-15 from (start + SBO), the k
// halves LBO = 128 bytes apart:
//   j = 0: start = pattern + 64 (x rows, then the next pattern's zero rows),
//          start + SBO = the trailing zero pad;
//   j = 1: start = pattern, start + SBO = the trailing zero pad;
//   j = 2: start = the leading zero pad, start + SBO = pattern + 64;
//   j = 3: start = the leading zero pad, start + SBO = pattern.
__device__ __forceinline__ uint32_t z_row_multi(int cr, int lane8, int PM, int n)
{
    return static_cast<uint32_t>((32 * cr + lane8) * PM + n);
}

__device__ __forceinline__ uint32_t z_off_one(int cr, int lane8, int p)
{
    return kTcZeroPad + static_cast<uint32_t>(32 * cr + lane8) * 128u + static_cast<uint32_t>(4 + p) * 16u;
}

// ---------------------------------------------------------------- activations
// Converts stages [c0, c0 + nst) of every phase for the current group into the
// B layout, run by the decode warps. Per (stage, phase, token) chunk of 256
// activations one warp (8 per lane, loads of several chunks in flight):
//   * reduces the largest and the smallest nonzero bf16 exponent field over
//     the chunk (finite values only); the prescale exponent e puts the
//     largest magnitude in [2^14, 2^15) (at most 126, so 2^-e stays normal);
//   * the chunk is exact in f16 under 2^e if its smallest nonzero value keeps
//     all 8 significant bits at or above 2^-24, i.e. scaled exponent >= -17
//     (a sufficient test; a chunk failing it is flagged);
//   * writes v * 2^e as f16 (an exact multiply, then an exact conversion)
//     and the factor 2^-e.
// If any chunk was flagged, a second pass rewrites every chunk of the stages
// that hold one as raw bf16 with factor 1 and marks those stages bf16.
// The RMSNorm factors r_m of the M tokens (dense launches), by the decode
// warps: every (token, chunk) sum of squares in the order all kernels share
// (8 values per lane, a warp butterfly), then each token's chunks in k order.
__device__ void tc_norm_factors(const TcArgs& a, uint8_t* smem, int warp, int lane)
{
    float* part = reinterpret_cast<float*>(smem + a.smem_rms);
    float* r = part + a.M * a.C;
    for (int it = warp; it < a.M * a.C; it += kTcDecodeWarps) {
        const int m = it / a.C, kc = it % a.C;
        const float ss = rms_chunk_ss(ldg_nc_128(a.x + static_cast<size_t>(m) * a.K + kc * kChunkK + lane * 8));
        if (lane == 0) part[it] = ss;
    }
    named_barrier_sync(1, kTcDecodeThreads);
    if (threadIdx.x < static_cast<unsigned>(a.M)) {
        float t = 0.f;
        for (int kc = 0; kc < a.C; ++kc) t += part[threadIdx.x * a.C + kc];
        r[threadIdx.x] = rms_factor(t, a.K, a.norm_eps);
    }
    named_barrier_sync(1, kTcDecodeThreads);
}

template <int MT, bool NORM>
__device__ void tc_convert(const TcArgs& a, uint8_t* smem, int c0, int nst, int ntok, const int* xrow, int warp,
                           int lane)
{
    const float* rnorm = reinterpret_cast<const float*>(smem + a.smem_rms) + a.M * a.C;
    constexpr bool DEF = (MT == 1);
    constexpr int kBatch = 4;  // chunks whose loads are in flight together, per warp
    int* any_flag = reinterpret_cast<int*>(smem + a.smem_ex);
    uint8_t* fl = smem + a.smem_fl;
    int* fs = reinterpret_cast<int*>(smem + a.smem_fs);
    float* pe = reinterpret_cast<float*>(smem + a.smem_pe);
    const uint32_t zb = smem_u32(smem + a.smem_z);
    const int PM = a.P * MT;
    const int items = nst * PM;
    // chunk `it` = (stage cr, phase p, token m); this lane's 8 k of it
    auto slot_of = [&](int it) -> uint32_t {
        const int m = it % MT;
        const int t = it / MT;
        const int pp = t % a.P;
        const int cr = t / a.P;
        return DEF ? zb + z_off_one(cr, lane, pp) : zb + z_row_multi(cr, lane, PM, pp * MT + m) * 16u;
    };
    auto load = [&](int it) -> uint4 {
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (it < items) {
            const int m = it % MT;
            const int t = it / MT;
            const int kc = (t % a.P) * a.Cp + c0 + t / a.P;
            if (m < ntok && kc < a.C) {
                const int xr = xrow ? xrow[m] : m;
                raw = ldg_nc_128(a.x + static_cast<size_t>(xr) * a.K + static_cast<size_t>(kc) * kChunkK + lane * 8);
                if (NORM)
                    raw = rms_apply8(raw, ldg_nc_128(a.norm_w + static_cast<size_t>(kc) * kChunkK + lane * 8),
                                     rnorm[m]);
            }
        }
        return raw;
    };

    // factors of phases beyond P (one-token layout) stay zero, as do the
    // one-token layout's padding rows; stages are f16 unless flagged
    for (int i = threadIdx.x; i < nst * a.PES; i += kTcDecodeThreads) pe[i] = 0.f;
    for (int i = threadIdx.x; i < nst; i += kTcDecodeThreads) fs[i] = 0;
    if (threadIdx.x == 0) *any_flag = 0;
    if (DEF)
        for (uint32_t o = threadIdx.x * 16u; o < a.z_bytes; o += kTcDecodeThreads * 16u)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(zb + o), "r"(0u) : "memory");
    named_barrier_sync(1, kTcDecodeThreads);

    bool flagged = false;
    if (!DEF && items >= 4 * kTcDecodeWarps) {
        // Several tokens, many chunks: a warp takes 8 consecutive chunks; lane l holds
        // chunk l % 8 at k-groups l / 8 + 4 i (i < 8), so each reduction runs
        // over four lanes and each store instruction writes 8 different
        // B rows of one k-group -- 8 distinct bank groups.
        const int cl = lane & 7;
        const int kq = lane >> 3;
        for (int g0 = warp * 8; g0 < items; g0 += kTcDecodeWarps * 8) {
            const int it = g0 + cl;
            const bool have = it < items;
            int m = 0, pp = 0, cr = 0, kc = 0;
            if (have) {
                m = it % MT;
                const int t = it / MT;
                pp = t % a.P;
                cr = t / a.P;
                kc = pp * a.Cp + c0 + cr;
            }
            const bool src = have && m < ntok && kc < a.C;
            const uint16_t* xs = a.x;
            if (src) xs += static_cast<size_t>(xrow ? xrow[m] : m) * a.K + static_cast<size_t>(kc) * kChunkK;
            uint4 raw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) raw[i] = src ? ldg_nc_128(xs + (kq + 4 * i) * 8) : make_uint4(0, 0, 0, 0);
            if (NORM && src) {
                const uint16_t* gw = a.norm_w + static_cast<size_t>(kc) * kChunkK;
                uint4 gam[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) gam[i] = ldg_nc_128(gw + (kq + 4 * i) * 8);
#pragma unroll
                for (int i = 0; i < 8; ++i) raw[i] = rms_apply8(raw[i], gam[i], rnorm[m]);
            }
            uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                bf16_range_acc(raw[i].x, mx2, mn2);
                bf16_range_acc(raw[i].y, mx2, mn2);
                bf16_range_acc(raw[i].z, mx2, mn2);
                bf16_range_acc(raw[i].w, mx2, mn2);
            }
            uint32_t emax, emin, magmax;
            bf16_range_fin(mx2, mn2, emax, emin, magmax);
#pragma unroll
            for (int sh = 8; sh <= 16; sh <<= 1) {
                emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, sh));
                emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, sh));
                magmax = max(magmax, __shfl_xor_sync(0xffffffffu, magmax, sh));
            }
            const int e = min(emax != 0u ? 141 - static_cast<int>(emax) : prescale_exponent(magmax), 126);
            const bool inexact = emin != 255u && static_cast<int>(emin) - 127 + e < -17;
            const float sc = __int_as_float((127 + e) << 23);
            if (have) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t wv[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
                    uint32_t o[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        o[w] = pack_f16x2(__uint_as_float(wv[w] << 16) * sc, __uint_as_float(wv[w] & 0xFFFF0000u) * sc);
                    const uint32_t addr = zb + z_row_multi(cr, kq + 4 * i, PM, pp * MT + m) * 16u;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]),
                                 "r"(o[2]), "r"(o[3])
                                 : "memory");
                }
                if (kq == 0) {
                    pe[cr * a.PES + pp * MT + m] = __int_as_float((127 - e) << 23);
                    fl[it] = inexact ? 1 : 0;
                }
            }
            flagged |= have && inexact;
        }
        flagged = __any_sync(0xffffffffu, flagged);
    } else {
    for (int base = warp; base < items; base += kTcDecodeWarps * kBatch) {
        uint4 raw[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) raw[u] = load(base + u * kTcDecodeWarps);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int it = base + u * kTcDecodeWarps;
            if (it >= items) break;
            const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
            uint32_t mx2 = 0, mn2 = 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < 4; ++i) bf16_range_acc(wv[i], mx2, mn2);
            uint32_t emax, emin, magmax;
            bf16_range_fin(mx2, mn2, emax, emin, magmax);
            emax = __reduce_max_sync(0xffffffffu, emax);
            emin = __reduce_min_sync(0xffffffffu, emin);
            // a subnormal largest value needs its full magnitude (rare)
            if (emax == 0u) magmax = __reduce_max_sync(0xffffffffu, magmax);
            const int e = min(emax != 0u ? 141 - static_cast<int>(emax) : prescale_exponent(magmax), 126);
            const bool inexact = emin != 255u && static_cast<int>(emin) - 127 + e < -17;
            const float sc = __int_as_float((127 + e) << 23);
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = pack_f16x2(__uint_as_float(wv[i] << 16) * sc, __uint_as_float(wv[i] & 0xFFFF0000u) * sc);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(slot_of(it)), "r"(o[0]), "r"(o[1]),
                         "r"(o[2]), "r"(o[3])
                         : "memory");
            if (lane == 0) {
                const int m = it % MT;
                const int t = it / MT;
                pe[(t / a.P) * a.PES + (t % a.P) * MT + m] = __int_as_float((127 - e) << 23);
                fl[it] = inexact ? 1 : 0;
            }
            flagged |= inexact;
        }
    }
    }
    if (flagged && lane == 0) *any_flag = 1;
    named_barrier_sync(1, kTcDecodeThreads);
    if (*any_flag != 0) {
        // Rare: stages holding a chunk that f16 cannot carry run in bf16.
        for (int it = warp; it < items; it += kTcDecodeWarps) {
            const int t = it / MT;
            const int cr = t / a.P;
            const bool stage_bf = __any_sync(0xffffffffu, lane < PM && fl[cr * PM + lane] != 0);
            if (!stage_bf) continue;
            const uint4 raw = load(it);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(slot_of(it)), "r"(raw.x), "r"(raw.y),
                         "r"(raw.z), "r"(raw.w)
                         : "memory");
            if (lane == 0) {
                pe[cr * a.PES + (t % a.P) * MT + it % MT] = 1.0f;
                if (it % PM == 0) fs[cr] = 1;
            }
        }
        named_barrier_sync(1, kTcDecodeThreads);
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, kTcDecodeThreads);
}

// ---------------------------------------------------------------- decode
// One 128-k granule of this lane's row: codes as f16 (BF: bf16) into TMEM,
// multiplied by their block scales unless those come after the MMA.
template <int MT, int EPI, bool BF>
__device__ __forceinline__ void tc_decode(const TcArgs& a, uint32_t stage, int gran, int r, int bx, bool live,
                                          uint32_t taddr)
{
    using Cfg = TcCfg<MT, EPI>;
    const uint32_t row = stage + static_cast<uint32_t>(bx * a.R8 + r) * 128u;
    uint2 sw = make_uint2(0u, 0u);
    if (live && !Cfg::DEF) sw = lds64(stage + a.scales_off + static_cast<uint32_t>(bx * a.R8 + r) * 16u + 8 * gran);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint4 w[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (live) {
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
                w[c2] = lds128(row + ((static_cast<uint32_t>(4 * gran + 2 * half + c2) ^ static_cast<uint32_t>(r & 7))
                                      << 4));
        }
        uint32_t av[32];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const uint32_t ws[4] = {w[c2].x, w[c2].y, w[c2].z, w[c2].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t o[4];
                e2m1x8_to_f16x2x4(ws[q], o);
                if (!Cfg::DEF) {
                    // block 2 c2 + q / 2 of this half: its E4M3 byte
                    // duplicated, then converted, is the scale in both halves
                    const uint32_t blk = static_cast<uint32_t>(2 * c2 + (q >> 1));
                    const uint32_t s2 = e4m3x2_to_f16x2(__byte_perm(half ? sw.y : sw.x, 0, blk * 0x11u));
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = hmul2(o[i], s2);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) av[c2 * 16 + q * 4 + i] = BF ? f16x2_to_bf16x2(o[i]) : o[i];
            }
        }
        tc_st_x32(taddr + 32u * half, av);
    }
}

template <int MT>
__device__ __forceinline__ float tc_pick(const uint32_t* v, int p, int m)
{
    float r = __uint_as_float(tc_after_wait(v[m]));
    const float r1 = __uint_as_float(tc_after_wait(v[MT + m]));
    const float r2 = __uint_as_float(tc_after_wait(v[2 * MT + m]));
    const float r3 = __uint_as_float(tc_after_wait(v[3 * MT + m]));
    r = p == 1 ? r1 : r;
    r = p == 2 ? r2 : r;
    r = p == 3 ? r3 : r;
    return r;
}

// NPC: one-token phase columns the fold accumulates (1, 2 or 4 >= P).
// NORM: the RMSNorm prologue (dense launches).
template <int MT, int EPI, int NPC, bool NORM>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemv_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales)
{
    using Cfg = TcCfg<MT, EPI>;
    constexpr int NGU = Cfg::NGU;
    constexpr int NB = Cfg::NB;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = warp_index_uniform();
    const int lane = threadIdx.x & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.smem_bar);
    uint64_t* empty = full + kTcMaxStages;
    uint64_t* a_ready = empty + kTcMaxStages;  // [NB] A of a TMEM buffer written (4 decode warps)
    uint64_t* mma_done = a_ready + kTcMaxBufs; // [NB] MMAs of a buffer complete (commit)
    uint64_t* d_free = mma_done + kTcMaxBufs;  // [NB] D of a buffer read back (4 fold warps)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(d_free + kTcMaxBufs);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int* fs = reinterpret_cast<const int*>(smem + a.smem_fs);

    // Let the next kernel on the stream start its weight streaming as soon
    // as SMs free up; it waits for this grid before reading our outputs.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTcFoldWarps * kTcGran);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(&a_ready[b], 4);
            mbar_init(&mma_done[b], 1);
            mbar_init(&d_free[b], 4);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kTcMmaWarp0) {
        tc_alloc(tmem_slot, kTcCols);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Grouped launches read their unit list from the previous kernel's output.
    if (a.units != nullptr) asm volatile("griddepcontrol.wait;" ::: "memory");
    int ub, ue, us;
    tc_unit_range(a, ub, ue, us);

    // TMEM lanes of this warp's quadrant hold (row, gate/up, phase) triples.
    const int q = warp & 3;
    const int L = a.R * NGU * a.P;
    const int Lq = (L + 3) >> 2;
    const int j = q * Lq + lane;
    const bool valid = lane < Lq && j < L;
    int r = 0, gu = 0, p = 0;
    if (valid) {
        r = j % a.R;
        const int t = j / a.R;
        gu = t % NGU;
        p = t / NGU;
    }
    const int bx = p * NGU + gu;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t ring = smem_u32(smem + a.smem_ring);

    if (warp == kTcTmaWarp) {
        // ------------------------------------------------------------ producer
        if (elect_one()) {
            prefetch_tensormap(&tm_codes);
            prefetch_tensormap(&tm_scales);
        }
        __syncwarp();
        int slot = 0, lap = 0, issued = 0;
        bool stop = false;
        for (int u = ub; u < ue && !stop; u += us) {
            const TcUnit un = tc_unit(a, u);
            for (int c = 0; c < a.Cp; ++c) {
                if (lap > 0 && !tc_wait_warp(&empty[slot], (lap - 1) & 1, a, abort_flag)) {
                    stop = true;
                    break;
                }
                if (*abort_flag || a.starve) {
                    stop = true;
                    break;
                }
                // phases whose range ends before this stage load nothing
                int live = 0;
                for (int pp = 0; pp < a.P; ++pp) live += (pp * a.Cp + c < a.C) ? 1 : 0;
                uint8_t* sb = smem + a.smem_ring + slot * a.stage_bytes;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(live * NGU) * a.box_tx);
                    for (int pp = 0; pp < a.P; ++pp) {
                        const int kc = pp * a.Cp + c;
                        if (kc >= a.C) continue;
#pragma unroll
                        for (int g = 0; g < NGU; ++g) {
                            const int b2 = pp * NGU + g;
                            const int row = un.w_row0 + g * a.up_row_offset;
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
        // No copy may still be landing in shared memory when the CTA exits.
        if (lane == 0)
            for (int g = max(0, issued - a.n_stages); g < issued; ++g)
                mbar_wait_bounded(&full[g % a.n_stages], (g / a.n_stages) & 1, a.wait_ns, a.status);
        __syncwarp();
    } else if (warp >= kTcMmaWarp0) {
        // ------------------------------------------------------------ MMA issue
        // One MMA warp per decode set (on its own sub-partition), so each
        // issues one granule every two stages. The whole warp runs the loop,
        // so descriptors and TMEM addresses are warp-uniform; one elected
        // lane issues the MMAs and the commit.
        const int mset = warp - kTcMmaWarp0;
        const uint32_t zb = smem_u32(smem + a.smem_z);
        const int PM = a.P * MT;
        constexpr uint32_t idesc_h = tc_idesc_f16(128, Cfg::N, false);
        constexpr uint32_t idesc_b = tc_idesc_f16(128, Cfg::N, true);
        int gi = 0, issued = 0;
        bool stop = false;
        for (int u = ub; u < ue && !stop; u += us) {
            int cr = 0;
            for (int c = 0; c < a.Cp && !stop; ++c) {
                for (int gr = 0; gr < kTcGran; ++gr, ++gi) {
                    if ((gi & 3) != mset) continue;
                    const int b = gi % NB;
                    // "A written" also means the previous use's D was read back.
                    if (!tc_wait_warp(&a_ready[b], (gi / NB) & 1, a, abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t idesc = fs[cr] ? idesc_b : idesc_h;
                    const uint32_t tb = tmem + static_cast<uint32_t>(b * Cfg::BUFC);
                    const int s0 = cr * 16 + gr * Cfg::STEPS;  // first MMA step of the granule
                    if (elect_one()) {
                        if constexpr (Cfg::DEF) {
                            const uint32_t z_lead = zb;
                            const uint32_t z_trail = zb + a.z_bytes - kTcZeroPad;
#pragma unroll
                            for (int i = 0; i < Cfg::STEPS; ++i) {
                                const uint32_t pat = zb + kTcZeroPad + static_cast<uint32_t>(2 * (s0 + i)) * 128u;
                                const int jj = i & 3;
                                const uint32_t start = jj == 0 ? pat + 64u : jj == 1 ? pat : z_lead;
                                const uint32_t second = jj == 0 || jj == 1 ? z_trail : jj == 2 ? pat + 64u : pat;
                                tc_mma_f16_ts(tb + Cfg::ACOLS + (i >> 2) * Cfg::N, tb + i * 8,
                                              tc_smem_desc(start, 128u, second - start), idesc, jj != 0);
                            }
                        } else {
                            const uint32_t lbo = static_cast<uint32_t>(PM) * 16u;
                            const uint32_t zstep = static_cast<uint32_t>(2 * PM) * 16u;
#pragma unroll
                            for (int i = 0; i < Cfg::STEPS; ++i)
                                tc_mma_f16_ts(tb + Cfg::ACOLS, tb + i * 8,
                                              tc_smem_desc(zb + static_cast<uint32_t>(s0 + i) * zstep, lbo, 128u),
                                              idesc, i > 0);
                        }
                        tc_commit(&mma_done[b]);
                    }
                    __syncwarp();
                    ++issued;
                }
                if (++cr == a.SC) cr = 0;
            }
        }
        // Every MMA this warp issued completes before TMEM is released: its
        // last granule's commit arrives after all of them.
        if (lane == 0 && issued > 0) {
            int last = gi - 1;
            while ((last & 3) != mset) --last;
            mbar_wait_bounded(&mma_done[last % NB], (last / NB) & 1, a.wait_ns, a.status);
        }
        __syncwarp();
    } else if (warp < kTcDecodeWarps) {
        // ------------------------------------------------------------ decode warps
        const int dset = warp >> 2;
        // Activations may come from the previous kernel.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (NORM) tc_norm_factors(a, smem, warp, lane);
        bool aborted = false;
        int slot = 0, lap = 0, gi = 0;
        int conv_key = -1, conv_c0 = -1;
        for (int u = ub; u < ue; u += us) {
            const TcUnit un = tc_unit(a, u);
            int ntok = a.M, xkey = 0;
            const int* xrow = nullptr;
            if (a.units != nullptr) {
                const GroupDesc* gd = a.groups + un.grp;
                ntok = gd->ntok;
                xkey = gd->xkey;
                xrow = gd->x_row;
            }
            int cr = 0;
            for (int c = 0; c < a.Cp; ++c) {
                if (cr == 0 && (c != conv_c0 || xkey != conv_key)) {
                    // New B operand: every granule issued so far must have
                    // been read back (its MMAs done, its factors read). Once
                    // all decode warps are here, each buffer's last use is the
                    // phase its d_free barrier is on or has just completed.
                    named_barrier_sync(1, kTcDecodeThreads);
                    if (!aborted)
                        for (int s = max(0, gi - NB); s < gi; ++s)
                            if (!tc_wait_warp(&d_free[s % NB], (s / NB) & 1, a, abort_flag)) {
                                aborted = true;
                                break;
                            }
                    named_barrier_sync(1, kTcDecodeThreads);
                    tc_convert<MT, NORM>(a, smem, c, min(a.SC, a.Cp - c), ntok, xrow, warp, lane);
                    conv_c0 = c;
                    conv_key = xkey;
                }
                // this set's granule of the stage, if any
                const bool mine = ((gi & 3) == dset) || (((gi + 1) & 3) == dset);
                if (mine && !aborted && !tc_wait_warp(&full[slot], lap & 1, a, abort_flag)) aborted = true;
                const bool bf = fs[cr] != 0;
                const bool live = valid && (p * a.Cp + c < a.C);
                const uint32_t stage = ring + slot * a.stage_bytes;
#pragma unroll 1
                for (int gr = 0; gr < kTcGran; ++gr, ++gi) {
                    if ((gi & 3) != dset || aborted) continue;
                    const int b = gi % NB;
                    // Buffer b is free once its previous use was read back.
                    if (gi >= NB && !tc_wait_warp(&d_free[b], ((gi / NB) - 1) & 1, a, abort_flag)) {
                        aborted = true;
                        continue;
                    }
                    tc_fence_after();
                    const uint32_t ta = tl + static_cast<uint32_t>(b * Cfg::BUFC);
                    if (bf)
                        tc_decode<MT, EPI, true>(a, stage, gr, r, bx, live, ta);
                    else
                        tc_decode<MT, EPI, false>(a, stage, gr, r, bx, live, ta);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_ready[b]);
                }
                if (++slot == a.n_stages) {
                    slot = 0;
                    ++lap;
                }
                if (++cr == a.SC) cr = 0;
            }
        }
    } else {
        // ------------------------------------------------------------ fold warps
        float* red = reinterpret_cast<float*>(smem + a.smem_red);
        const float* pe_all = reinterpret_cast<const float*>(smem + a.smem_pe);
        const int ftid = threadIdx.x - kTcDecodeThreads;  // 0 .. 127
        // Residuals and the output buffer may belong to the previous kernel.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        bool aborted = false;
        int slot = 0, gi = 0;
        for (int u = ub; u < ue; u += us) {
            const TcUnit un = tc_unit(a, u);
            int ntok = a.M;
            float gsc = a.g;
            if (a.units != nullptr) {
                ntok = a.groups[un.grp].ntok;
                gsc = a.gscales[a.groups[un.grp].e];
            }
            constexpr int NACC = Cfg::DEF ? NPC : MT;
            float acc[NACC];
#pragma unroll
            for (int n = 0; n < NACC; ++n) acc[n] = 0.f;
            int cr = 0;
            for (int c = 0; c < a.Cp; ++c) {
                const uint32_t stage = ring + slot * a.stage_bytes;
                const bool live = valid && (p * a.Cp + c < a.C);
                const float* pe_stage = pe_all + cr * a.PES;
#pragma unroll 1
                for (int gr = 0; gr < kTcGran; ++gr, ++gi) {
                    if (aborted) continue;
                    const int b = gi % NB;
                    if (!tc_wait_warp(&mma_done[b], (gi / NB) & 1, a, abort_flag)) {
                        aborted = true;
                        continue;
                    }
                    tc_fence_after();
                    const uint32_t tb = tl + static_cast<uint32_t>(b * Cfg::BUFC);
                    if constexpr (Cfg::DEF) {
                        uint32_t v[2][16];
                        tc_ld<16>(tb + Cfg::ACOLS, v[0]);
                        tc_ld<16>(tb + Cfg::ACOLS + Cfg::N, v[1]);
                        uint2 sw = make_uint2(0u, 0u);
                        if (live) sw = lds64(stage + a.scales_off + static_cast<uint32_t>(bx * a.R8 + r) * 16u + 8 * gr);
                        const float4 f = *reinterpret_cast<const float4*>(pe_stage);
                        tc_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_free[b]);
                        float part[NPC];
#pragma unroll
                        for (int n = 0; n < NPC; ++n) part[n] = 0.f;
#pragma unroll
                        for (int rg = 0; rg < 2; ++rg) {
                            const uint32_t s_lo = e4m3x2_to_f16x2((rg ? sw.y : sw.x) & 0xFFFFu);
                            const uint32_t s_hi = e4m3x2_to_f16x2((rg ? sw.y : sw.x) >> 16);
                            const float sc[4] = {half_bits_to_f32(s_lo & 0xFFFFu), half_bits_to_f32(s_lo >> 16),
                                                 half_bits_to_f32(s_hi & 0xFFFFu), half_bits_to_f32(s_hi >> 16)};
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                                for (int n = 0; n < NPC; ++n)
                                    part[n] = fmaf(__uint_as_float(tc_after_wait(v[rg][4 * jj + n])), sc[jj], part[n]);
                        }
                        const float fe[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                        for (int n = 0; n < NPC; ++n) acc[n] = fmaf(part[n], fe[n], acc[n]);
                    } else {
                        uint32_t v[Cfg::W];
                        tc_ld<Cfg::W>(tb + Cfg::ACOLS, v);
                        float fe[MT];
#pragma unroll
                        for (int m = 0; m < MT; ++m) fe[m] = pe_stage[p * MT + m];
                        tc_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_free[b]);
#pragma unroll
                        for (int m = 0; m < MT; ++m) acc[m] = fmaf(tc_pick<MT>(v, p, m), fe[m], acc[m]);
                    }
                    // This warp is done with the stage's shared memory.
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                }
                if (++slot == a.n_stages) slot = 0;
                if (++cr == a.SC) cr = 0;
            }

            // ---------------- fixed-order reduction over fold warps and phases, epilogue
            named_barrier_sync(2, kTcFoldThreads);
            if (valid) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = acc[Cfg::DEF ? 0 : m];
                    if constexpr (Cfg::DEF) {
#pragma unroll
                        for (int n = 1; n < NPC; ++n)
                            if (p == n) v = acc[n];
                    }
                    red[((p * NGU + gu) * a.R + r) * MT + m] = v;
                }
            }
            named_barrier_sync(2, kTcFoldThreads);
            if (!aborted) {
                for (int idx = ftid; idx < a.R * MT; idx += kTcFoldThreads) {
                    const int rr = idx / MT;
                    const int m = idx % MT;
                    if (rr >= un.rows || m >= ntok) continue;
                    const int orow = a.units == nullptr ? m : a.groups[un.grp].out_row[m];
                    if (orow < 0) continue;
                    float v[NGU];
#pragma unroll
                    for (int gg = 0; gg < NGU; ++gg) {
                        float s = 0.f;
                        for (int pp = 0; pp < a.P; ++pp) s += red[((pp * NGU + gg) * a.R + rr) * MT + m];
                        v[gg] = s * gsc;
                    }
                    float val = v[0];
                    if (EPI == EPI_SWIGLU) val = (val / (1.0f + expf(-val))) * v[NGU - 1];
                    const size_t o = static_cast<size_t>(orow) * a.out_pitch + un.out_col0 + rr;
                    if (EPI == EPI_RESID) val += bf16_bits_to_f32(a.residual[o]);
                    if (a.out_f32)
                        reinterpret_cast<float*>(a.y)[o] = val;
                    else
                        reinterpret_cast<uint16_t*>(a.y)[o] = f32_to_bf16_bits_rn(val);
                }
            }
        }
    }

    // TMEM goes back only after every role is done with it.
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp0) {
        tc_fence_after();
        tc_dealloc(tmem, kTcCols);
    }
}

constexpr uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

// Shared-memory bytes of the activation super-chunk (B operand, exponents,
// flags, stage flags, factors) for `sc` stages.
struct ZPlan {
    uint32_t z, ex, fl, fs, pe;
    uint32_t total() const { return z + ex + fl + fs + pe; }
};

ZPlan z_plan(int sc, int P, int MT, int N, int PES)
{
    const uint32_t PM = static_cast<uint32_t>(P * MT);
    ZPlan zp;
    if (MT == 1)  // zero pad, 32 eight-row patterns per stage, zero pad
        zp.z = align_up(2u * kTcZeroPad + static_cast<uint32_t>(sc) * 32u * 128u, 128);
    else
        zp.z = align_up((static_cast<uint32_t>(sc) * 32u * PM + static_cast<uint32_t>(N)) * 16u, 128);
    zp.ex = align_up(static_cast<uint32_t>(sc) * PM * 4u, 16);
    zp.fl = align_up(static_cast<uint32_t>(sc) * PM, 16);
    zp.fs = align_up(static_cast<uint32_t>(sc) * 4u, 16);
    zp.pe = align_up(static_cast<uint32_t>(sc * PES) * 4u, 16);
    return zp;
}

// Completes the launch-time fields of `a` (status word, debug limits, stage
// and shared-memory plan) and launches with programmatic dependent launch.
template <int MT, int EPI, int NPC, bool NORM = false>
qg_status tc_launch(TcArgs a, const CUtensorMap& tmc, const CUtensorMap& tms, int grid, cudaStream_t stream)
{
    using Cfg = TcCfg<MT, EPI>;
    a.status = device_status_ptr();
    if (!a.status) return QG_ERR_CUDA;
    const DebugState dbg = debug_state();
    a.wait_ns = dbg.wait_ns;
    a.starve = dbg.starve;

    const int NGU = Cfg::NGU;
    a.R8 = (a.R + 7) / 8 * 8;
    const uint32_t nbox = static_cast<uint32_t>(a.P * NGU);
    a.scales_off = nbox * a.R8 * 128u;
    a.stage_bytes = align_up(a.scales_off + nbox * a.R8 * 16u, 1024);
    a.box_tx = static_cast<uint32_t>(a.R) * (128u + 16u);
    a.PES = Cfg::DEF ? 4 : a.P * MT;

    const uint32_t red_bytes = align_up(nbox * a.R * MT * 4u, 128);
    const uint32_t rms_bytes = a.norm_w ? align_up(static_cast<uint32_t>(a.M * a.C + 8) * 4u, 16) : 0u;
    const uint32_t bar_bytes = (2 * kTcMaxStages + 3 * kTcMaxBufs) * 8 + 16 + rms_bytes;
    // Keep at least ~96 KB (or 4 stages) of weights in flight; the
    // activations get the rest, as few super-chunks as possible.
    const uint32_t ring_min = std::max<uint32_t>(96u * 1024u, 4u * a.stage_bytes);
    int sc = a.Cp;
    while (sc > 1 && red_bytes + bar_bytes + z_plan(sc, a.P, MT, Cfg::N, a.PES).total() + ring_min > kTcSmemMax)
        --sc;
    a.SC = sc;
    const ZPlan zp = z_plan(sc, a.P, MT, Cfg::N, a.PES);
    a.z_bytes = zp.z;
    const uint32_t fixed = red_bytes + bar_bytes + zp.total();
    if (fixed + 2 * a.stage_bytes > kTcSmemMax) return QG_ERR_UNSUPPORTED;
    int n_stages = static_cast<int>((kTcSmemMax - fixed) / a.stage_bytes);
    n_stages = std::min(n_stages, kTcMaxStages);
    // An even ring: slot c % n_stages then always holds stages of the same
    // parity, i.e. the same pair of decode sets waits on each slot's barrier,
    // every phase in order.
    n_stages &= ~1;
    if (n_stages < 2) return QG_ERR_UNSUPPORTED;
    a.n_stages = n_stages;

    uint32_t so = 0;
    a.smem_ring = so;
    so += n_stages * a.stage_bytes;
    a.smem_z = so;
    so += zp.z;
    a.smem_ex = so;
    so += zp.ex;
    a.smem_fl = so;
    so += zp.fl;
    a.smem_fs = so;
    so += zp.fs;
    a.smem_pe = so;
    so += zp.pe;
    a.smem_red = so;
    so += red_bytes;
    a.smem_bar = so;
    a.smem_rms = so + bar_bytes - rms_bytes;
    so += bar_bytes;
    so = std::max(so, kTcSmemMin);
    if (so > kTcSmemMax) return QG_ERR_UNSUPPORTED;

    auto kern = tc_gemv_kernel<MT, EPI, NPC, NORM>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QG_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemMax) != cudaSuccess)
            return QG_ERR_CUDA;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
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
qg_status tc_dispatch_mt(const TcArgs& a, const CUtensorMap& tmc, const CUtensorMap& tms, int grid,
                         cudaStream_t stream)
{
    if (a.norm_w != nullptr) {
        // one token with the prologue runs on the CUDA-core kernel
        if (a.M <= 1) return QG_ERR_UNSUPPORTED;
        if (a.M <= 2) return tc_launch<2, EPI, 4, true>(a, tmc, tms, grid, stream);
        if (a.M <= 4) return tc_launch<4, EPI, 4, true>(a, tmc, tms, grid, stream);
        return tc_launch<8, EPI, 4, true>(a, tmc, tms, grid, stream);
    }
    if (a.M <= 1) {
        if (a.P <= 1) return tc_launch<1, EPI, 1>(a, tmc, tms, grid, stream);
        if (a.P <= 2) return tc_launch<1, EPI, 2>(a, tmc, tms, grid, stream);
        return tc_launch<1, EPI, 4>(a, tmc, tms, grid, stream);
    }
    if (a.M <= 2) return tc_launch<2, EPI, 4>(a, tmc, tms, grid, stream);
    if (a.M <= 4) return tc_launch<4, EPI, 4>(a, tmc, tms, grid, stream);
    return tc_launch<8, EPI, 4>(a, tmc, tms, grid, stream);
}

// K phases for units of R rows: as many as the 128 TMEM lanes hold, at most
// 4 (one D column group each) and at most one per 256-k chunk.
int tc_phases(int R, int ngu, int C)
{
    int P = 128 / (R * ngu);
    P = std::min(P, 4);
    P = std::min(P, C);
    return std::max(P, 1);
}

bool tc_maps(CUtensorMap* tmc, CUtensorMap* tms, const uint8_t* codes, const uint8_t* scales, int rows, int K,
             int R)
{
    memset(tmc, 0, sizeof(*tmc));
    memset(tms, 0, sizeof(*tms));
    if (!encode_tmap_2d(tmc, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, 128, R, true)) return false;
    return encode_tmap_2d(tms, scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, rows, 16, R, false);
}

}  // namespace

qg_status launch_tc_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w, float norm_eps)
{
    const int ngu = swiglu ? 2 : 1;
    const int n_out = swiglu ? N / 2 : N;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    // Smallest number of units per CTA whose rows fit the 128 TMEM lanes;
    // R = ceil(n_out / (SMs * units)) gives every SM the same byte count.
    int R = 1;
    for (int U = 1;; ++U) {
        R = (n_out + sms * U - 1) / (sms * U);
        if (R * ngu <= 128) break;
    }
    R = std::max(R, 1);
    TcArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.residual = static_cast<const uint16_t*>(residual);
    a.M = M;
    a.K = K;
    a.C = K / kChunkK;
    a.n_out = n_out;
    a.out_pitch = n_out;
    a.R = R;
    a.P = tc_phases(R, ngu, a.C);
    a.Cp = (a.C + a.P - 1) / a.P;
    a.up_row_offset = swiglu ? n_out : 0;
    a.out_f32 = swiglu ? 0 : out_f32;
    a.g = g;
    a.norm_w = static_cast<const uint16_t*>(norm_w);
    a.norm_eps = norm_eps;
    a.n_units = (n_out + R - 1) / R;
    const int grid = std::min(sms, a.n_units);
    CUtensorMap tmc, tms;
    if (!tc_maps(&tmc, &tms, codes, scales, N, K, R)) return QG_ERR_CUDA;
    if (swiglu) return tc_dispatch_mt<EPI_SWIGLU>(a, tmc, tms, grid, stream);
    if (residual) return tc_dispatch_mt<EPI_RESID>(a, tmc, tms, grid, stream);
    return tc_dispatch_mt<EPI_NONE>(a, tmc, tms, grid, stream);
}

qg_status launch_tc_grouped_nvfp4(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu,
                                  int up_offset, const void* x, int max_cols, void* y, int out_pitch, int out_f32,
                                  const GroupDesc* groups, const UnitDesc* units, const int* n_units,
                                  const float* gscales, int rows_per_unit, cudaStream_t stream)
{
    const int ngu = swiglu ? 2 : 1;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    if (rows_per_unit * ngu > 128) return QG_ERR_UNSUPPORTED;
    TcArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.M = max_cols;
    a.K = K;
    a.C = K / kChunkK;
    a.out_pitch = out_pitch;
    a.R = rows_per_unit;
    a.P = tc_phases(rows_per_unit, ngu, a.C);
    a.Cp = (a.C + a.P - 1) / a.P;
    a.up_row_offset = up_offset;
    a.out_f32 = out_f32;
    a.g = 1.f;
    a.groups = groups;
    a.units = units;
    a.n_units_dev = n_units;
    a.gscales = gscales;
    CUtensorMap tmc, tms;
    if (!tc_maps(&tmc, &tms, codes, scales, total_rows, K, rows_per_unit)) return QG_ERR_CUDA;
    if (swiglu) return tc_dispatch_mt<EPI_SWIGLU>(a, tmc, tms, sms, stream);
    return tc_dispatch_mt<EPI_NONE>(a, tmc, tms, sms, stream);
}

}  // namespace qg
