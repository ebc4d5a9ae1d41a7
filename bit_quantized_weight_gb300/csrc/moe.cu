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
    pdl_enter();
    const int m = blockIdx.x;
    const int lane = threadIdx.x;
    if (m >= M) return;
    const float* l = logits + static_cast<size_t>(m) * E;
    // E <= 1024: this lane's logits (experts lane + 32 j) stay in registers,
    // and bit j of `taken` marks expert lane + 32 j as already selected
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (32 * j >= E) break;
        v[j] = lane + 32 * j < E ? l[lane + 32 * j] : 0.f;
    }
    uint32_t taken = 0;
    float sel_l[8];
    int sel_id[8];
    for (int i = 0; i < topk; ++i) {
        float best = -INFINITY;
        int best_id = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (32 * j >= E) break;  // the same for every lane
            const int e = lane + 32 * j;
            if (e >= E || ((taken >> j) & 1u)) continue;
            if (v[j] > best || (v[j] == best && e < best_id)) {
                best = v[j];
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
        if ((best_id & 31) == lane) taken |= 1u << (best_id >> 5);
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
    if (launch_pdl(route_kernel, dim3(M), dim3(32), 0, stream, logits, M, E, topk, ids, w) != cudaSuccess)
        return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

namespace {

constexpr int kMaxPairs = kMaxTokens * 8;

struct MoeLayout {
    size_t h, yslot, ctrl, g_gu, g_dn, u_gu, u_dn, p_gu, p_dn, total;
    int r_gu, r_dn, units_gu_max, units_dn_max;
    int rc_gu, rc_dn;  // the CUDA-core kernels' rows per pass
};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Rows per unit: the gate/up launch walks (expert, 64-row block) units (64
// gate plus 64 up rows fill one 128-lane accumulator) and the down launch
// (expert, 128-row block) units, so the ~50 active experts spread evenly over
// the SMs. H and I are multiples of 256, so both divide evenly.
MoeLayout moe_layout(int M, int topk, int H, int I)
{
    MoeLayout L{};
    const size_t P = static_cast<size_t>(M) * topk;
    L.r_gu = 64;
    L.r_dn = 128;
    L.units_gu_max = kMaxPairs * (I / L.r_gu);
    L.units_dn_max = kMaxPairs * (H / L.r_dn);
    // CUDA-core passes: 32 gate/up row pairs (4 phases of 2 x 32 rows fill a
    // 256-row stage) and 256 down rows (one phase, three full stages per pass
    // at I = 768; on the 35B-A3B-class layer 64- and 128-row passes were 6 %
    // and 2 % slower, 64-pair gate/up passes 1 % slower); every pair group
    // holds at least one valid (token, slot) pair, so P bounds the groups of
    // either launch.
    L.rc_gu = 32;
    L.rc_dn = 256;
    size_t o = 0;
    L.h = o;
    o += up256(P * I * 2);
    L.yslot = o;
    o += up256(P * H * 4);
    L.ctrl = o;
    o += 256;
    L.g_gu = o;
    o += up256(sizeof(GroupDesc) * kMaxPairs);
    L.g_dn = o;
    o += up256(sizeof(GroupDesc) * kMaxPairs);
    L.u_gu = o;
    o += up256(sizeof(UnitDesc) * L.units_gu_max);
    L.u_dn = o;
    o += up256(sizeof(UnitDesc) * L.units_dn_max);
    L.p_gu = o;
    o += up256(sizeof(CcPair) * P);
    L.p_dn = o;
    o += up256(sizeof(CcPair) * P);
    L.total = o;
    return L;
}

// Groups the (token, slot) pairs by expert and writes the unit lists.
// Gate/up: one group per active expert; its 8 columns are the 8 token rows of
// x (shared by every expert, xkey 0) and column m writes h row m * topk + i of
// the slot that routed token m there. Down: the pairs of an expert, at most 8
// per group; column j reads h row x_row[j] and writes slot row out_row[j].
// A token listing one expert twice reuses the first slot's h row.
//
// It also writes the CUDA-core kernels' pair groups. Gate/up: per expert, its
// distinct tokens in pairs (x row = token, output row = that token's first
// slot for the expert). Down: per expert, its (token, slot) pairs in pairs (x
// row = the h row the token's first slot wrote, output row = the slot).
// ctrl[2] and ctrl[3] receive the counts.
__global__ void moe_group_kernel(const int32_t* ids, int M, int topk, int E, int I, int H, int r_gu, int r_dn,
                                 GroupDesc* g_gu, GroupDesc* g_dn, UnitDesc* u_gu, UnitDesc* u_dn, CcPair* p_gu,
                                 CcPair* p_dn, int emit_tc, int* ctrl, int* status)
{
    __shared__ int s_pair_e[kMaxPairs];
    __shared__ int s_order[kMaxPairs];    // valid pairs sorted by (expert, pair)
    __shared__ int s_gu_at[kMaxPairs];    // gate/up group of sorted position i
    __shared__ int s_run0[kMaxPairs];     // first sorted position of that group's expert run
    __shared__ int s_dn_start[kMaxPairs]; // sorted position starting each down group
    __shared__ int s_gu_e[kMaxPairs], s_dn_e[kMaxPairs];  // expert of each group
    __shared__ int s_nv, s_n_gu, s_n_dn;
    pdl_enter();
    const int P = M * topk;
    const int tid = threadIdx.x;
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e < 0 || e >= E) {
            atomicCAS(status, 0, QG_ERR_INVALID_ARG);
            s_pair_e[p] = -1;
        } else {
            s_pair_e[p] = e;
        }
    }
    __syncthreads();
    // rank of each valid pair in (expert, pair) order: one thread per pair
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = s_pair_e[p];
        if (e < 0) continue;
        int r = 0;
        for (int q = 0; q < P; ++q) {
            const int f = s_pair_e[q];
            r += (f >= 0 && (f < e || (f == e && q < p))) ? 1 : 0;
        }
        s_order[r] = p;
    }
    if (tid == 0) {
        int nv = 0;
        for (int p = 0; p < P; ++p) nv += s_pair_e[p] >= 0 ? 1 : 0;
        s_nv = nv;
    }
    __syncthreads();
    const int nv = s_nv;
    // The tcgen05 kernels' lists, only when they will run (emit_tc is the
    // same for every thread, so the barriers inside are reached by all).
    if (emit_tc) {
    // group boundaries along the sorted pairs (at most 64 positions: the
    // first two warps, one position per lane, ballots for the prefix counts)
    if (tid < 64) {
        const int nv = s_nv;
        const int i = tid;
        const bool in = i < nv;
        const int e = in ? s_pair_e[s_order[i]] : -1;
        const bool run_start = in && (i == 0 || e != s_pair_e[s_order[i - 1]]);
        // start of this position's run: the last run start at or before i
        int run0 = 0;
        for (int j = i; j >= 0 && in; --j)
            if (j == 0 || s_pair_e[s_order[j]] != s_pair_e[s_order[j - 1]]) {
                run0 = j;
                break;
            }
        const bool dn_start = in && ((i - run0) % 8 == 0);
        const unsigned lanes_below = (1u << (tid & 31)) - 1u;
        const unsigned rs = __ballot_sync(0xffffffffu, run_start), ds = __ballot_sync(0xffffffffu, dn_start);
        s_run0[i] = run0;
        // runs started at or before i, and down groups started before i, in this warp
        const int my_gu = __popc(rs & lanes_below) + (run_start ? 1 : 0);
        const int my_dn = __popc(ds & lanes_below);
        // positions 32..63 add the first warp's totals
        __shared__ int s_part[2][2];
        if ((tid & 31) == 31) {
            s_part[tid >> 5][0] = __popc(rs);
            s_part[tid >> 5][1] = __popc(ds);
        }
        asm volatile("bar.sync 3, 64;" ::: "memory");
        const int base_gu = tid >= 32 ? s_part[0][0] : 0, base_dn = tid >= 32 ? s_part[0][1] : 0;
        if (in) {
            s_gu_at[i] = base_gu + my_gu - 1;
            if (dn_start) s_dn_start[base_dn + my_dn] = i;
            if (run_start) s_gu_e[base_gu + my_gu - 1] = e;
            if (dn_start) s_dn_e[base_dn + my_dn] = e;
        }
        if (tid == 0) {
            s_n_gu = s_part[0][0] + s_part[1][0];
            s_n_dn = s_part[0][1] + s_part[1][1];
        }
    }
    __syncthreads();
    // one gate/up group per expert run: all M token rows of x, the first
    // slot of each token writes its h row
    for (int i = tid; i < nv; i += blockDim.x) {
        if (s_run0[i] != i) continue;
        const int e = s_pair_e[s_order[i]];
        GroupDesc gg;
        gg.ntok = M;
        gg.e = e;
        gg.xkey = 0;
        for (int j = 0; j < 8; ++j) {
            gg.x_row[j] = j < M ? j : 0;
            gg.out_row[j] = -1;
        }
        for (int q = i; q < nv && s_pair_e[s_order[q]] == e; ++q) {
            const int p = s_order[q];
            const int m = p / topk;
            if (gg.out_row[m] < 0) gg.out_row[m] = p;
        }
        g_gu[s_gu_at[i]] = gg;
    }
    // down groups: chunks of at most 8 pairs of one run; a pair reads the h
    // row its token's first slot for that expert wrote
    for (int d = tid; d < s_n_dn; d += blockDim.x) {
        const int i0 = s_dn_start[d];
        const int e = s_pair_e[s_order[i0]];
        const int run0 = s_run0[i0];
        int iend = i0;
        while (iend < nv && iend - i0 < 8 && s_pair_e[s_order[iend]] == e) ++iend;
        GroupDesc gd;
        gd.ntok = iend - i0;
        gd.e = e;
        gd.xkey = 1 + d;
        for (int j = 0; j < 8; ++j) {
            if (j < gd.ntok) {
                const int p = s_order[i0 + j];
                const int m = p / topk;
                int first = p;
                for (int q = run0; q < i0 + j; ++q)
                    if (s_order[q] / topk == m) {
                        first = s_order[q];
                        break;
                    }
                gd.out_row[j] = p;
                gd.x_row[j] = first;
            } else {
                gd.out_row[j] = -1;
                gd.x_row[j] = 0;
            }
        }
        g_dn[d] = gd;
    }
    __syncthreads();
    const int per_gu = I / r_gu, per_dn = H / r_dn;
    const int n_gu = s_n_gu * per_gu, n_dn = s_n_dn * per_dn;
    for (int u = tid; u < n_gu; u += blockDim.x) {
        const int gi = u / per_gu, rb = u % per_gu;
        UnitDesc d;
        d.grp = gi;
        d.w_row0 = s_gu_e[gi] * 2 * I + rb * r_gu;
        d.rows = r_gu;
        d.out_col0 = rb * r_gu;
        u_gu[u] = d;
    }
    for (int u = tid; u < n_dn; u += blockDim.x) {
        const int gi = u / per_dn, rb = u % per_dn;
        UnitDesc d;
        d.grp = gi;
        d.w_row0 = s_dn_e[gi] * H + rb * r_dn;
        d.rows = r_dn;
        d.out_col0 = rb * r_dn;
        u_dn[u] = d;
    }
    if (tid == 0) {
        ctrl[0] = n_gu;
        ctrl[1] = n_dn;
    }
    }

    // ---- pair groups of the CUDA-core passes: (expert, n, x rows, output rows),
    // one thread per sorted position (at most 64), with 64-bit masks of the
    // run starts and of each (expert, token)'s first position
    __shared__ int s_pg[2][kMaxPairs][6];
    __shared__ int s_npg[2];
    __shared__ unsigned s_msk[2][2];           // [run start | first of token][warp]
    __shared__ int s_cnt[2][kMaxPairs];        // per run: gate/up groups, down groups
    __shared__ int s_base[2][kMaxPairs];       // per run: index of its first group
    __shared__ int s_nrun;
    const int pi = tid;
    const bool pin = pi < nv;
    const int pp_ = pin ? s_order[pi] : 0;
    const int pe_ = pin ? s_pair_e[pp_] : -1;
    const int pm_ = pp_ / topk;
    if (tid < 64) {
        const int pe_prev = pin && pi > 0 ? s_pair_e[s_order[pi - 1]] : -1;
        const int pm_prev = pin && pi > 0 ? s_order[pi - 1] / topk : -1;
        const bool rstart = pin && (pi == 0 || pe_prev != pe_);
        const bool first = pin && (rstart || pm_prev != pm_);
        const unsigned rb = __ballot_sync(0xffffffffu, rstart), fb = __ballot_sync(0xffffffffu, first);
        if ((tid & 31) == 0) {
            s_msk[0][tid >> 5] = rb;
            s_msk[1][tid >> 5] = fb;
        }
    }
    __syncthreads();
    const unsigned long long rsm = s_msk[0][0] | (static_cast<unsigned long long>(s_msk[0][1]) << 32);
    const unsigned long long fsm = s_msk[1][0] | (static_cast<unsigned long long>(s_msk[1][1]) << 32);
    // bits [lo, hi) of a 64-bit mask
    auto bits = [](int lo, int hi) -> unsigned long long {
        const unsigned long long h = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
        return h & ~((1ull << lo) - 1ull);
    };
    int run = 0, r0 = 0, r1 = 0;
    if (pin) {
        run = __popcll(rsm & bits(0, pi + 1)) - 1;
        r0 = 63 - __clzll(rsm & bits(0, pi + 1));
        const unsigned long long above = rsm & ~bits(0, pi + 1);
        r1 = above ? __ffsll(static_cast<long long>(above)) - 1 : nv;
        if (r0 == pi) {
            s_cnt[0][run] = (__popcll(fsm & bits(r0, r1)) + 1) / 2;
            s_cnt[1][run] = (r1 - r0 + 1) / 2;
        }
    }
    if (tid == 0) s_nrun = __popcll(rsm);
    __syncthreads();
    if (tid < 32) {
        // exclusive prefix over the runs, two per lane
        const int nr = s_nrun;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int a0 = 2 * tid < nr ? s_cnt[k][2 * tid] : 0;
            const int a1 = 2 * tid + 1 < nr ? s_cnt[k][2 * tid + 1] : 0;
            int incl = a0 + a1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += o;
            }
            const int excl = incl - a0 - a1;
            if (2 * tid < nr) s_base[k][2 * tid] = excl;
            if (2 * tid + 1 < nr) s_base[k][2 * tid + 1] = excl + a0;
            if (tid == 31) s_npg[k] = incl;
        }
    }
    __syncthreads();
    if (pin) {
        // gate/up: the token's first position in the run, its rank among them
        if (fsm & bits(pi, pi + 1)) {
            const int dr = __popcll(fsm & bits(r0, pi + 1)) - 1;
            const int nd = __popcll(fsm & bits(r0, r1));
            int* g = s_pg[0][s_base[0][run] + dr / 2];
            if (dr % 2 == 0) {
                g[0] = pe_;
                g[1] = min(2, nd - dr);
            }
            g[2 + dr % 2] = pm_;
            g[4 + dr % 2] = pp_;
        }
        // down: every pair, reading the h row of its token's first position
        const int j = pi - r0;
        const int fpos = 63 - __clzll(fsm & bits(0, pi + 1));
        int* d = s_pg[1][s_base[1][run] + j / 2];
        if (j % 2 == 0) {
            d[0] = pe_;
            d[1] = min(2, r1 - r0 - j);
        }
        d[2 + j % 2] = s_order[fpos];
        d[4 + j % 2] = pp_;
    }
    __syncthreads();
    const int ng = s_npg[0], nd = s_npg[1];
    for (int u = tid; u < ng + nd; u += blockDim.x) {
        const bool dn = u >= ng;
        const int v = dn ? u - ng : u;
        const int* g = s_pg[dn ? 1 : 0][v];
        CcPair pr;
        pr.e = g[0];
        pr.ntok = g[1];
        pr.x_row[0] = g[2];
        pr.x_row[1] = g[1] > 1 ? g[3] : g[2];
        pr.out_row[0] = g[4];
        pr.out_row[1] = g[1] > 1 ? g[5] : -1;
        (dn ? p_dn : p_gu)[v] = pr;
    }
    if (tid == 0) {
        ctrl[2] = ng;
        ctrl[3] = nd;
    }
}

// y[m][j] = bf16_rne( sum_{i ascending} w[m][i] * yslot[m * topk + i][j] ), fp32.
__global__ void moe_combine_kernel(const float* yslot, const int32_t* ids, const float* w, uint16_t* y, int M,
                                   int topk, int H, int E)
{
    pdl_enter();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= M * H) return;
    const int m = idx / H, j = idx % H;
    float acc = 0.f;
    for (int i = 0; i < topk; ++i) {
        const int e = ids[m * topk + i];
        if (e < 0 || e >= E) continue;
        acc = fmaf(w[m * topk + i], yslot[static_cast<size_t>(m * topk + i) * H + j], acc);
    }
    y[idx] = f32_to_bf16_bits_rn(acc);
}

// Expert-gathered NVFP4 GEMV: the tcgen05 kernel, else the mma.sync one.
qg_status grouped_nvfp4(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu, int up_offset,
                        const void* x, int max_cols, void* y, int out_pitch, int out_f32, const GroupDesc* groups,
                        const UnitDesc* units, const int* n_units, const float* gscales, int rows_per_unit,
                        cudaStream_t stream)
{
    const qg_status s = launch_tc_grouped_nvfp4(codes, scales, total_rows, K, swiglu, up_offset, x, max_cols, y,
                                                out_pitch, out_f32, groups, units, n_units, gscales, rows_per_unit,
                                                stream);
    if (s != QG_ERR_UNSUPPORTED) return s;
    return launch_grouped_nvfp4(codes, scales, total_rows, K, swiglu, up_offset, x, max_cols, y, out_pitch, out_f32,
                                groups, units, n_units, gscales, rows_per_unit, stream);
}

}  // namespace

size_t moe_workspace_bytes(int M, int topk, int H, int I, int E)
{
    (void)E;
    return moe_layout(M, topk, H, I).total;
}

qg_status launch_moe(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_g, const uint8_t* dn_codes,
                     const uint8_t* dn_scales, const float* dn_g, const void* x, const int32_t* ids, const float* tw,
                     void* y, void* ws, size_t ws_bytes, int M, int H, int I, int E, int topk, cudaStream_t stream)
{
    const MoeLayout L = moe_layout(M, topk, H, I);
    if (ws_bytes < L.total) return QG_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint16_t* h = reinterpret_cast<uint16_t*>(w + L.h);
    float* yslot = reinterpret_cast<float*>(w + L.yslot);
    int* ctrl = reinterpret_cast<int*>(w + L.ctrl);
    GroupDesc* g_gu = reinterpret_cast<GroupDesc*>(w + L.g_gu);
    GroupDesc* g_dn = reinterpret_cast<GroupDesc*>(w + L.g_dn);
    UnitDesc* u_gu = reinterpret_cast<UnitDesc*>(w + L.u_gu);
    UnitDesc* u_dn = reinterpret_cast<UnitDesc*>(w + L.u_dn);
    CcPair* p_gu = reinterpret_cast<CcPair*>(w + L.p_gu);
    CcPair* p_dn = reinterpret_cast<CcPair*>(w + L.p_dn);
    int* status = device_status_ptr();
    if (!status) return QG_ERR_CUDA;

    // The CUDA-core grouped kernels where their plans fit, else the tcgen05
    // ones (whose lists the grouping kernel then writes too).
    const int P = M * topk;
    auto cc_gu = [&](bool launch) {
        return launch_cc_moe(gu_codes, gu_scales, E * 2 * I, H, 1, I, 2 * I, I / L.rc_gu, x, M, h, I, 0, p_gu,
                             ctrl + 2, P, gu_g, L.rc_gu, stream, launch);
    };
    auto cc_dn = [&](bool launch) {
        return launch_cc_moe(dn_codes, dn_scales, E * H, I, 0, 0, H, H / L.rc_dn, h, P, yslot, H, 1, p_dn, ctrl + 3,
                             P, dn_g, L.rc_dn, stream, launch);
    };
    const qg_status fit_gu = cc_gu(false), fit_dn = cc_dn(false);
    if (fit_gu != QG_OK && fit_gu != QG_ERR_UNSUPPORTED) return fit_gu;
    if (fit_dn != QG_OK && fit_dn != QG_ERR_UNSUPPORTED) return fit_dn;
    const int emit_tc = (fit_gu != QG_OK || fit_dn != QG_OK) ? 1 : 0;
    if (launch_pdl(moe_group_kernel, dim3(1), dim3(256), 0, stream, ids, M, topk, E, I, H, L.r_gu, L.r_dn, g_gu,
                   g_dn, u_gu, u_dn, p_gu, p_dn, emit_tc, ctrl, status) != cudaSuccess)
        return QG_ERR_CUDA;
    qg_status s = fit_gu == QG_OK ? cc_gu(true)
                                  : grouped_nvfp4(gu_codes, gu_scales, E * 2 * I, H, 1, I, x, M, h, I, 0, g_gu, u_gu,
                                                  ctrl + 0, gu_g, L.r_gu, stream);
    if (s != QG_OK) return s;
    s = fit_dn == QG_OK ? cc_dn(true)
                        : grouped_nvfp4(dn_codes, dn_scales, E * H, I, 0, 0, h, 8, yslot, H, 1, g_dn, u_dn, ctrl + 1,
                                        dn_g, L.r_dn, stream);
    if (s != QG_OK) return s;
    const int n = M * H;
    if (launch_pdl(moe_combine_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, yslot, ids, tw,
                   static_cast<uint16_t*>(y), M, topk, H, E) != cudaSuccess)
        return QG_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
