// common.cuh -- device helpers shared by the qgemv kernels (sm_103a).
//
// Inline PTX for the Blackwell data path: mbarrier phases, TMA tensor loads
// (cp.async.bulk.tensor) into shared memory, the f16 tensor-core MMA, and the
// FP4/FP8 -> f16 conversion instructions. Every wait on an mbarrier is
// bounded: after the time limit it records QG_ERR_DEVICE_TIMEOUT in the
// library's device status word and lets the kernel return instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemv_internal.h"

namespace qg {

// Record the first device-side error in the library's status word (a
// device global owned by api.cu whose address every kernel receives).
__device__ __forceinline__ void set_device_status(int* status, int code)
{
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` while the phase
// is incomplete; it wakes when the phase completes, so waiting costs no issue
// slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}


// One lane of the warp is elected (true for exactly one active lane).
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile("{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}\n" : "=r"(pred));
    return pred != 0;
}

// Warp index the compiler can treat as uniform across the warp.
__device__ __forceinline__ int warp_index_uniform()
{
    return __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns nanoseconds. Returns false (and records a device timeout) when the
// limit runs out; the caller then stops issuing work and returns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0u && global_timer_ns() - t0 > limit_ns) {
            set_device_status(status, QG_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// ----------------------------------------------------------------- launch
// Launches `kern` with programmatic dependent launch: it may start while the
// previous kernel on the stream finishes, so it must execute
// griddepcontrol.wait before its first read of that kernel's results and
// before its first global write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Start of a kernel launched with launch_pdl: let the next kernel launch
// early, then wait for the previous one to complete.
__device__ __forceinline__ void pdl_enter()
{
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// A 3-D box (coordinates innermost first), as tma_load_2d.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Plain bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on the mbarrier.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------- conversions
// Two E2M1 codes (low nibble -> low half) to f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8)
{
    uint32_t r;
    asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n" : "=r"(r) : "r"(byte_in_low8));
    return r;
}

// The four codes bytes of a register, each as two E2M1 codes -> f16x2
// (low nibble -> low half), exact.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&out)[4])
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// Two E4M3 codes (low byte -> low half) to f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t r;
    asm("{\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}\n" : "=r"(r) : "r"(two_bytes));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits_rn(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float half_bits_to_f32(uint32_t bits16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// v * 2^e, exact whenever the result is a normal float. e is clamped to
// [-252, 252] (beyond that an fp32 result is 0 or inf anyway); the two steps
// keep each factor a normal float.
__device__ __forceinline__ float ldexp_exact(float v, int e)
{
    e = max(-252, min(252, e));
    const int e1 = e / 2;
    const int e2 = e - e1;
    return v * __int_as_float((127 + e1) << 23) * __int_as_float((127 + e2) << 23);
}

// ----------------------------------------------------------------- loads
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ldg_nc_128(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 128-bit global load cached in L2 only: coherent with stores other CTAs of
// the same kernel made before a grid-wide barrier.
__device__ __forceinline__ uint4 ldg_cg_128(const void* p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

template <bool CG>
__device__ __forceinline__ uint4 ldg_128(const void* p)
{
    return CG ? ldg_cg_128(p) : ldg_nc_128(p);
}

__device__ __forceinline__ uint32_t ldg_cg_u16(const uint16_t* p)
{
    uint16_t v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
    return v;
}

// ----------------------------------------------------------------- RMSNorm prologue
// The normalisation fused ahead of a projection: for one token of K bf16
// values, r = 1 / sqrt(sum(x^2) / K + eps) and h_k = bf16_rne(x_k * r * gamma_k);
// the projection then reads h. Every kernel derives r in one fixed order, so
// all CTAs of all kernels get the same bits: the squares of a 256-value chunk
// held 8 values per lane (lane l: values 8l .. 8l+7) are summed in order per
// lane, then by a butterfly over the warp; the chunks' sums are added in k
// order.
__device__ __forceinline__ float rms_chunk_ss(const uint4 raw)
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
        s = fmaf(lo, lo, s);
        s = fmaf(hi, hi, s);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// r from the sum of squares (IEEE division and square root).
__device__ __forceinline__ float rms_factor(float ss, int K, float eps)
{
    return 1.0f / sqrtf(__fdiv_rn(ss, static_cast<float>(K)) + eps);
}

// Eight bf16 activations (two per word) -> bf16(x * r * gamma), one rounding
// of the fp32 product (x * r) * gamma.
__device__ __forceinline__ uint4 rms_apply8(const uint4 x, const uint4 g, float r)
{
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = (__uint_as_float(xw[i] << 16) * r) * __uint_as_float(gw[i] << 16);
        const float hi = (__uint_as_float(xw[i] & 0xFFFF0000u) * r) * __uint_as_float(gw[i] & 0xFFFF0000u);
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ----------------------------------------------------------------- activation prescale
// Power-of-two prescale exponent p for a chunk whose largest finite |x| has
// bf16 magnitude bits `mag` (0 if every value is zero): max * 2^p in [2^14, 2^15).
__device__ __forceinline__ int prescale_exponent(uint32_t mag)
{
    if (mag == 0) return 0;
    uint32_t e = mag >> 7;
    if (e > 0) return 141 - static_cast<int>(e);
    // subnormal bf16: value = mag * 2^-133
    int lg = 31 - __clz(static_cast<int>(mag));
    return 147 - lg;
}

// Range of bf16 magnitudes (15-bit patterns) over 32-bit words of two bf16
// values each, both halves at once with 16-bit SIMD min/max: mx2 collects
// the largest magnitude with non-finite ones counted as the largest finite
// (0x7F7F), mn2 the smallest magnitude minus one (zero wraps to 0xFFFF and
// drops out). A chunk holding inf or NaN thus takes the prescale of 0x7F7F,
// which its other values do not survive exactly, so it is flagged and runs on
// raw bf16 (still exact); a borrow from the low into the high half can only
// lower the minimum, which makes the exactness test stricter, never looser.
__device__ __forceinline__ void bf16_range_acc(uint32_t w, uint32_t& mx2, uint32_t& mn2)
{
    const uint32_t m = w & 0x7FFF7FFFu;
    mx2 = __vmaxu2(mx2, __vminu2(m, 0x7F7F7F7Fu));
    mn2 = __vminu2(mn2, m - 0x00010001u);
}

// Exponent fields of the largest magnitude and of the smallest nonzero one
// (255 when there is none), and the largest magnitude itself, from the
// accumulators of bf16_range_acc.
__device__ __forceinline__ void bf16_range_fin(uint32_t mx2, uint32_t mn2, uint32_t& emax, uint32_t& emin,
                                               uint32_t& magmax)
{
    magmax = max(mx2 & 0xFFFFu, mx2 >> 16);
    const uint32_t mn = min(mn2 & 0xFFFFu, mn2 >> 16) + 1u;  // 0x10000: no nonzero value
    emax = magmax >> 7;
    emin = mn > 0x7FFFu ? 255u : min(mn >> 7, 255u);
}

// Exact f16x2 -> bf16x2 for values with at most 8 significant bits in the
// bf16 normal range (the decoded weights): through fp32, both steps exact.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2)
{
    const float lo = half_bits_to_f32(h2 & 0xFFFFu), hi = half_bits_to_f32(h2 >> 16);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ----------------------------------------------------------------- MMA
// D = A * B + C, m16n8k16, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace qg
