// qgemv_simple.cu -- exact CUDA-core GEMV for shapes the TMA kernel does not
// take (K not a multiple of 256), and the dequantisation export kernels.
//
// One warp per output row (per gate/up row pair for SwiGLU), lanes striding
// over k, fp32 accumulation of exact products, a butterfly reduction across
// the warp. Slow, simple and exact for every finite input.
#include "common.cuh"

#include <algorithm>

#include <cuda_bf16.h>

namespace qg {
namespace {

__device__ __forceinline__ float e2m1_value(uint32_t code)
{
    // f16 of the E2M1 code via the hardware conversion, then to fp32 (exact)
    const uint32_t h2 = e2m1x2_to_f16x2(code & 0xFu);
    return half_bits_to_f32(h2 & 0xFFFFu);
}

__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    const uint32_t h2 = e4m3x2_to_f16x2(code & 0xFFu);
    return half_bits_to_f32(h2 & 0xFFFFu);
}

// Weight w[n][k] in fp32: NVFP4 w = e2m1 * e4m3 (exact; g applied by the
// caller); Q w = fmaf(scale, q, min).
__device__ __forceinline__ float weight_at(int fmt, const uint8_t* codes, const uint8_t* q_hi,
                                           const void* scales, const void* mins, int K, int n, int k)
{
    const uint8_t b = codes[static_cast<size_t>(n) * (K / 2) + k / 2];
    const uint32_t nib = (k & 1) ? (b >> 4) : (b & 0xFu);
    if (fmt == FMT_NVFP4) {
        const uint8_t s = static_cast<const uint8_t*>(scales)[static_cast<size_t>(n) * (K / 16) + k / 16];
        return e2m1_value(nib) * e4m3_value(s);
    }
    uint32_t q = nib;
    if (fmt == FMT_Q5) q |= ((q_hi[static_cast<size_t>(n) * (K / 8) + k / 8] >> (k & 7)) & 1u) << 4;
    const size_t gi = static_cast<size_t>(n) * (K / 32) + k / 32;
    const float s = half_bits_to_f32(static_cast<const uint16_t*>(scales)[gi]);
    const float m = half_bits_to_f32(static_cast<const uint16_t*>(mins)[gi]);
    return fmaf(s, static_cast<float>(q), m);
}

// One warp per output row (gate/up row pair for SwiGLU). With the RMSNorm
// prologue, the CTA's first warps first derive each token's factor in the
// shared fixed order (chunks of 256 values, 8 per lane, then k order) and
// every k reads h = bf16((x * r) * gamma) instead of x.
__global__ void simple_kernel(const SimpleArgs a)
{
    __shared__ float s_r[kMaxTokens];
    const int M = a.M, K = a.K, n_out = a.n_out;
    const int lane = threadIdx.x & 31;
    if (a.norm_w != nullptr) {
        const int w = threadIdx.x >> 5;
        if (w < M) {
            const uint16_t* xr = a.x + static_cast<size_t>(w) * K;
            float t = 0.f;
            for (int k0 = 0; k0 < K; k0 += kChunkK) {
                const int k = k0 + lane * 8;
                const uint4 raw = k < K ? ldg_nc_128(xr + k) : make_uint4(0, 0, 0, 0);
                t += rms_chunk_ss(raw);
            }
            if (lane == 0) s_r[w] = rms_factor(t, K, a.norm_eps);
        }
        __syncthreads();
    }
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= n_out) return;
    const int n = warp;
    const bool sep_up = a.ucodes != nullptr;
    float acc[2][kMaxTokens];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m) acc[j][m] = 0.f;
    for (int k = lane; k < K; k += 32) {
        const float w0 = weight_at(a.fmt, a.codes, a.q_hi, a.scales, a.mins, K, n, k);
        float w1 = 0.f;
        if (a.swiglu)
            w1 = sep_up ? weight_at(a.ufmt, a.ucodes, a.uq_hi, a.uscales, a.umins, K, n, k)
                        : weight_at(a.fmt, a.codes, a.q_hi, a.scales, a.mins, K, n + n_out, k);
        const float gk = a.norm_w != nullptr ? bf16_bits_to_f32(a.norm_w[k]) : 0.f;
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m) {
            if (m < M) {
                float xv = bf16_bits_to_f32(a.x[static_cast<size_t>(m) * K + k]);
                if (a.norm_w != nullptr) xv = __bfloat162float(__float2bfloat16_rn((xv * s_r[m]) * gk));
                acc[0][m] = fmaf(w0, xv, acc[0][m]);
                if (a.swiglu) acc[1][m] = fmaf(w1, xv, acc[1][m]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[j][m] += __shfl_xor_sync(0xffffffffu, acc[j][m], o);
    if (lane != 0) return;
    for (int m = 0; m < M; ++m) {
        float v = acc[0][m] * a.g;
        if (a.swiglu) {
            const float u = acc[1][m] * (sep_up ? a.ug : a.g);
            v = (v / (1.0f + expf(-v))) * u;
        }
        if (a.residual) v += bf16_bits_to_f32(a.residual[static_cast<size_t>(m) * n_out + n]);
        if (a.out_f32)
            static_cast<float*>(a.y)[static_cast<size_t>(m) * n_out + n] = v;
        else
            static_cast<uint16_t*>(a.y)[static_cast<size_t>(m) * n_out + n] = f32_to_bf16_bits_rn(v);
    }
}

// Dequantise with the same device decode as the tensor-core kernel:
// NVFP4: f16(e2m1) * f16(e4m3) (exact f16 product) -> fp32, times g.
// Q: q through the 1024 + q f16 mantissa, then fmaf(scale, q, min).
__global__ void dequant_kernel(int fmt, const uint8_t* codes, const uint8_t* q_hi, const void* scales,
                               const void* mins, float g, float* w, int N, int K)
{
    const size_t pair = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t total_pairs = static_cast<size_t>(N) * (K / 2);
    if (pair >= total_pairs) return;
    const int n = static_cast<int>(pair / (K / 2));
    const int k = static_cast<int>(pair % (K / 2)) * 2;
    const uint32_t b = codes[pair];
    float w0, w1;
    if (fmt == FMT_NVFP4) {
        const uint32_t s = static_cast<const uint8_t*>(scales)[static_cast<size_t>(n) * (K / 16) + k / 16];
        const uint32_t sc = e4m3x2_to_f16x2(s | (s << 8));
        const uint32_t p = hmul2(e2m1x2_to_f16x2(b), sc);
        w0 = half_bits_to_f32(p & 0xFFFFu) * g;
        w1 = half_bits_to_f32(p >> 16) * g;
    } else {
        uint32_t u = (b & 0xFu) | ((b >> 4) << 16) | 0x64006400u;
        if (fmt == FMT_Q5) {
            const uint32_t hb = q_hi[static_cast<size_t>(n) * (K / 8) + k / 8] >> (k & 7);
            u |= ((hb & 1u) << 4) | (((hb >> 1) & 1u) << 20);
        }
        const uint32_t q = hsub2(u, 0x64006400u);
        const size_t gi = static_cast<size_t>(n) * (K / 32) + k / 32;
        const float s = half_bits_to_f32(static_cast<const uint16_t*>(scales)[gi]);
        const float m = half_bits_to_f32(static_cast<const uint16_t*>(mins)[gi]);
        w0 = fmaf(s, half_bits_to_f32(q & 0xFFFFu), m);
        w1 = fmaf(s, half_bits_to_f32(q >> 16), m);
    }
    w[static_cast<size_t>(n) * K + k] = w0;
    w[static_cast<size_t>(n) * K + k + 1] = w1;
}

}  // namespace

qg_status launch_simple_args(const SimpleArgs& a, cudaStream_t stream)
{
    const int threads = 256;  // 8 warps: one per token for the RMSNorm factors
    const long long blocks = (static_cast<long long>(a.n_out) * 32 + threads - 1) / threads;
    simple_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status launch_simple(int fmt, const uint8_t* codes, const uint8_t* q_hi, const void* scales,
                        const void* mins, float g, const void* x, void* y, int out_f32,
                        const void* residual, int M, int N, int K, int swiglu, cudaStream_t stream)
{
    SimpleArgs a{};
    a.fmt = fmt;
    a.codes = codes;
    a.q_hi = q_hi;
    a.scales = scales;
    a.mins = mins;
    a.g = g;
    a.x = static_cast<const uint16_t*>(x);
    a.y = y;
    a.out_f32 = out_f32;
    a.residual = static_cast<const uint16_t*>(residual);
    a.M = M;
    a.n_out = swiglu ? N / 2 : N;
    a.K = K;
    a.swiglu = swiglu;
    return launch_simple_args(a, stream);
}

// Streaming-read probe: every thread keeps kProbeUnroll 128-bit loads in
// flight over a grid-stride walk of the buffer and XORs the words it reads;
// the warps' results are XORed into *sink.
namespace {

constexpr int kProbeUnroll = 8;
constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4* __restrict__ p, size_t n16,
                                                                   uint32_t* sink)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
    size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) v[u] = ldg_nc_128(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ldg_nc_128(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    acc = __reduce_xor_sync(0xffffffffu, acc);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

qg_status launch_read_probe(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream)
{
    const size_t n16 = bytes / 16;
    if (n16 == 0) return QG_OK;
    const int sms = sm_count(-1);
    if (sms <= 0) return QG_ERR_CUDA;
    // four resident CTAs per SM, fewer for small buffers
    const size_t per_cta = static_cast<size_t>(kProbeThreads) * kProbeUnroll;
    const size_t blocks = std::min<size_t>(static_cast<size_t>(4) * sms, (n16 + per_cta - 1) / per_cta);
    read_probe_kernel<<<static_cast<unsigned>(blocks), kProbeThreads, 0, stream>>>(
        static_cast<const uint4*>(buf), n16, sink);
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

qg_status launch_dequant(int fmt, const uint8_t* codes, const uint8_t* q_hi, const void* scales,
                         const void* mins, float g, float* w, int N, int K, cudaStream_t stream)
{
    const size_t pairs = static_cast<size_t>(N) * (K / 2);
    const int threads = 256;
    const size_t blocks = (pairs + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFull) return QG_ERR_UNSUPPORTED;
    dequant_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(fmt, codes, q_hi, scales, mins, g, w, N,
                                                                           K);
    return cudaPeekAtLastError() == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}

}  // namespace qg
