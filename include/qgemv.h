/*
 * qgemv.h -- C ABI of libqgemv: decode-step GEMV / skinny GEMM (M = 1..8
 * tokens) over low-bit block-scaled weights on one NVIDIA GB300 (sm_103a).
 *
 * What the pages say this is: single-GPU decode is memory-bandwidth bound and
 * engines write one native fused kernel per weight format -- matmul, residual
 * add and SwiGLU done in "one read, one write" -- with NVFP4 artefacts and a
 * groupwise-int Q4/Q5 recipe (NInfer article, section 2 "自研 CUDA 算子
 * 混合量化权重"); an "NVFP4 / MXFP8 block matvec" kernel and a "Top-8 gating
 * and softmax" MoE router (Decapybara README, "Blackwell CUDA 内核套件",
 * mx_gemv.cu and moe.cu); 1..8 concurrent decode lanes batched into one step
 * (NInfer article, section 1 "单卡专用架构"). The pages print no bit layout;
 * the layouts below are this library's contract.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *     16-byte aligned (else QG_ERR_MISALIGNED). The library allocates no
 *     device memory per call; it owns one 4-byte device status word.
 *   - Work is enqueued on `stream` (0 = legacy default stream) and the call
 *     returns without synchronising. Inputs must stay valid and unmodified,
 *     and outputs untouched by others, until the stream work completes.
 *     Outputs must not alias inputs, except `residual` == `y` (in place).
 *   - Arguments are validated before anything is launched; a rejected call
 *     launches nothing. A launch failure returns QG_ERR_CUDA and leaves the
 *     CUDA error retrievable with cudaGetLastError().
 *   - The library caches per-device state (the status word's address,
 *     kernel attributes) for the life of the process; after cudaDeviceReset
 *     it must not be called again on that device.
 *   - Activations x and residuals are bf16 [M][K] / [M][N]; M in [1, 8]
 *     (the 1..8 decode lanes); K % 32 == 0 and K >= 32; N >= 1.
 *   - Weights are read once per call; accumulation is fp32.
 *
 * Weight formats
 *   NVFP4: codes u8[N][K/2], two FP4 E2M1 codes per byte, the low nibble
 *          holding the even k; scales u8[N][K/16], one FP8 E4M3 (OCP "FN"
 *          variant) per 16 consecutive k; one fp32 per-tensor scale g.
 *          w[n][k] = e2m1(code) * e4m3(scale[n][k/16]) * g.
 *   Q4/Q5: q_lo u8[N][K/2] (low 4 bits of the unsigned code, low nibble =
 *          even k); Q5 adds q_hi u8[N][K/8] holding the 5th bit of k as bit
 *          k%8 of byte k/8; scale and min are fp16 [N][K/32].
 *          w[n][k] = scale[n][k/32] * q + min[n][k/32].
 *
 * Output accuracy: for every output element, with B = 1e-4 * sum_k |w x| +
 * 1e-6, an fp32 output lies within B of the exact sum, and a bf16 output is
 * the round-to-nearest-even of a value within B of it. Dequantised weights
 * (qdequant_*) are bit-exact fp32 roundings of the exact weight values.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,    /* a size, pointer or enum is out of range   */
    QG_ERR_UNSUPPORTED = 2,    /* valid request this build does not serve    */
    QG_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned           */
    QG_ERR_WORKSPACE = 4,      /* a workspace missing or too small           */
    QG_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed       */
    QG_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait ran out         */
} qg_status;

typedef enum { QG_OUT_BF16 = 0, QG_OUT_F32 = 1 } qg_out;

/*
 * y[m][n] = g * sum_k e2m1(code[n][k]) * e4m3(scale[n][k/16]) * x[m][k]
 *           (+ residual[m][n])
 * NVFP4 dense GEMV with an optional fused residual add (NInfer article,
 * section 2: fused matmul + residual add per weight format).
 *   codes    u8[N][K/2]     scales u8[N][K/16]     global_scale g (by value)
 *   x        bf16[M][K]     y bf16 or fp32 [M][N] per y_dtype
 *   residual bf16[M][N] or NULL (added in fp32 before the output rounding)
 */
QG_API qg_status qgemv_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale,
                      const void* x, void* y, qg_out y_dtype, const void* residual,
                      int M, int N, int K, cudaStream_t stream);

/*
 * y[m][n] = sum_k (scale[n][k/32] * q[n][k] + min[n][k/32]) * x[m][k]
 *           (+ residual[m][n])
 * Groupwise-int Q4/Q5 GEMV (NInfer article, section 2: the groupwise-int
 * recipe puts Q/K projections in Q4 and gate/V in Q5).
 *   q_lo u8[N][K/2]; q_hi u8[N][K/8] for bits == 5, must be NULL for bits == 4
 *   scale, min fp16[N][K/32]; bits in {4, 5}; x, y, y_dtype, residual as above.
 */
QG_API qg_status qgemv_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min,
                    int bits, const void* x, void* y, qg_out y_dtype, const void* residual,
                    int M, int N, int K, cudaStream_t stream);

/*
 * SwiGLU-fused NVFP4 gate/up projection (NInfer article, section 2: fused
 * SwiGLU). The N = 2I weight rows are the gate rows [0, I) followed by the up
 * rows [I, 2I); with a = gate row i and b = up row i,
 *   y[m][i] = bf16_rne( silu(a . x[m]) * (b . x[m]) ),  silu(v) = v / (1 + e^-v).
 *   codes u8[N][K/2], scales u8[N][K/16], g by value, x bf16[M][K],
 *   y bf16[M][N/2]; N must be even.
 */
QG_API qg_status qgemv_swiglu_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale,
                             const void* x, void* y, int M, int N, int K, cudaStream_t stream);

/*
 * MoE router (Decapybara README, moe.cu: "Top-8 gating and softmax"):
 * p = softmax(logits[m]); the topk largest p in descending order, ties to the
 * lower expert id; w = p_top / sum(p_top).
 *   logits fp32[M][E]; topk_ids int32[M][topk] out; topk_w fp32[M][topk] out;
 *   1 <= topk <= 8, topk <= E <= 1024, M in [1, 8].
 */
QG_API qg_status moe_route_topk(const float* logits, int M, int E, int topk, int32_t* topk_ids,
                         float* topk_w, cudaStream_t stream);

/* Bytes of device workspace moe_qgemv_nvfp4 needs for these sizes. */
QG_API qg_status moe_qgemv_nvfp4_workspace_size(int M, int topk, int H, int I, int E, size_t* bytes);

/*
 * Expert-gathered MoE FFN over NVFP4 experts (35B-A3B-class decode layer;
 * NInfer article, section 2, and Decapybara README, moe.cu). For each token m
 * and slot i < topk with e = topk_ids[m][i]:
 *   h[m][i] = bf16_rne( silu(G_e x[m]) * (U_e x[m]) )      (length I)
 *   y[m]    = bf16_rne( sum_{i ascending} topk_w[m][i] * g_dn[e] * D_e h[m][i] )
 * where gate/up rows of expert e are rows [0, I) and [I, 2I) of
 * gu_codes[e] (scaled by gu_gscale[e]) and D_e is dn_codes[e] (scaled by
 * dn_gscale[e]). Each active expert's weights are read once for all of its
 * tokens; the combine is deterministic (fixed slot order, no atomics).
 *   gu_codes u8[E][2I][H/2], gu_scales u8[E][2I][H/16], gu_gscale fp32[E] (device)
 *   dn_codes u8[E][H][I/2],  dn_scales u8[E][H][I/16],  dn_gscale fp32[E] (device)
 *   x bf16[M][H]; topk_ids int32[M][topk]; topk_w fp32[M][topk]; y bf16[M][H]
 *   workspace: caller-owned device memory of at least
 *   moe_qgemv_nvfp4_workspace_size() bytes, 256-byte aligned. It starts with
 *   h as bf16[M][topk][I] (a slot that repeats an expert of the same token,
 *   or names an invalid one, leaves its row unwritten); the rest is private
 *   scratch.
 * Expert ids outside [0, E) are not checked on the host (they are device
 * data); such a slot contributes nothing and records QG_ERR_INVALID_ARG in the
 * device status word (see qg_last_device_status).
 * H % 256 == 0, I % 256 == 0, 1 <= topk <= 8, M in [1, 8].
 */
QG_API qg_status moe_qgemv_nvfp4(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_gscale,
                          const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_gscale,
                          const void* x, const int32_t* topk_ids, const float* topk_w, void* y,
                          void* workspace, size_t workspace_bytes, int M, int H, int I, int E,
                          int topk, cudaStream_t stream);

/*
 * moe_qgemv_nvfp4 without a workspace argument, for callers that cannot
 * allocate device memory: a plugin whose host framework owns all device
 * memory and offers no allocator, or a latency-critical decode loop that may
 * not call cudaMalloc. The pages have no counterpart; this is a library
 * convenience. Arguments and results are those of moe_qgemv_nvfp4.
 *   - The scratch is a fixed 4 MiB device array inside the library image;
 *     once loaded on a GPU it stays there until the process exits. Sizes whose
 *     moe_qgemv_nvfp4_workspace_size() exceeds 4 MiB return QG_ERR_WORKSPACE
 *     (at M = 8 and top-8, H = 4096 with I = 2048 still fits). Arguments are
 *     checked as moe_qgemv_nvfp4 checks them, before the size limit.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture on that device. Under lazy
 *     module loading (the CUDA default) that first call is also when the
 *     driver loads the library's device code on that device and reserves the
 *     4 MiB, so it can fail with QG_ERR_CUDA if device memory is exhausted;
 *     later calls reserve nothing.
 *   - The address is cached per device for the life of the process: do not
 *     call this after cudaDeviceReset on that device.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero). Calls that overlap on the GPU
 *     -- on different streams, or from several host threads -- race; order
 *     them on one stream.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating routine.
 */
QG_API qg_status moe_qgemv_nvfp4_noalloc(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                         const float* gu_gscale, const uint8_t* dn_codes,
                                         const uint8_t* dn_scales, const float* dn_gscale, const void* x,
                                         const int32_t* topk_ids, const float* topk_w, void* y, int M, int H,
                                         int I, int E, int topk, cudaStream_t stream);

/* Weight formats and epilogues of one projection in a chained call. */
typedef enum { QG_FMT_NVFP4 = 0, QG_FMT_Q4 = 1, QG_FMT_Q5 = 2 } qg_format;
typedef enum { QG_EPI_NONE = 0, QG_EPI_RESIDUAL = 1, QG_EPI_SWIGLU = 2 } qg_epilogue;

/*
 * One projection of qgemv_chain: the arguments of qgemv_nvfp4,
 * qgemv_swiglu_nvfp4 or qgemv_q45 in one record (same layouts and rules).
 *   format          qg_format
 *   epilogue        QG_EPI_NONE, QG_EPI_RESIDUAL (residual != NULL) or
 *                   QG_EPI_SWIGLU (NVFP4: N = 2I rows, gate then up, y bf16
 *                   [M][I]; groupwise-int: separate up matrix, see up_*)
 *   y_dtype         qg_out; QG_OUT_BF16 for QG_EPI_SWIGLU
 *   after_previous  nonzero if the op reads memory that an earlier op of the
 *                   same call writes (its x or residual is an earlier y); the
 *                   op then starts reading only once every earlier op of the
 *                   call is complete. Without it the op may overlap earlier
 *                   ops: it must then neither read nor write anything an
 *                   earlier op of the call writes, nor write what one reads.
 *   codes           NVFP4 codes or Q q_lo, u8[N][K/2]
 *   q_hi            Q5 high-bit plane u8[N][K/8]; NULL for NVFP4 and Q4
 *   scales          NVFP4 e4m3 u8[N][K/16], or Q fp16 [N][K/32]
 *   mins            Q fp16 [N][K/32]; NULL for NVFP4
 *   global_scale    NVFP4 tensor scale g (ignored for Q)
 *   x, residual, y  as in the single-projection calls
 *   norm_weight     RMSNorm prologue (NInfer article, section 2: the
 *                   normalisation fused with the matmul, "one read, one
 *                   write"): gamma, bf16 [K], or NULL for none. With it the
 *                   projection reads, per token m, h = bf16_rne(x * r * gamma)
 *                   with r = 1 / sqrt(sum_k x^2 / K + norm_eps), r computed in
 *                   fp32 in one fixed order shared by every kernel.
 *   norm_eps        the RMSNorm epsilon (ignored without norm_weight)
 *   up_format       SwiGLU over separate groupwise-int gate and up matrices
 *   up_codes ...    (NInfer article, section 2: gate in Q5, up in Q4): with
 *                   QG_EPI_SWIGLU and a Q format, the record's own matrix holds
 *                   the I gate rows (N = I), up_codes / up_q_hi / up_scales /
 *                   up_mins the I up rows in up_format (QG_FMT_Q4 or Q5), and
 *                   y is bf16 [M][I]. NULL / 0 otherwise.
 */
typedef struct {
    int format;
    int epilogue;
    int y_dtype;
    int after_previous;
    int N;
    int K;
    const uint8_t* codes;
    const uint8_t* q_hi;
    const void* scales;
    const void* mins;
    float global_scale;
    const void* x;
    const void* residual;
    void* y;
    const void* norm_weight;
    float norm_eps;
    int up_format;
    const uint8_t* up_codes;
    const uint8_t* up_q_hi;
    const void* up_scales;
    const void* up_mins;
} qg_gemv_op;

/*
 * The projections of a decode layer in order, as one call (NInfer article,
 * section 1: a decode step is one fixed sequence replayed per batch size;
 * Decapybara README, "Blackwell CUDA 内核套件": a persistent single-launch
 * decode loop, megakernel.cu). Each op computes exactly what its
 * single-projection call computes, with the same accuracy.
 *   ops     host array of n_ops records, 1 <= n_ops <= 8 (read during the call)
 *   M       tokens, 1..8, shared by every op
 *   sync    two caller-owned device words (uint32_t[2], 16-byte aligned), zero
 *           before their first use; every call returns the first word to zero
 *           (the second counts completed barriers), so they are reusable. Needed
 *           (else QG_ERR_INVALID_ARG) when some op after the first has
 *           after_previous set; may be NULL otherwise. Calls that overlap on
 *           the GPU must use different words, and after a call that reported
 *           QG_ERR_DEVICE_TIMEOUT the words must be zeroed again.
 * When K is a multiple of 256 for every op, the list runs as one persistent
 * kernel (one CTA per SM, launched cooperatively when an op waits for earlier
 * ones): the weight stream runs on across op boundaries. Other lists (an op
 * whose K is not a multiple of 256, or one that does not fit the kernel's
 * shared memory) run as one launch per op,
 * in order, on `stream`; a single record is thus also the way to call any
 * projection with the RMSNorm prologue.
 * Every op is validated before anything is launched.
 */
QG_API qg_status qgemv_chain(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, cudaStream_t stream);

/*
 * qgemv_chain with a workspace: the same ops, the same results (bit for
 * bit), and at M = 3..8 a faster plan. A small kernel first converts every
 * op's activations once (the exact f16 prescale per 256-k chunk that each
 * kernel otherwise repeats per CTA) into the workspace, and the layer
 * kernel's TMA warp streams them into shared memory beside the weights; an
 * op with after_previous is converted inside the layer kernel after its
 * grid-wide barrier (an op with after_previous and norm_weight falls back to
 * qgemv_chain's plan). At M = 1..2 the workspace is not used.
 *   workspace        device memory of at least
 *                    qgemv_chain_workspace_size() bytes, 256-byte aligned
 *                    (else QG_ERR_MISALIGNED); NULL runs qgemv_chain. Its
 *                    contents need no initialisation and are scratch after
 *                    the call; calls that may overlap on the GPU need
 *                    separate workspaces.
 *   workspace_bytes  its size (QG_ERR_WORKSPACE if too small)
 * Other arguments and errors as for qgemv_chain.
 */
QG_API qg_status qgemv_chain_ws(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * Bytes of qgemv_chain_ws's workspace for these ops and M: for each op,
 * K/256 blocks of M * 576 + 48 bytes (NVFP4) or M * 576 + 304 bytes
 * (Q4/Q5), rounded up to 256. QG_ERR_INVALID_ARG for a null pointer, n_ops
 * outside 1..8, M outside 1..8 or K < 1; nothing is launched.
 */
QG_API qg_status qgemv_chain_workspace_size(const qg_gemv_op* ops, int n_ops, int M, size_t* bytes);

/*
 * SwiGLU over separate groupwise-int gate and up matrices, for the recipe
 * that puts gate in Q5 and up in Q4 (NInfer article, section 2), with an
 * optional fused RMSNorm prologue:
 *   y[m][i] = bf16_rne( silu(gate_i . h_m) * (up_i . h_m) ),
 *   h_m = x_m, or bf16(x_m * r_m * gamma) with norm_weight (see qg_gemv_op)
 *   gate_lo u8[I][K/2], gate_hi u8[I][K/8] (gate_bits == 5, else NULL),
 *   gate_scale, gate_min fp16 [I][K/32]; the same for up_*; bits in {4, 5}
 *   x bf16 [M][K]; norm_weight bf16 [K] or NULL; y bf16 [M][I].
 * Validation and errors as for qgemv_q45.
 */
QG_API qg_status qgemv_swiglu_q45(const uint8_t* gate_lo, const uint8_t* gate_hi, const void* gate_scale,
                                  const void* gate_min, int gate_bits, const uint8_t* up_lo, const uint8_t* up_hi,
                                  const void* up_scale, const void* up_min, int up_bits, const void* x,
                                  const void* norm_weight, float norm_eps, void* y, int M, int I, int K,
                                  cudaStream_t stream);

/*
 * Dequantise to fp32 w[N][K] with the same device decode the GEMV kernels
 * use (test hook for the bit-exact check). NVFP4: w = fp32(e2m1 * e4m3) * g,
 * one rounding. Q4/Q5: w = fmaf(scale, q, min), one rounding.
 */
QG_API qg_status qdequant_nvfp4(const uint8_t* codes, const uint8_t* scales, float global_scale,
                         float* w, int N, int K, cudaStream_t stream);
QG_API qg_status qdequant_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min,
                       int bits, float* w, int N, int K, cudaStream_t stream);

/*
 * Streaming-read probe for the measurement of a GEMV against the memory
 * roofline: reads the `bytes` of device buffer `buf` once, with 128-bit
 * non-coherent loads from every SM, and XORs all its 32-bit words into the
 * device word *sink (caller-owned, not cleared: afterwards *sink equals its
 * old value XOR the buffer's words), so the loads cannot be elided and the
 * result can be checked. Timing it with events gives the read-only HBM
 * bandwidth a weight-streaming kernel can reach, next to the copy bandwidth.
 *   buf: 16-byte aligned, bytes a multiple of 16 (0 launches nothing, and
 *   buf may then be null);
 *   sink: 4-byte aligned.
 * QG_ERR_INVALID_ARG for a null pointer or a ragged size, QG_ERR_MISALIGNED
 * for misaligned pointers; asynchronous on `stream`.
 */
QG_API qg_status qg_read_probe(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream);

/*
 * Synchronise `stream`, then return and clear the device status word:
 * QG_OK, QG_ERR_DEVICE_TIMEOUT when a bounded device-side wait gave up (the
 * kernel stopped early; its outputs are undefined), or QG_ERR_INVALID_ARG for
 * out-of-range device data (MoE expert ids).
 */
QG_API qg_status qg_last_device_status(cudaStream_t stream);

/* Static, NUL-terminated name of a status code. */
QG_API const char* qg_status_string(qg_status status);

/*
 * Fault-injection hook for testing the bounded-wait path. Sets the time
 * limit (ns) of every device-side wait for subsequent launches on this host
 * thread's process (0 restores the default of two seconds). With
 * starve != 0, the weight-streaming warps of the dense kernels issue no copies, so
 * the consumer waits run out and the kernels return early with
 * QG_ERR_DEVICE_TIMEOUT recorded. Not for production use.
 */
QG_API qg_status qg_debug_set_wait(uint64_t limit_ns, int starve);

#ifdef __cplusplus
}
#endif
#endif /* QGEMV_H */
