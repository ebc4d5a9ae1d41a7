// qgemv_internal.h -- types shared by the host launchers and the kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "qgemv.h"

namespace qg {

enum Fmt : int { FMT_NVFP4 = 0, FMT_Q4 = 1, FMT_Q5 = 2 };
enum Epi : int { EPI_NONE = 0, EPI_RESID = 1, EPI_SWIGLU = 2 };

constexpr int kConsumerWarps = 16;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one weight-streaming warp
constexpr int kChunkK = 256;                          // k per pipeline stage
constexpr int kMaxTokens = 8;                         // MMA n dimension
constexpr int kMaxRowsPerCta = 256;                   // TMA box limit
constexpr int kMaxStages = 32;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;    // 2 s

// Per-stage shared-memory layout (byte offsets inside one stage buffer).
struct StageLayout {
    uint32_t codes;      // NVFP4 codes / Q q_lo: rows x 128 B, 128B-swizzled (gate rows for SwiGLU)
    uint32_t codes2;     // SwiGLU up rows (same shape)
    uint32_t scales;     // NVFP4 scales rows x 16 B; Q scale rows x 16 B (8 x fp16)
    uint32_t scales2;    // SwiGLU up-row scales
    uint32_t mins;       // Q min rows x 16 B
    uint32_t hi;         // Q5 high plane rows x 32 B
    uint32_t x;          // Q4/Q5: the stage's raw bf16 activations, M rows x 512 B
    uint32_t bytes;      // total stage size (multiple of 1024)
    uint32_t tx_bytes;   // bytes the TMA writes per stage
};

// A group shares one set of activation rows (the MMA's 8 token columns):
// column j reads activation row x_row[j] and writes output row out_row[j]
// (-1: not stored). Grouped launches (MoE) take their units from device memory.
struct GroupDesc {
    int ntok;        // columns in use (the rest are zero)
    int e;           // expert id (per-expert global scale)
    int xkey;        // groups with equal xkey read the same activation rows
    int x_row[8];
    int out_row[8];
};

// A pair group of the grouped CUDA-core MoE kernels: one or two tokens of one
// expert. Pass v of a launch is group v / blocks over the expert's row block
// v % blocks.
struct CcPair {
    int e;           // expert id (per-expert global scale)
    int ntok;        // 1 or 2
    int x_row[2];    // activation rows (x_row[1] repeats x_row[0] for one token)
    int out_row[2];  // output rows
};

struct UnitDesc {
    int grp;         // index into the group array
    int w_row0;      // first weight row (gate row for SwiGLU)
    int rows;        // rows in this unit (<= rows_per_cta)
    int out_col0;    // first output column
};

struct DenseArgs {
    const uint16_t* x;         // bf16 activations, rows of K values
    void* y;                   // output rows of out_pitch values
    const uint16_t* residual;  // bf16, same layout as y, or nullptr
    int M;                     // dense: tokens; grouped: max columns per group
    int K;
    int n_out;                 // dense: output columns (logical rows)
    int out_pitch;             // elements per output row
    int rows_per_cta;          // R (box rows)
    int up_row_offset;         // SwiGLU: up row = gate row + this
    int out_f32;
    float g;
    const GroupDesc* groups;   // grouped mode (nullptr for dense)
    const UnitDesc* units;
    const int* n_units;
    const float* gscales;      // per-expert global scale (grouped mode)
    int n_stages;
    int ksc;                   // k per activation super-chunk
    int x_pitch;               // f16 elements per token row of the activation buffer
    uint32_t smem_ring;        // offsets in dynamic shared memory
    uint32_t smem_x;
    uint32_t smem_xraw;
    uint32_t smem_exp;
    uint32_t smem_flag;
    uint32_t smem_sum;
    uint32_t smem_red;
    uint32_t smem_bar;
    StageLayout st;
    uint64_t wait_ns;
    int starve;
    int* status;               // device status word
};

// The exact warp-per-row kernel (qgemv_simple.cu): any K, any M, every
// epilogue, the RMSNorm prologue and SwiGLU with a separate up matrix.
struct SimpleArgs {
    int fmt;                   // FMT_NVFP4, FMT_Q4, FMT_Q5 (the gate matrix for SwiGLU)
    const uint8_t* codes;
    const uint8_t* q_hi;
    const void* scales;
    const void* mins;
    float g;
    int ufmt;                  // SwiGLU up matrix when ucodes != nullptr, else the up rows
    const uint8_t* ucodes;     // follow the gate rows in the same matrix
    const uint8_t* uq_hi;
    const void* uscales;
    const void* umins;
    float ug;
    const uint16_t* x;
    void* y;
    int out_f32;
    const uint16_t* residual;
    const uint16_t* norm_w;    // RMSNorm gamma (bf16 [K]) or nullptr
    float norm_eps;
    int M;
    int n_out;
    int K;
    int swiglu;
};

// Host-side helpers implemented in api.cu.
struct DebugState {
    uint64_t wait_ns;
    int starve;
};
DebugState debug_state();
int* device_status_ptr();  // address of the status word on the current device
int sm_count(int device);
bool encode_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                    uint64_t inner_elems, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                    bool swizzle128);
bool encode_tmap_chunks(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                        uint64_t inner_elems, uint64_t rows, uint64_t chunks, uint32_t box_rows, uint32_t box_chunks,
                        bool swizzle128);

qg_status launch_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                             int out_f32, const void* residual, int M, int N, int K, int swiglu,
                             cudaStream_t stream);
// One groupwise-int matrix: q_lo u8[rows][K/2], q_hi (Q5) u8[rows][K/8],
// fp16 scale and min [rows][K/32].
struct Q45Matrix {
    const uint8_t* q_lo;
    const uint8_t* q_hi;
    const void* scale;
    const void* min;
    int bits;
};

// One-token kernels on the CUDA cores (qgemv_cc.cu): QG_ERR_UNSUPPORTED for
// M != 1 or when a shape does not fit their shared-memory plan. norm_w: the
// RMSNorm prologue's gamma (bf16 [K]) or nullptr.
qg_status launch_cc_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_cc_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                              const void* x, void* y, int out_f32, const void* residual, int M, int N, int K,
                              cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_cc_swiglu_q45(const Q45Matrix& gate, const Q45Matrix& up, const void* x, void* y, int M, int I,
                               int K, cudaStream_t stream, const void* norm_w, float norm_eps);
// tcgen05 kernels (NVFP4): QG_ERR_UNSUPPORTED when a shape does not fit their
// shared-memory plan; the callers then use the mma.sync kernels above.
qg_status launch_tc_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_tc_grouped_nvfp4(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu,
                                  int up_offset, const void* x, int max_cols, void* y, int out_pitch, int out_f32,
                                  const GroupDesc* groups, const UnitDesc* units, const int* n_units,
                                  const float* gscales, int rows_per_unit, cudaStream_t stream);
qg_status launch_mt_dense_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, const void* x, void* y,
                                int out_f32, const void* residual, int M, int N, int K, int swiglu,
                                cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_mt_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min, int bits,
                              const void* x, void* y, int out_f32, const void* residual, int M, int N, int K,
                              cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_mt_swiglu_q45(const Q45Matrix& gate, const Q45Matrix& up, const void* x, void* y, int M, int I, int K,
                               cudaStream_t stream, const void* norm_w = nullptr, float norm_eps = 0.f);
qg_status launch_cc_moe(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu, int up_offset,
                        int expert_rows, int blocks, const void* x, int n_x_rows, void* y, int out_pitch, int out_f32,
                        const CcPair* pairs, const int* n_pairs, int max_pairs, const float* gscales, int R,
                        cudaStream_t stream, bool launch = true);
qg_status launch_dense_q45(const uint8_t* q_lo, const uint8_t* q_hi, const void* scale, const void* min,
                           int bits, const void* x, void* y, int out_f32, const void* residual, int M,
                           int N, int K, cudaStream_t stream);
qg_status launch_grouped_nvfp4(const uint8_t* codes, const uint8_t* scales, int total_rows, int K, int swiglu,
                               int up_offset, const void* x, int max_cols, void* y, int out_pitch, int out_f32,
                               const GroupDesc* groups, const UnitDesc* units, const int* n_units,
                               const float* gscales, int rows_per_unit, cudaStream_t stream);
qg_status launch_simple(int fmt, const uint8_t* codes, const uint8_t* q_hi, const void* scales,
                        const void* mins, float g, const void* x, void* y, int out_f32,
                        const void* residual, int M, int N, int K, int swiglu, cudaStream_t stream);
qg_status launch_simple_args(const SimpleArgs& a, cudaStream_t stream);
qg_status launch_read_probe(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream);
qg_status launch_dequant(int fmt, const uint8_t* codes, const uint8_t* q_hi, const void* scales,
                         const void* mins, float g, float* w, int N, int K, cudaStream_t stream);
qg_status launch_route(const float* logits, int M, int E, int topk, int32_t* ids, float* w,
                       cudaStream_t stream);
qg_status launch_moe(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_g,
                     const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_g, const void* x,
                     const int32_t* ids, const float* tw, void* y, void* ws, size_t ws_bytes, int M,
                     int H, int I, int E, int topk, cudaStream_t stream);
size_t moe_workspace_bytes(int M, int topk, int H, int I, int E);
// One persistent launch for a list of one-token projections (qgemv_chain.cu);
// QG_ERR_UNSUPPORTED when the list does not fit its plan.
qg_status launch_chain(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, cudaStream_t stream);
// 3..8 tokens with the activations converted once into a workspace of
// chain_workspace_bytes() (qgemv_chain_ws.cu).
size_t chain_workspace_bytes(const qg_gemv_op* ops, int n_ops, int M);
qg_status launch_chain_ws(const qg_gemv_op* ops, int n_ops, int M, uint32_t* sync, void* workspace,
                          cudaStream_t stream);

}  // namespace qg
