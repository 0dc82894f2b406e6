// Host-side launchers of the mixer-core kernels, called by the C ABI layer
// after it has validated every argument (m2_abi.cu). Each returns the
// cudaError_t of its launches.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mamba2.h"

namespace m2 {

struct Shape {
    int H, P, N, G, K;
    bool bf16;  // activation dtype: true = bf16, false = fp32
    __host__ __device__ long HP() const { return (long)H * P; }
    __host__ __device__ long GN() const { return (long)G * N; }
    __host__ __device__ long CH() const { return HP() + 2 * GN(); }
};

struct StepArgs {
    Shape s;
    int S;  // sessions
    const void *x, *B, *C, *dt_raw;
    // elements from one session's row of x, of B and C, and of dt_raw to the
    // next (dense: H*P, G*N, H; rows of one projection output: its width)
    long sx, sbc, sdt;
    const float *A_log, *D, *dt_bias, *conv_w, *conv_b;
    float* ssm;
    void* conv;
    void* y;
    float* ws_u;   // [S, CH] post-conv, post-SiLU activations of this frame
    float* ws_dt;  // [S, H] softplus'd step sizes
};

size_t step_workspace_bytes(const Shape& s, int S);
cudaError_t launch_step(const StepArgs& a, cudaStream_t st);

struct ScanArgs {
    Shape s;
    int batch, T, chunk;
    const void *x, *B, *C, *dt_raw;
    // elements from one frame's row of x, of B and C, and of dt_raw to the
    // next (dense: H*P, G*N, H); sequence b starts at row b*T
    long fx, fbc, fdt;
    const float *A_log, *D, *dt_bias, *conv_w, *conv_b;
    const float* init_ssm;
    const void* init_conv;
    void* y;
    float* final_ssm;
    void* final_conv;
    void* ws;
    size_t ws_bytes;
    unsigned int* err;  // device error word
    const int* lens;    // [batch] frames used per sequence, device (NULL: T for all)
};

struct NormArgs {
    Shape s;
    int rows;  // positions
    const void* y;
    const void* z;
    const float* weight;
    float eps;
    void* out;
};

// Gated RMSNorm of the mixer output (y * silu(z), grouped RMS, weight).
cudaError_t launch_gated_norm(const NormArgs& a, cudaStream_t st);

// How each row of a linear layer's input is formed before the product:
// kind 0: x as it is; kind 1: RMSNorm of the whole row, x * weight /
// sqrt(mean(x^2) + eps); kind 2: gated RMSNorm, v = x * silu(z) normalised
// over `groups` contiguous blocks, v * weight / sqrt(mean_block(v^2) + eps).
// The normalised row is rounded to bf16 (as a separate norm kernel would
// store it) before it enters the product.
constexpr int kMaxNormGroups = 64;
struct RowNorm {
    int kind;
    const float* weight;  // [in] fp32 (kinds 1, 2)
    float eps;
    int groups;           // kind 2 (kind 1: 1)
    const void* gate;     // kind 2: z, bf16, one row per row of x
    long gate_stride;     // elements between rows of z
};

// 4-bit affine group-quantized linear layer (group 64): y = x W^T (+ residual).
constexpr int kQlMaxIn = 16384;  // input features, at most
struct QLinearArgs {
    int rows, in, out;
    const void* x;            // [rows, in] bf16, rows x_stride elements apart
    long x_stride;
    RowNorm norm;
    const uint32_t* wq;       // [out, in/8]: eight 4-bit fields per word, the first input lowest
    const uint16_t* scales;   // [out, in/64] bf16
    const uint16_t* biases;   // [out, in/64] bf16
    const void* residual;     // NULL, or [rows, out] bf16 added before the rounding (may alias y)
    void* y;                  // [rows, out] bf16
    unsigned int* err;        // device error word
};
// Rows of x the kernel takes per pass over the weights (0: `in` too large).
int qlinear_rows_per_pass(int in);
cudaError_t launch_qlinear(const QLinearArgs& a, cudaStream_t st);
// The same layer as a tensor-core GEMM over tiles of 128 rows of x (no row
// norm; x 16-byte aligned with rows a multiple of 16 bytes apart).
cudaError_t launch_qgemm(const QLinearArgs& a, cudaStream_t st);
// out[r] = row r of x normalised (RowNorm kind 1 or 2) and rounded to bf16,
// bit for bit as the fused linear layers stage it; out is [rows, in].
cudaError_t launch_row_norm(const RowNorm& nm, const void* x, long x_stride, int rows, int in, void* out,
                            cudaStream_t st);
// Rows of x from which launch_qlinear takes the GEMM (when no norm is fused):
// measured, the decode kernel's passes of four rows cost more from about 20
// rows (in_proj's shape) to 36 (out_proj's, whose 70 output tiles fill half
// the SMs).
constexpr int kQgemmMinRows = 40;

// Dense bf16 linear layer for the few rows of a decode step: y = x W^T (+ residual).
constexpr int kLinMaxIn = 16384;
struct LinearArgs {
    int rows, in, out;
    const void* x;        // [rows, in] bf16, rows x_stride elements apart
    long x_stride;
    RowNorm norm;
    const void* w;        // [out, in] bf16
    const void* residual; // NULL, or [rows, out] bf16 (may alias y)
    void* y;              // [rows, out] bf16, rows y_stride elements apart
    long y_stride;
};
cudaError_t launch_linear_bf16(const LinearArgs& a, cudaStream_t st);

// One cached decode position of grouped-query attention with KV-cache append.
constexpr int kAttnD = 128;     // head_dim
constexpr int kAttnMaxR = 8;    // query heads per kv head, at most
struct AttnArgs {
    int S, Hq, Hkv, Tmax;
    bool bf16;                  // activation dtype: true = bf16, false = fp32
    const int* lens;            // [S] positions already cached (device)
    const void *q, *k_new, *v_new;
    void *k_cache, *v_cache;    // [S, Hkv, Tmax, D], updated at position lens[s]
    float scale;                // softmax scale of q.k
    void* out;                  // [S, Hq, D]
    float* ws;                  // per-chunk partial results
    unsigned int* err;          // device error word
    int tc;                     // positions per chunk (set by the launcher)
    // elements from one session's q, k_new / v_new and out to the next's
    // (dense: Hq*D, Hkv*D, Hq*D), and a count added to every length (the
    // positions of a prefill after the first)
    long q_ss, kv_ss, out_ss;
    int len_add;
};
size_t attn_workspace_bytes(int S, int Hq, int Hkv, int Tmax, bool bf16);
cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st);

// Records a CUDA error for mamba2_last_cuda_error() on the calling thread.
void record_cuda_error(cudaError_t e);

// The argument checks of mamba2_step before its workspace check: dimensions,
// session count, NULL and misaligned pointers (M2_OK when they pass).
m2_status check_step_args(const m2_dims* d, int n_sessions, const void* x, const void* B, const void* C,
                          const void* dt_raw, const float* A_log, const float* D, const float* dt_bias,
                          const float* conv_w, const float* conv_b, const float* ssm_state,
                          const void* conv_state, const void* y);
// M2_OK when the current device is an sm_103 GPU (and its set-up is done).
m2_status check_device();
// The device error word of the current device (after check_device).
unsigned int* device_error_word();

size_t scan_workspace_bytes(const Shape& s, int batch, int T, int chunk);
// B/C conv prologue into the workspace tiles (first half of a scan).
cudaError_t launch_scan_prepare(const ScanArgs& a, cudaStream_t st);
// Fused chunked SSD over prepared tiles, final state and conv tail (second half).
// after_prologue: the launch directly follows launch_scan_prepare of the same
// call on the stream (allows an early, programmatically dependent start).
cudaError_t launch_scan_chunks(const ScanArgs& a, bool after_prologue, cudaStream_t st);

}  // namespace m2
