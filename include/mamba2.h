/*
 * mamba2.h — C ABI of libmamba2.so, the GB300 (sm_103a) Mamba2 mixer core.
 *
 * The mixer core is the per-layer state-space part of each Mamba ('M') layer
 * of the Nemotron-H language model inside NemotronLabs VoiceChat (issue
 * "feat(nemotron_voicechat): load the VoiceChat checkpoint and run offline
 * duplex inference", sections config.json / text_config and "Network 2";
 * "docs/nemotron-voicechat.md", sections Offline timeline and Online
 * session). Per layer it computes, for every frame t and head h (group
 * g = h / (H/G)):
 *
 *   u_t      = SiLU(conv_b + sum_k conv_w[:,k] * xin_{t-(K-1)+k})   over x|B|C
 *   dt_t,h   = softplus(dt_raw_t,h + dt_bias_h),   A_h = -exp(A_log_h)
 *   h_t      = exp(dt A) h_{t-1} + dt x~_t (outer) B~_t,g
 *   y_t      = h_t . C~_t,g + D_h x~_t
 *
 * (the Mamba-2 selective state-space recurrence, Dao & Gu 2024). It runs in
 * two modes that must agree (VoiceChat doc, Offline timeline: recompute and
 * cached mode give identical tokens):
 *   mamba2_conv_scan — whole history / prefill, chunked (SSD) evaluation;
 *   mamba2_step      — one frame for a batch of sessions from cached state.
 * Around it: the gated output norm and the 4-bit projections of the Mamba
 * layer, and the cached decode of the model's attention layers
 * (mamba2_gated_norm, mamba2_qlinear, mamba2_attn_decode).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every pointer argument is DEVICE memory owned by the caller
 *           (for instance from torch). The library allocates nothing on the
 *           device and keeps no pointer after a call returns.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *           All work is enqueued asynchronously on it; nothing synchronises.
 * Errors.   Argument, shape and alignment checks happen on the host before
 *           anything is enqueued; on failure nothing is launched and the
 *           return value says why. A failed launch returns M2_ECUDA and
 *           mamba2_last_cuda_error() gives the cudaError_t. Errors of kernels
 *           already running surface at the caller's next synchronisation, as
 *           for any CUDA work. Device-side waits are bounded: a wait that
 *           runs out records a code readable with mamba2_device_error().
 * Devices. The library looks up, once per device and on the first call
 *           made there, the device addresses of its own device variables
 *           (the error word; the scratch of mamba2_step_noalloc) and keeps
 *           them for the life of the process. Calls on a device after a
 *           cudaDeviceReset of it are not supported.
 * Layouts.  Contiguous, innermost index last:
 *             x [b,T,H,P]   B, C [b,T,G,N]   dt_raw [b,T,H]   y [b,T,H,P]
 *             ssm state [b,H,P,N] fp32
 *             conv tail [b,K-1,CH], oldest frame first, CH = H*P + 2*G*N,
 *             channel order x | B | C (x at h*P+p, B at H*P+g*N+n,
 *             C at H*P+G*N+g*N+n)
 *             conv_w [CH,K] fp32 (the checkpoint's [CH,K,1] tensor read as
 *             [CH,K]; a torch export [CH,1,K] has the same bytes)
 *             conv_b [CH], A_log, D, dt_bias [H] fp32
 *           The activation dtype (x, B, C, dt_raw, y, conv tail) is
 *           m2_dims.act: bf16 or fp32.
 * Alignment. Every pointer must be 16-byte aligned (M2_EALIGN otherwise).
 * Shapes.   K == 4; N in {16, 32, 64, 128}; P a multiple of 16, at most 80;
 *           H a multiple of G; H*P and G*N multiples of 8. (The Nemotron-H
 *           mixer is H=128, P=80, N=128, G=8, K=4.) M2_ESHAPE otherwise.
 */
#ifndef MAMBA2_H
#define MAMBA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    M2_OK = 0,
    M2_EINVAL = 1,       /* a required pointer is NULL, or a count/size is negative or zero */
    M2_ESHAPE = 2,       /* dimensions outside the supported set (see Shapes above) */
    M2_EALIGN = 3,       /* a pointer is not 16-byte aligned */
    M2_EUNSUPPORTED = 4, /* the current device is not an sm_103 GPU */
    M2_ECUDA = 5,        /* a CUDA runtime call or kernel launch failed */
    M2_EWORKSPACE = 6    /* workspace is NULL or smaller than the query returned */
} m2_status;

typedef enum { M2_BF16 = 0, M2_F32 = 1 } m2_dtype;

typedef struct {
    int batch;     /* b: sequences in a scan (mamba2_step takes n_sessions instead) */
    int T;         /* frames per sequence in a scan (ignored by mamba2_step) */
    int nheads;    /* H, mamba_num_heads */
    int headdim;   /* P, mamba_head_dim */
    int dstate;    /* N, ssm_state_size */
    int ngroups;   /* G, n_groups: B and C are shared by H/G consecutive heads */
    int dconv;     /* K, conv_kernel (must be 4) */
    m2_dtype act;  /* dtype of x, B, C, dt_raw, y and the conv tail */
} m2_dims;

/* Bytes of device scratch that mamba2_conv_scan needs for these dims and
 * chunk length (0 if `d` or `chunk` is invalid). */
size_t mamba2_scan_workspace_bytes(const m2_dims* d, int chunk);

/* Whole-history (or prefill) evaluation of the mixer core over d->T frames
 * of d->batch independent sequences, chunked in pieces of `chunk` frames
 * (SSD form; 1 <= chunk <= 128; T need not be a multiple of it; results do
 * not depend on it beyond rounding).
 *
 * Inputs : x, B, C, dt_raw (act dtype), A_log, D, dt_bias, conv_w, conv_b.
 *          init_ssm [b,H,P,N] fp32 and init_conv [b,K-1,CH] (act dtype) are
 *          the state to continue from; NULL means zeros (a fresh sequence).
 * Outputs: y [b,T,H,P] (act dtype); final_ssm [b,H,P,N] fp32;
 *          final_conv [b,K-1,CH] (act dtype): the last K-1 pre-conv input
 *          frames, bit copies, taken from init_conv where T < K-1.
 *          final_ssm and final_conv may alias init_ssm and init_conv (state
 *          updated in place); no other output may alias any input.
 * Scratch: workspace of at least mamba2_scan_workspace_bytes(d, chunk).
 * T == 0 is valid: y is untouched and the final state equals the initial. */
m2_status mamba2_conv_scan(const m2_dims* d, const void* x, const void* B, const void* C,
                           const void* dt_raw, const float* A_log, const float* D,
                           const float* dt_bias, const float* conv_w, const float* conv_b,
                           int chunk, const float* init_ssm, const void* init_conv, void* y,
                           float* final_ssm, void* final_conv, void* workspace,
                           size_t workspace_bytes, void* stream);

/* mamba2_conv_scan over a batch of sequences of different lengths: catching
 * up several sessions at once, or prefilling prompts of different lengths
 * (each optionally continuing from its own cached state), padded to one T.
 *
 * lengths: device int32 [d->batch], 4-byte aligned; sequence b uses frames
 *   [0, lengths[b]) of its T-frame slots of x, B, C, dt_raw. Values are read
 *   on the device (so they may be produced by earlier work on the stream) and
 *   clamped to [0, T].
 * y: rows t < lengths[b] of sequence b are written; rows at or past it are
 *   left as they were.
 * final_ssm / final_conv: the states after frame lengths[b] - 1 (for a
 *   length of 0, the initial states, copied).
 * Everything else (arguments, layouts, workspace, aliasing, tolerances,
 * errors) is that of mamba2_conv_scan; a NULL lengths returns M2_EINVAL.
 * With every length equal to T the results are those of mamba2_conv_scan. */
m2_status mamba2_conv_scan_varlen(const m2_dims* d, const int* lengths, const void* x, const void* B,
                                  const void* C, const void* dt_raw, const float* A_log, const float* D,
                                  const float* dt_bias, const float* conv_w, const float* conv_b, int chunk,
                                  const float* init_ssm, const void* init_conv, void* y, float* final_ssm,
                                  void* final_conv, void* workspace, size_t workspace_bytes, void* stream);

/* mamba2_conv_scan on inputs that are column slices of wider rows: the x, B,
 * C and dt_raw of frame t of sequence b start in_row_stride * (b*T + t)
 * elements past the x, B, C and dt_raw pointers. That is the layout of the
 * Mamba layer's input projection output, one row per frame holding
 * z | x | B | C | dt (VoiceChat issue, section config.json / text_config:
 * the mixer's in_proj), so x = proj + H*P, B = proj + 2*H*P,
 * C = B + G*N, dt_raw = C + G*N and in_row_stride = 2*H*P + 2*G*N + H (22656
 * at the Nemotron-H shape) read the frame straight from it.
 * in_row_stride > 0 (M2_EINVAL), and in_row_stride times the element size a
 * multiple of 16 bytes (M2_EALIGN). Everything else is mamba2_conv_scan's:
 * with in_row_stride equal to the dense widths the results are identical. */
m2_status mamba2_conv_scan_strided(const m2_dims* d, const void* x, const void* B, const void* C, const void* dt_raw,
                                   long in_row_stride, const float* A_log, const float* D, const float* dt_bias,
                                   const float* conv_w, const float* conv_b, int chunk, const float* init_ssm,
                                   const void* init_conv, void* y, float* final_ssm, void* final_conv,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* The two halves of mamba2_conv_scan, with the same arguments, for callers
 * that schedule or time them separately. mamba2_conv_scan(args) is exactly
 * mamba2_scan_prepare_bc(args) followed by mamba2_scan_chunks(args) on the
 * same stream.
 *   mamba2_scan_prepare_bc: causal conv + SiLU of the B and C channels into
 *     the workspace as tensor-core operand tiles. Reads B, C, conv_w, conv_b,
 *     init_conv; writes only the workspace.
 *   mamba2_scan_chunks: the chunked SSD evaluation over those tiles, with the
 *     head's own x-channel conv, dt, y, final_ssm and final_conv. It must run
 *     after mamba2_scan_prepare_bc with the same B, C, conv weights,
 *     init_conv, chunk and workspace, and before the workspace is reused.
 * Validation and error behaviour are those of mamba2_conv_scan. */
m2_status mamba2_scan_prepare_bc(const m2_dims* d, const void* x, const void* B, const void* C,
                                 const void* dt_raw, const float* A_log, const float* D,
                                 const float* dt_bias, const float* conv_w, const float* conv_b,
                                 int chunk, const float* init_ssm, const void* init_conv, void* y,
                                 float* final_ssm, void* final_conv, void* workspace,
                                 size_t workspace_bytes, void* stream);
m2_status mamba2_scan_chunks(const m2_dims* d, const void* x, const void* B, const void* C,
                             const void* dt_raw, const float* A_log, const float* D,
                             const float* dt_bias, const float* conv_w, const float* conv_b,
                             int chunk, const float* init_ssm, const void* init_conv, void* y,
                             float* final_ssm, void* final_conv, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Gated RMSNorm of the mixer output: the standard Mamba-2 output norm that
 * follows the mixer core in each Mamba layer (the VoiceChat issue
 * "feat(nemotron_voicechat): load the VoiceChat checkpoint and run offline
 * duplex inference", section config.json / text_config, gives
 * rms_norm_eps 1e-5; the pages do not spell out its form, this is the
 * standard one). For each of `rows` positions and each of d->ngroups
 * contiguous blocks of H*P/ngroups channels:
 *     v   = y * silu(z)
 *     out = weight * v / sqrt(mean over the block of v^2 + eps)
 * computed in fp32 and rounded once to the activation dtype.
 *
 * y, z, out: [rows, H*P] (act dtype; any batch x time flattening of the
 *   scan's y [b,T,H,P] or the step's y [S,H,P]); out may alias y or z.
 * weight: [H*P] fp32. eps >= 0 and finite.
 * Errors: M2_EINVAL (NULL pointer, rows < 0, bad eps, bad dims), M2_ESHAPE,
 * M2_EUNSUPPORTED (groups wider than 32768 channels), M2_EALIGN (a pointer
 * not 16-byte aligned), M2_ECUDA. rows == 0 is a no-op once the arguments
 * check out. Asynchronous on `stream`. */
m2_status mamba2_gated_norm(const m2_dims* d, int rows, const void* y, const void* z, const float* weight,
                            float eps, void* out, void* stream);

/* Affine group-quantized linear layer: the Mamba layer's input and output
 * projections as the VoiceChat 4-bit checkpoint stores them (Nemotron
 * VoiceChat page, config.json: `quantization` with group_size 64, bits 4 for
 * the Nemotron-H mixer projections; no bias). Weight (o, i) is the 4-bit
 * field q at bits 4*(i%8) of the 32-bit word wq[o][i/8] (the first input in
 * the lowest bits), dequantized per group of 64 inputs:
 *     W[o][i] = scales[o][i/64] * q + biases[o][i/64]
 *     y[r][o] = sum_i W[o][i] * x[r][i]
 * accumulated in fp32 and rounded once to bf16.
 *
 * x: [rows, in_features] bf16, 16-byte aligned. wq: [out_features,
 *   in_features/8] uint32, 16-byte aligned. scales, biases: [out_features,
 *   in_features/64] bf16. y: [rows, out_features] bf16; must not alias x.
 * Sizes: in_features a multiple of 64, at most 16384 (the Nemotron-H in_proj
 *   has 4480 -> 22656, out_proj 10240 -> 4480); rows >= 0 (rows == 0 is a
 *   no-op once the arguments check out).
 * Forms: below 40 rows (the few rows of a cached decode step) each pass over
 *   the weights takes up to 4 rows of x (2 for in_features above 12480);
 *   from 40 rows (a prefill) the layer runs as a tensor-core GEMM over tiles
 *   of 128 rows, the products of x with the exact bf16 (128 + q) per group
 *   of 64 inputs accumulated in fp32 and scaled per group in fp32. Both give
 *   the same sums in a different order (the results agree within rounding).
 * Errors: M2_EINVAL (NULL pointer, non-positive size), M2_EUNSUPPORTED
 *   (group_size other than 64 or bits other than 4, or not an sm_103 GPU),
 *   M2_ESHAPE (in_features), M2_EALIGN, M2_ECUDA. A bounded wait of the GEMM
 *   that runs out records 0x101 (mamba2_device_error). Asynchronous on
 *   `stream`. */
m2_status mamba2_qlinear(int rows, int in_features, int out_features, int group_size, int bits, const void* x,
                         const uint32_t* wq, const void* scales, const void* biases, void* y, void* stream);

/* The norm that precedes a linear layer in the Nemotron-H blocks, fused into
 * the layer's staging of its input rows (VoiceChat issue, section
 * config.json / text_config: layer_norm_epsilon 1e-5, n_groups 8):
 *   M2_NORM_RMS   (the pre-norm of every block):
 *                   x' = weight * x / sqrt(mean over the row of x^2 + eps)
 *   M2_NORM_GATED (the gated output norm of a Mamba layer, as
 *                   mamba2_gated_norm): v = x * silu(z),
 *                   x' = weight * v / sqrt(mean over each of `groups`
 *                   contiguous blocks of v^2 + eps)
 * computed in fp32 and rounded once to bf16 (what a separate norm kernel
 * would store) before the product. weight: [in_features] fp32, 16-byte
 * aligned. gate: z, bf16, one row per row of x, gate_stride elements apart
 * (a multiple of 8, at least in_features), 16-byte aligned. groups: at most
 * 64, dividing in_features into blocks of a multiple of 32 inputs. */
typedef enum { M2_NORM_NONE = 0, M2_NORM_RMS = 1, M2_NORM_GATED = 2 } m2_norm_kind;
typedef struct {
    m2_norm_kind kind;
    const float* weight;
    float eps;
    int groups;        /* M2_NORM_GATED only */
    const void* gate;  /* M2_NORM_GATED only */
    long gate_stride;  /* M2_NORM_GATED only */
} m2_row_norm;

/* mamba2_qlinear with the Mamba layer's neighbours fused in:
 *   x rows x_stride elements apart (a multiple of 8, at least in_features);
 *   norm (NULL or M2_NORM_NONE: none) applied to each row of x first: the
 *     block's pre-norm before in_proj, the gated output norm before out_proj;
 *   residual (NULL: none): [rows, out_features] bf16 added to the product
 *     before its one rounding, y = residual + x' W^T; may alias y (the
 *     residual stream updated in place).
 * Errors as mamba2_qlinear, and M2_EINVAL / M2_ESHAPE / M2_EALIGN for a bad
 * norm. With x_stride = in_features and no norm or residual the results are
 * mamba2_qlinear's. The GEMM form (40 rows or more) is taken without a norm
 * only: with one, every row count runs as passes of up to 4 rows (the
 * library allocates no buffer for the normalised rows; mamba2_lm_prefill
 * normalises into its workspace and then calls the GEMM). */
m2_status mamba2_qlinear_fused(int rows, int in_features, int out_features, int group_size, int bits,
                               const void* x, long x_stride, const m2_row_norm* norm, const uint32_t* wq,
                               const void* scales, const void* biases, const void* residual, void* y,
                               void* stream);

/* Dense bf16 linear layer for the few rows of a decode step: the attention
 * layers' q|k|v and output projections, which the VoiceChat checkpoints keep
 * in bf16 (VoiceChat issue, section config.json: only the embedding, the
 * heads and the mixer projections are quantized; attention_bias false).
 *     y[r][o] = residual[r][o] + sum_i w[o][i] x'[r][i]
 * with x' the (optionally normalised) row of x, fp32 sums, one rounding.
 * x: [rows, in_features] bf16, rows x_stride elements apart (a multiple of 8,
 *   at least in_features), 16-byte aligned. w: [out_features, in_features]
 *   bf16, 16-byte aligned. y, residual (NULL: none): rows y_stride elements
 *   apart (at least out_features); residual may alias y; y must not alias x.
 * Sizes: in_features a multiple of 32, at most 16384; rows >= 0 (rows == 0 is
 *   a no-op once the arguments check out). Each pass over the weights takes
 *   up to 8 rows of x.
 * Errors: M2_EINVAL, M2_ESHAPE, M2_EALIGN, M2_EUNSUPPORTED, M2_ECUDA. */
m2_status mamba2_linear_bf16(int rows, int in_features, int out_features, const void* x, long x_stride,
                             const m2_row_norm* norm, const void* w, const void* residual, void* y, long y_stride,
                             void* stream);

/* One cached decode position of the hybrid model's grouped-query attention
 * layers, with the KV-cache append: the Nemotron-H attention layers (VoiceChat
 * issue, section config.json / text_config: num_attention_heads 40,
 * num_key_value_heads 8, head_dim 128, attention_bias false, and no
 * positional rotation listed for them), whose KV caches are part of the state
 * a session keeps ("docs/nemotron-voicechat.md", section Online session).
 * For each session s, with lengths[s] = L positions already cached:
 *     k_cache[s][g][L] = k_new[s][g],  v_cache[s][g][L] = v_new[s][g]
 *     a_t   = scale * q[s][h] . k_cache[s][g][t]      for t = 0 .. L
 *     out[s][h] = sum_t softmax(a)_t v_cache[s][g][t]
 * where query head h reads kv head g = h / (n_heads / n_kv_heads). Scores,
 * softmax and sums in fp32 (exp2 of log2-scaled scores), out rounded once to
 * the activation dtype. Only slot L of each cache changes; slots past L are
 * neither read nor written. The caller advances lengths[] between positions
 * (all attention layers of one position share them).
 *
 * q, out [S, n_heads, 128]; k_new, v_new [S, n_kv_heads, 128];
 * k_cache, v_cache [S, n_kv_heads, max_len, 128]; all in `act` (bf16 or fp32),
 * 16-byte aligned; lengths: int32 [S] in DEVICE memory, 4-byte aligned.
 * out must not alias any input.
 * Sizes: head_dim 128; n_heads a multiple of n_kv_heads, at most 8 query heads
 *   per kv head; n_kv_heads and n_sessions at most 65535; max_len >= 1.
 *   n_sessions == 0 is a no-op once the arguments check out.
 * Scratch: workspace of at least mamba2_attn_decode_workspace_bytes(...).
 *   bf16 caches need none (workspace may be NULL with workspace_bytes 0):
 *   one kernel, whose CTAs each take a run of 64-position chunks of one
 *   (session, kv head) and, as one thread-block cluster per (session, kv
 *   head), merge their partial results in shared memory. The products
 *   (scores, and the softmax weights split into two bf16 terms times the
 *   values) run on the tensor cores with fp32 accumulation. fp32 caches (and
 *   bf16 caches of 2^31 rows or more) take two kernels: partial results per
 *   chunk of up to 64 positions (shorter where few sessions and kv heads
 *   would leave the GPU idle) in the workspace, then their merge.
 * Errors: M2_EINVAL (NULL pointer, non-positive size, non-finite scale),
 *   M2_ESHAPE, M2_EALIGN, M2_EWORKSPACE, M2_EUNSUPPORTED, M2_ECUDA. A length
 *   outside [0, max_len) is seen only on the device: that session's out is
 *   zero, its caches are untouched, and the device error word reads 0x104
 *   (mamba2_device_error). Asynchronous on `stream`. */
m2_status mamba2_attn_decode(int n_sessions, int n_heads, int n_kv_heads, int head_dim, int max_len, m2_dtype act,
                             const int32_t* lengths, const void* q, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, float scale, void* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Bytes of device scratch that mamba2_attn_decode needs (0 if the sizes are
 * invalid, n_sessions is 0, or the caches are bf16 of fewer than 2^31 rows,
 * n_sessions x n_kv_heads x max_len). */
size_t mamba2_attn_decode_workspace_bytes(int n_sessions, int n_heads, int n_kv_heads, int head_dim, int max_len,
                                          m2_dtype act);

/* Bytes of device scratch that mamba2_step needs for n_sessions sessions. */
size_t mamba2_step_workspace_bytes(const m2_dims* d, int n_sessions);

/* One cached frame for n_sessions independent sessions that share one
 * layer's weights (the per-position update of the "Mamba2 state" that the
 * VoiceChat online session keeps, "docs/nemotron-voicechat.md", section
 * Online session).
 *
 * Inputs : this frame's x [S,H,P], B, C [S,G,N], dt_raw [S,H] (act dtype);
 *          the layer's A_log, D, dt_bias, conv_w, conv_b.
 * In/out : ssm_state [S,H,P,N] fp32 and conv_state [S,K-1,CH] (act dtype)
 *          are read and updated in place.
 * Output : y [S,H,P] (act dtype). y must not alias any input.
 * Scratch: workspace of at least mamba2_step_workspace_bytes(d, S).
 * d->batch and d->T are ignored. */
m2_status mamba2_step(const m2_dims* d, int n_sessions, const void* x, const void* B,
                      const void* C, const void* dt_raw, const float* A_log, const float* D,
                      const float* dt_bias, const float* conv_w, const float* conv_b,
                      float* ssm_state, void* conv_state, void* y, void* workspace,
                      size_t workspace_bytes, void* stream);

/* mamba2_step on inputs that are column slices of wider rows, one row per
 * session: session s's x, B, C and dt_raw start in_row_stride * s elements
 * past the x, B, C and dt_raw pointers (for instance the rows of the Mamba
 * layer's input projection output z | x | B | C | dt, see
 * mamba2_conv_scan_strided). in_row_stride > 0 (M2_EINVAL) and in_row_stride
 * times the element size a multiple of 16 bytes (M2_EALIGN); everything else
 * is mamba2_step's. */
m2_status mamba2_step_strided(const m2_dims* d, int n_sessions, const void* x, const void* B, const void* C,
                              const void* dt_raw, long in_row_stride, const float* A_log, const float* D,
                              const float* dt_bias, const float* conv_w, const float* conv_b, float* ssm_state,
                              void* conv_state, void* y, void* workspace, size_t workspace_bytes, void* stream);

/* mamba2_step without a caller-provided workspace, for callers that cannot
 * allocate device memory: a real-time frame loop that must not call
 * cudaMalloc (it can synchronise the device mid-frame), a host that hands the
 * library only tensors it already owns, or a binding without a device
 * allocator. (This entry point has no counterpart in the VoiceChat pages; it
 * is a property of this library.)
 *
 * The scratch is a fixed array inside the library's device image,
 * mamba2_step_noalloc_max_bytes() bytes (1 MiB), present on every GPU that
 * loads the library until the process exits. A request whose
 * mamba2_step_workspace_bytes(d, n_sessions) exceeds it returns
 * M2_EWORKSPACE before anything runs (at the Nemotron-H shape that is more
 * than 21 sessions per call). The first call on a device looks up the
 * array's device address (with that device current); make that first call
 * before any stream capture. All calls share the one array: calls that may
 * overlap on the GPU (on different streams, or from different host threads
 * without ordering) race on it and give undefined results; calls ordered on
 * one stream are safe. Nothing in it needs clearing between calls. Arguments,
 * results and every other error are those of mamba2_step, checked in the
 * same order before the size (a NULL pointer is M2_EINVAL, another GPU
 * M2_EUNSUPPORTED). */
m2_status mamba2_step_noalloc(const m2_dims* d, int n_sessions, const void* x, const void* B,
                              const void* C, const void* dt_raw, const float* A_log, const float* D,
                              const float* dt_bias, const float* conv_w, const float* conv_b,
                              float* ssm_state, void* conv_state, void* y, void* stream);

/* Size in bytes of the fixed scratch used by mamba2_step_noalloc. */
size_t mamba2_step_noalloc_max_bytes(void);

/* ------------------------------------------------------------------------
 * One cached position of the hybrid language model, and its full-history
 * recompute. The Nemotron-H model of VoiceChat interleaves Mamba ('M') and
 * attention ('*') blocks (VoiceChat issue, section config.json /
 * text_config: hybrid_override_pattern; its 27 'M' and 4 '*' layers; the 25
 * MLP ('-') layers are not part of this library); the session keeps each
 * Mamba layer's SSM state and conv tail and each attention layer's KV caches
 * across positions ("docs/nemotron-voicechat.md", section Online session),
 * and stepping positions from these caches gives the tokens a full-history
 * recompute gives (same doc, section Offline timeline).
 *
 * Per block, on the residual stream h (bf16):
 *   'M': proj = in_proj(RMSNorm(h))         z | x | B | C | dt per row
 *        y    = mixer core (mamba2_step / mamba2_conv_scan) on x, B, C, dt
 *        h    = h + out_proj(gated_norm(y, z))
 *   '*': qkv  = [Wq; Wk; Wv] RMSNorm(h)      bf16 projections, no bias
 *        o    = attention (mamba2_attn_decode) with the KV-cache append
 *        h    = h + Wo o
 * in_proj and out_proj are 4-bit group-64 (mamba2_qlinear layout); the norms
 * and the residual adds are fused into the projections (m2_row_norm). Every
 * activation stored between kernels is bf16, each computed in fp32 and
 * rounded once. The final norm and the heads are not part of this call. */
typedef struct {
    const float* norm_w;          /* [hidden] fp32: the block's pre-norm */
    /* 'M' blocks */
    const uint32_t* in_wq;        /* in_proj [2*H*P + 2*G*N + H, hidden], 4-bit */
    const void* in_scales;        /* [.., hidden/64] bf16 */
    const void* in_biases;
    const float *A_log, *D, *dt_bias, *conv_w, *conv_b;  /* the mixer core's, as mamba2_step */
    const float* gnorm_w;         /* [H*P] fp32: the gated output norm */
    const uint32_t* out_wq;       /* out_proj [hidden, H*P], 4-bit */
    const void* out_scales;
    const void* out_biases;
    float* ssm_state;             /* [S,H,P,N] fp32, updated in place */
    void* conv_state;             /* [S,K-1,CH] bf16, updated in place */
    /* '*' blocks */
    const void* wqkv;             /* [(n_heads + 2 n_kv_heads) * head_dim, hidden] bf16 */
    const void* wo;               /* [hidden, n_heads * head_dim] bf16 */
    void* k_cache;                /* [S, n_kv_heads, max_len, head_dim] bf16, updated at the new slots */
    void* v_cache;
} m2_lm_layer;

typedef struct {
    int n_layers;
    const char* kinds;            /* n_layers characters, 'M' or '*' */
    const m2_lm_layer* layers;    /* host array of n_layers */
    int hidden;                   /* residual width (4480 in Nemotron-H) */
    m2_dims mixer;                /* the mixer core's dims (batch, T ignored; act M2_BF16) */
    int n_heads, n_kv_heads, head_dim, max_len;  /* attention blocks (40, 8, 128) */
    float norm_eps;               /* all norms (1e-5) */
    float attn_scale;             /* softmax scale (1/sqrt(head_dim)) */
} m2_lm;

/* Bytes of device scratch mamba2_lm_prefill needs for S sessions of T
 * positions with this chunk length (mamba2_lm_step: T = 1, chunk ignored);
 * 0 if the model description is invalid. */
size_t mamba2_lm_workspace_bytes(const m2_lm* m, int n_sessions, int T, int chunk);

/* One cached position for S sessions: hidden [S, hidden] bf16 holds the
 * position's input (the fused embedding) and receives the residual stream
 * after the last block. lengths [S] int32 in device memory: positions
 * already in the KV caches (read on the device; the caller advances them
 * by one after the call). Every Mamba block runs mamba2_step on its rows of
 * the in_proj output (strided), every attention block mamba2_attn_decode.
 * All host arrays (m, m->kinds, m->layers) are read during the call only.
 * Errors: those of the calls it makes, checked for every block before the
 * first launch (M2_EINVAL for a NULL pointer or an unknown kind, M2_ESHAPE
 * for sizes the kernels do not take, M2_EALIGN, M2_EWORKSPACE). */
m2_status mamba2_lm_step(const m2_lm* m, int n_sessions, void* hidden, const int32_t* lengths, void* workspace,
                         size_t workspace_bytes, void* stream);

/* T positions for S sessions at once, continuing from the caches (the
 * full-history recompute when the caches start empty): hidden [S, T, hidden]
 * bf16 in/out as mamba2_lm_step per position; the Mamba blocks run the
 * chunked scan (mamba2_conv_scan_strided, `chunk`) over the T positions, the
 * attention blocks the T positions in order (position t of session s at
 * slot lengths[s] + t). Afterwards the caches are those after the last
 * position; the caller advances lengths by T. Errors as mamba2_lm_step. */
m2_status mamba2_lm_prefill(const m2_lm* m, int n_sessions, int T, void* hidden, const int32_t* lengths, int chunk,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Static description of a status code. */
const char* mamba2_status_string(m2_status s);

/* cudaError_t of the most recent M2_ECUDA returned on the calling thread. */
int mamba2_last_cuda_error(void);

/* Reads and clears the device-side error word of the current device
 * (0 = no error; otherwise the code of a bounded wait that ran out).
 * Synchronises `stream`. Returns M2_ECUDA if the read itself fails. */
m2_status mamba2_device_error(void* stream, unsigned int* code);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA2_H */
