// 4-bit affine group-quantized linear layer: the Mamba layer's input and
// output projections as the VoiceChat 4-bit checkpoint stores them
// (group_size 64, bits 4). Weight (o, i) is the 4-bit field q at bits
// 4*(i%8) of the 32-bit word wq[o][i/8], dequantized per group of 64 inputs
// as scale * q + bias (scale, bias bf16 [out, in/64]); y[r][o] = sum_i W[o][i] x[r][i].
//
// At the batch sizes of a cached decode step (a few sessions) the layer is a
// stream of the packed weights: 0.5 byte per weight against a few flops. One
// persistent CTA per SM stages up to four rows of x in shared memory, as bf16
// pairs laid out like the weight pairs below, together with the fp32 sum of
// x over every 32-input chunk; each warp then streams whole weight rows with
// coalesced 16-byte loads (a lane takes one 32-input chunk at a time; the
// next batch of chunks is loaded while the current one is computed) and
// reduces across the warp. Per 32-bit word the four bf16 pairs (128 + q) are
// built with one mask and one OR each (bf16 0x4300 is 128 and q fills the low
// mantissa bits) and go straight into mixed-precision fmas (bf16 x bf16
// products, exact in fp32, added to an fp32 accumulator), so
//     sum_i (scale q_i + bias) x_i
//   = scale * sum_i (128 + q_i) x_i + (bias - 128 scale) * sum_i x_i
// costs about one integer operation and one fma per weight and row of x,
// plus one correction per chunk.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_rowprep.cuh"

namespace m2 {

namespace {

constexpr int kQlThreads = 512;
constexpr int kQlWarps = kQlThreads / 32;
constexpr int kChunk = 32;     // inputs per 16-byte weight load
constexpr int kInFlight = 5;   // weight chunks per lane and batch (a 4480-wide row in one batch)
constexpr int kGroup = 64;
// x of one 32-input chunk in shared memory: 16 words of bf16 pairs, padded
// to 20: the lanes of a warp read consecutive chunks, and an 80-byte stride
// spreads their 16-byte reads over all banks
constexpr int kChunkPitch = 20;

// 16-byte load of streamed data (read once: not kept in L1).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// acc + (128 + q_lo) x_lo + (128 + q_hi) x_hi for the bf16 pairs p (weights)
// and xp (inputs): exact products, one rounding per fma
__device__ __forceinline__ float pair_fma(uint32_t p, uint32_t xp, float acc) {
    asm("{\n\t.reg .b16 pl, ph, xl, xh;\n\t"
        "mov.b32 {pl, ph}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, pl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ph, xh, %0;\n\t}"
        : "+f"(acc)
        : "r"(p), "r"(xp));
    return acc;
}

// (v & 0x000F000F) | hi, one three-input logic operation: hi (the bf16 pair
// 0x4300 0x4300) is passed in a register so that the mask can be the one
// immediate operand
__device__ __forceinline__ uint32_t nib_pair(uint32_t v, uint32_t hi) {
    uint32_t r;
    asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(r) : "r"(v), "r"(hi));
    return r;
}

// sum over the 8 inputs of one word of (128 + q) * x; xw holds the word's x
// as the pairs (x_k, x_{k+4}), k = 0..3, matching the weight pairs
__device__ __forceinline__ float word_dot(uint32_t w, const uint4& xw, uint32_t hi, float acc) {
    acc = pair_fma(nib_pair(w, hi), xw.x, acc);
    acc = pair_fma(nib_pair(w >> 4, hi), xw.y, acc);
    acc = pair_fma(nib_pair(w >> 8, hi), xw.z, acc);
    acc = pair_fma(nib_pair(w >> 12, hi), xw.w, acc);
    return acc;
}

// The weight chunks (16-byte loads) and packed (scale, bias) of batch `bi`
// of row `o` for this lane: chunks bi*kInFlight*32 + lane + 32k.
__device__ __forceinline__ void load_batch(const QLinearArgs& a, int o, int bi, int nchunks, int ngroups, int lane,
                                           uint4 (&w)[kInFlight], uint32_t (&sb)[kInFlight]) {
    const uint4* wrow = reinterpret_cast<const uint4*>(a.wq + (size_t)o * (uint32_t)(a.in / 8));
    const uint16_t* srow = a.scales + (size_t)o * ngroups;
    const uint16_t* brow = a.biases + (size_t)o * ngroups;
#pragma unroll
    for (int k = 0; k < kInFlight; ++k) {
        const int c = bi * kInFlight * 32 + lane + k * 32;
        if (c < nchunks) {
            w[k] = ld_stream(wrow + c);
            sb[k] = (uint32_t)__ldg(srow + c / 2) | ((uint32_t)__ldg(brow + c / 2) << 16);
        }
    }
}

// NB rows of x per pass over the weights.
template <int NB, int KIND, bool RES>
__global__ void __launch_bounds__(kQlThreads, 1) qlinear_kernel(QLinearArgs a) {
    extern __shared__ float4 ql_smem4[];
    const int in = a.in, nchunks = in / kChunk, ngroups = in / kGroup;
    uint32_t* sx = reinterpret_cast<uint32_t*>(ql_smem4);                        // [NB][nchunks][kChunkPitch]
    float* ssum = reinterpret_cast<float*>(sx + (size_t)NB * nchunks * kChunkPitch);  // [NB][nchunks]
    float* srs = ssum + (size_t)NB * nchunks;                                    // [NB][norm groups]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gwarp = blockIdx.x * kQlWarps + warp, nwarps = gridDim.x * kQlWarps;
    uint16_t* yb = reinterpret_cast<uint16_t*>(a.y);
    const uint16_t* rb = reinterpret_cast<const uint16_t*>(a.residual);
    // the bf16 pair (128, 128), kept in a register (not folded into an immediate)
    uint32_t hi;
    asm volatile("mov.b32 %0, 0x43004300;" : "=r"(hi));

    pdl_wait();  // x (and z, the residual) may come from the previous kernel
    for (int r0 = 0; r0 < a.rows; r0 += NB) {
        const int nr = min(NB, a.rows - r0);
        // the norm's scales of this pass's rows (ssum serves as scratch)
        if (KIND != 0) rowprep::norm_scales<kQlThreads, KIND>(a.x, a.x_stride, a.norm, in, r0, nr, NB, ssum, srs);
        // stage x as the bf16 pairs of each word, (x_k, x_{k+4}), and the fp32
        // sum of x over each chunk
        for (int e = tid; e < NB * nchunks; e += kQlThreads) {
            const int r = e / nchunks, c = e % nchunks;
            uint32_t wd[16];
            rowprep::staged32<KIND>(a.x, a.x_stride, a.norm, in, r0, r, nr, c * kChunk, srs, wd);
            float s = 0.f;
            uint4* dst = reinterpret_cast<uint4*>(sx + ((size_t)r * nchunks + c) * kChunkPitch);
#pragma unroll
            for (int v = 0; v < kChunk / 8; ++v) {
                // word v holds x_0..x_7 as (x0 x1) (x2 x3) (x4 x5) (x6 x7)
                const uint4 u = make_uint4(wd[4 * v], wd[4 * v + 1], wd[4 * v + 2], wd[4 * v + 3]);
                dst[v] = make_uint4(__byte_perm(u.x, u.z, 0x5410), __byte_perm(u.x, u.z, 0x7632),
                                    __byte_perm(u.y, u.w, 0x5410), __byte_perm(u.y, u.w, 0x7632));
                const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) s += bf16_bits_to_float(uw[k] & 0xFFFFu) + bf16_bits_to_float(uw[k] >> 16);
            }
            ssum[r * nchunks + c] = s;
        }
        __syncthreads();

        // Each warp walks (row, batch) items: a batch is up to kInFlight chunks
        // per lane of one weight row. The next item's loads are issued before
        // the current item is computed, so a batch is always in flight.
        const int nbatch = (nchunks + kInFlight * 32 - 1) / (kInFlight * 32);
        int o = gwarp, bi = 0;
        float acc[NB];
#pragma unroll
        for (int r = 0; r < NB; ++r) acc[r] = 0.f;
        // one item: the batch in (w, sb) of row o; finishes the row at its last batch
        auto compute = [&](const uint4 (&w)[kInFlight], const uint32_t (&sb)[kInFlight], int o, int bi) {
#pragma unroll
            for (int k = 0; k < kInFlight; ++k) {
                const int c = bi * kInFlight * 32 + lane + k * 32;
                if (c < nchunks) {
                    const float scale = bf16_bits_to_float(sb[k] & 0xFFFFu);
                    const float corr = bf16_bits_to_float(sb[k] >> 16) - 128.f * scale;
#pragma unroll
                    for (int r = 0; r < NB; ++r) {
                        const uint4* xr = reinterpret_cast<const uint4*>(sx + ((size_t)r * nchunks + c) * kChunkPitch);
                        float d0 = word_dot(w[k].x, xr[0], hi, 0.f);
                        float d1 = word_dot(w[k].y, xr[1], hi, 0.f);
                        d0 = word_dot(w[k].z, xr[2], hi, d0);
                        d1 = word_dot(w[k].w, xr[3], hi, d1);
                        acc[r] = fmaf(scale, d0 + d1, fmaf(corr, ssum[r * nchunks + c], acc[r]));
                    }
                }
            }
            if (bi == nbatch - 1) {
                // the row is complete: reduce across the warp and store
#pragma unroll
                for (int r = 0; r < NB; ++r) {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
                }
                if (lane == 0) {
#pragma unroll
                    for (int r = 0; r < NB; ++r) {
                        if (r < nr) {
                            const size_t i = (size_t)(r0 + r) * a.out + o;
                            const float res = RES ? bf16_bits_to_float(rb[i]) : 0.f;
                            yb[i] = float_to_bf16_bits(acc[r] + res);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < NB; ++r) acc[r] = 0.f;
            }
        };
        auto advance = [&](int& o, int& bi) {
            if (++bi == nbatch) {
                bi = 0;
                o += nwarps;
            }
        };
        // two register sets in turn: the next item's loads go into one while
        // the other is computed (no copies between them)
        uint4 wa[kInFlight], wb[kInFlight];
        uint32_t sa[kInFlight], sbb[kInFlight];
        if (o < a.out) load_batch(a, o, bi, nchunks, ngroups, lane, wa, sa);
        while (o < a.out) {
            int on = o, bn = bi;
            advance(on, bn);
            if (on < a.out) load_batch(a, on, bn, nchunks, ngroups, lane, wb, sbb);
            compute(wa, sa, o, bi);
            o = on;
            bi = bn;
            if (o >= a.out) break;
            on = o;
            bn = bi;
            advance(on, bn);
            if (on < a.out) load_batch(a, on, bn, nchunks, ngroups, lane, wa, sa);
            compute(wb, sbb, o, bi);
            o = on;
            bi = bn;
        }
        __syncthreads();  // x of this pass is consumed before the next is staged
    }
    pdl_trigger();
}

constexpr int kQlSmemCap = 128 * 1024;  // shared memory of one pass: x as fp32 and its chunk sums

size_t smem_bytes(int nb, int in) {
    return ((size_t)nb * (in / kChunk) * (kChunkPitch + 1) + (size_t)nb * kMaxNormGroups) * sizeof(uint32_t);
}

template <int NB, int KIND, bool RES>
cudaError_t launch_variant(const QLinearArgs& a, cudaStream_t st) {
    const size_t smem = smem_bytes(NB, a.in);
    static int configured_device = -1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(qlinear_kernel<NB, KIND, RES>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQlSmemCap);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const long want = ((long)a.out + kQlWarps - 1) / kQlWarps;
    const int blocks = (int)(want < sms ? want : (long)sms);
    return launch_pdl(qlinear_kernel<NB, KIND, RES>, dim3(blocks), dim3(kQlThreads), smem, st, a);
}

// The kernel variant for this norm kind and residual.
template <int NB>
cudaError_t launch_nb(const QLinearArgs& a, cudaStream_t st) {
    const bool res = a.residual != nullptr;
    switch (a.norm.kind) {
        case 0: return res ? launch_variant<NB, 0, true>(a, st) : launch_variant<NB, 0, false>(a, st);
        case 1: return res ? launch_variant<NB, 1, true>(a, st) : launch_variant<NB, 1, false>(a, st);
        case 2: return res ? launch_variant<NB, 2, true>(a, st) : launch_variant<NB, 2, false>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

// One row of x normalised as the fused layers stage it (the same code, so the
// same bf16 bits), written out: the input of the GEMM for many rows.
template <int KIND>
__global__ void __launch_bounds__(256) row_norm_kernel(RowNorm nm, const void* x, long x_stride, int in, void* out) {
    __shared__ float scratch[kQlMaxIn / rowprep::kChunk];
    __shared__ float srs[kMaxNormGroups];
    const int r = blockIdx.x;
    pdl_wait();  // x (and the gate) may come from the previous kernel
    pdl_trigger();
    rowprep::norm_scales<256, KIND>(x, x_stride, nm, in, r, 1, 1, scratch, srs);
    for (int c = threadIdx.x; c < in / rowprep::kChunk; c += 256) {
        uint32_t wd[16];
        rowprep::staged32<KIND>(x, x_stride, nm, in, r, 0, 1, c * rowprep::kChunk, srs, wd);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + (size_t)r * in + c * rowprep::kChunk);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(wd[4 * k], wd[4 * k + 1], wd[4 * k + 2], wd[4 * k + 3]);
    }
}

}  // namespace

cudaError_t launch_row_norm(const RowNorm& nm, const void* x, long x_stride, int rows, int in, void* out,
                            cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (in > kQlMaxIn || in % rowprep::kChunk != 0) return cudaErrorInvalidValue;
    switch (nm.kind) {
        case 1: return launch_pdl(row_norm_kernel<1>, dim3(rows), dim3(256), 0, st, nm, x, x_stride, in, out);
        case 2: return launch_pdl(row_norm_kernel<2>, dim3(rows), dim3(256), 0, st, nm, x, x_stride, in, out);
        default: return cudaErrorInvalidValue;
    }
}

int qlinear_rows_per_pass(int in) {
    // x of a pass, as fp32, within the shared-memory cap
    for (int nb : {4, 2, 1})
        if (smem_bytes(nb, in) <= (size_t)kQlSmemCap) return nb;
    return 0;
}

cudaError_t launch_qlinear(const QLinearArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    // many rows (a prefill): the tensor-core GEMM, which reads each weight
    // once per 128 rows instead of once per pass of up to four
    if (a.norm.kind == 0 && a.rows >= kQgemmMinRows) return launch_qgemm(a, st);
    int nb = qlinear_rows_per_pass(a.in);
    while (nb > 1 && nb / 2 >= a.rows) nb /= 2;  // no wider pass than the rows there are
    switch (nb) {
        case 4: return launch_nb<4>(a, st);
        case 2: return launch_nb<2>(a, st);
        case 1: return launch_nb<1>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m2
