// Dense bf16 linear layer for the few rows of a cached decode step: the
// attention layers' projections of the hybrid model, which the VoiceChat
// checkpoints keep in bf16 (VoiceChat issue, section config.json: only the
// embedding, the heads and the Mamba mixer projections are quantized;
// attention_bias false). y[r][o] = sum_i W[o][i] x[r][i] (+ residual[r][o]),
// fp32 sums, one rounding to bf16.
//
// At a handful of rows the layer streams its weights: 2 bytes per weight
// against 2 flops per row. One persistent CTA per SM stages the rows of x
// (optionally normalised, m2_rowprep.cuh) in shared memory as bf16; each warp
// streams whole weight rows with 16-byte loads (a lane takes 8 inputs at a
// time, consecutive lanes consecutive 16-byte pieces, the next batch in
// flight while the current one is computed, the two batches in two register
// sets taken in turn), multiplies with mixed-precision
// fmas (bf16 x bf16 products, exact in fp32) and reduces across the warp.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_rowprep.cuh"

namespace m2 {

namespace {

constexpr int kLinThreads = 512;
constexpr int kLinWarps = kLinThreads / 32;
constexpr int kPiece = 8;      // inputs per 16-byte weight load
constexpr int kInFlight = 6;   // weight pieces per lane and batch (1536 inputs per warp and batch)
constexpr int kLinSmemCap = 160 * 1024;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// acc + w_lo x_lo + w_hi x_hi for the bf16 pairs w and x: exact products, one
// rounding per fma
__device__ __forceinline__ float pair_fma(uint32_t w, uint32_t x, float acc) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %1;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x));
    return acc;
}

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
    acc = pair_fma(w.x, x.x, acc);
    acc = pair_fma(w.y, x.y, acc);
    acc = pair_fma(w.z, x.z, acc);
    return pair_fma(w.w, x.w, acc);
}

__device__ __forceinline__ void load_batch(const LinearArgs& a, int o, int bi, int npieces, int lane,
                                           uint4 (&w)[kInFlight]) {
    const uint4* wrow = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.w) + (size_t)o * a.in);
#pragma unroll
    for (int k = 0; k < kInFlight; ++k) {
        const int c = bi * kInFlight * 32 + lane + k * 32;
        if (c < npieces) w[k] = ld_stream(wrow + c);
    }
}

// NB rows of x per pass over the weights.
template <int NB, int KIND, bool RES>
__global__ void __launch_bounds__(kLinThreads, 1) linear_bf16_kernel(LinearArgs a) {
    extern __shared__ float4 lin_smem4[];
    const int in = a.in, npieces = in / kPiece, nchunks = in / rowprep::kChunk;
    uint4* sx = reinterpret_cast<uint4*>(lin_smem4);                        // [NB][npieces] bf16 x8
    float* scratch = reinterpret_cast<float*>(sx + (size_t)NB * npieces);   // [NB][nchunks]
    float* srs = scratch + (size_t)NB * nchunks;                            // [NB][norm groups]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gwarp = blockIdx.x * kLinWarps + warp, nwarps = gridDim.x * kLinWarps;
    uint16_t* yb = reinterpret_cast<uint16_t*>(a.y);
    const uint16_t* rb = reinterpret_cast<const uint16_t*>(a.residual);

    pdl_wait();  // x (and the residual) may come from the previous kernel
    for (int r0 = 0; r0 < a.rows; r0 += NB) {
        const int nr = min(NB, a.rows - r0);
        if (KIND != 0)
            rowprep::norm_scales<kLinThreads, KIND>(a.x, a.x_stride, a.norm, in, r0, nr, NB, scratch, srs);
        for (int e = tid; e < NB * nchunks; e += kLinThreads) {
            const int r = e / nchunks, c = e % nchunks;
            uint32_t wd[16];
            rowprep::staged32<KIND>(a.x, a.x_stride, a.norm, in, r0, r, nr, c * rowprep::kChunk, srs, wd);
            uint4* dst = sx + (size_t)r * npieces + c * (rowprep::kChunk / kPiece);
#pragma unroll
            for (int v = 0; v < rowprep::kChunk / kPiece; ++v)
                dst[v] = make_uint4(wd[4 * v], wd[4 * v + 1], wd[4 * v + 2], wd[4 * v + 3]);
        }
        __syncthreads();

        const int nbatch = (npieces + kInFlight * 32 - 1) / (kInFlight * 32);
        int o = gwarp, bi = 0;
        float acc[NB];
#pragma unroll
        for (int r = 0; r < NB; ++r) acc[r] = 0.f;
        // one item: the batch in w of row o; finishes the row at its last batch
        auto compute = [&](const uint4 (&w)[kInFlight], int o, int bi) {
#pragma unroll
            for (int k = 0; k < kInFlight; ++k) {
                const int c = bi * kInFlight * 32 + lane + k * 32;
                if (c < npieces) {
#pragma unroll
                    for (int r = 0; r < NB; ++r) acc[r] = dot8(w[k], sx[(size_t)r * npieces + c], acc[r]);
                }
            }
            if (bi == nbatch - 1) {
#pragma unroll
                for (int r = 0; r < NB; ++r) {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
                }
                if (lane == 0) {
#pragma unroll
                    for (int r = 0; r < NB; ++r) {
                        if (r < nr) {
                            const size_t i = (size_t)(r0 + r) * a.y_stride + o;
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
        if (o < a.out) load_batch(a, o, bi, npieces, lane, wa);
        while (o < a.out) {
            int on = o, bn = bi;
            advance(on, bn);
            if (on < a.out) load_batch(a, on, bn, npieces, lane, wb);
            compute(wa, o, bi);
            o = on;
            bi = bn;
            if (o >= a.out) break;
            on = o;
            bn = bi;
            advance(on, bn);
            if (on < a.out) load_batch(a, on, bn, npieces, lane, wa);
            compute(wb, o, bi);
            o = on;
            bi = bn;
        }
        __syncthreads();  // x of this pass is consumed before the next is staged
    }
    pdl_trigger();
}

size_t lin_smem_bytes(int nb, int in) {
    return (size_t)nb * in * 2 + ((size_t)nb * (in / rowprep::kChunk) + (size_t)nb * kMaxNormGroups) * 4;
}

template <int NB, int KIND, bool RES>
cudaError_t launch_variant(const LinearArgs& a, cudaStream_t st) {
    const size_t smem = lin_smem_bytes(NB, a.in);
    static int configured_device = -1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(linear_bf16_kernel<NB, KIND, RES>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLinSmemCap);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const long want = ((long)a.out + kLinWarps - 1) / kLinWarps;
    const int blocks = (int)(want < sms ? want : (long)sms);
    return launch_pdl(linear_bf16_kernel<NB, KIND, RES>, dim3(blocks), dim3(kLinThreads), smem, st, a);
}

// The kernel variant for this norm kind and residual.
template <int NB>
cudaError_t launch_nb(const LinearArgs& a, cudaStream_t st) {
    const bool res = a.residual != nullptr;
    switch (a.norm.kind) {
        case 0: return res ? launch_variant<NB, 0, true>(a, st) : launch_variant<NB, 0, false>(a, st);
        case 1: return res ? launch_variant<NB, 1, true>(a, st) : launch_variant<NB, 1, false>(a, st);
        case 2: return res ? launch_variant<NB, 2, true>(a, st) : launch_variant<NB, 2, false>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_linear_bf16(const LinearArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    int nb = 8;
    while (nb > 1 && lin_smem_bytes(nb, a.in) > (size_t)kLinSmemCap) nb /= 2;
    while (nb > 1 && nb / 2 >= a.rows) nb /= 2;  // no wider pass than the rows there are
    switch (nb) {
        case 8: return launch_nb<8>(a, st);
        case 4: return launch_nb<4>(a, st);
        case 2: return launch_nb<2>(a, st);
        case 1: return launch_nb<1>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m2
