// Staging of the input rows of the decode-step linear layers (the 4-bit
// projections and the dense bf16 ones) in shared memory, with the norm that
// precedes each of them in the Nemotron-H blocks fused in:
//   kind 1 (the pre-norm of every block): x * w / sqrt(mean(x^2) + eps);
//   kind 2 (the gated output norm of a Mamba layer): v = x * silu(z), then
//     v * w / sqrt(mean over each of `groups` blocks of v^2 + eps).
// (Hybrid-model configuration in the VoiceChat issue, section config.json /
// text_config: layer_norm_epsilon 1e-5, n_groups 8.) The normalised value is
// rounded to bf16, as a separate norm kernel would store it, and staged.
//
// Every CTA of a persistent linear kernel stages the same rows: the norm's
// sums are recomputed per CTA (a row is at most a few tens of KB from L2),
// which costs less than a launch and a round trip through memory. The sums
// are taken in a fixed order (per 32-input chunk, then chunk after chunk), so
// the result does not depend on the thread schedule.
#pragma once

#include "m2_common.cuh"
#include "m2_launch.h"

namespace m2 {
namespace rowprep {

constexpr int kChunk = 32;  // inputs per staging unit

// The 32 values of inputs [i0, i0+32) of row `row` before the norm's scaling:
// x, or x * silu(z) for the gated norm.
template <int KIND>
__device__ __forceinline__ void load32(const void* x, long x_stride, const RowNorm& nm, int row, int i0,
                                       float (&v)[kChunk]) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(x) + (size_t)row * x_stride + i0);
    uint4 u[4], zu[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __ldg(src + k);
    if (KIND == 2) {
        const uint4* zs = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(nm.gate) +
                                                         (size_t)row * nm.gate_stride + i0);
#pragma unroll
        for (int k = 0; k < 4; ++k) zu[k] = __ldg(zs + k);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * k + 2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
            v[8 * k + 2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
        }
    }
    if (KIND == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t w[4] = {zu[k].x, zu[k].y, zu[k].z, zu[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * k + 2 * j] *= silu_fast(bf16_bits_to_float(w[j] & 0xFFFFu));
                v[8 * k + 2 * j + 1] *= silu_fast(bf16_bits_to_float(w[j] >> 16));
            }
        }
    }
}

// KIND is RowNorm::kind, fixed at compile time.
//
// Phase 1 of a normalised staging: srs[r * groups + g] = 1 / sqrt(mean of the
// squares over block g of row r0 + r + eps) for the nr rows of this pass.
// `scratch` holds nb * (in / 32) floats. Ends with a block barrier.
template <int NTHREADS, int KIND>
__device__ void norm_scales(const void* x, long x_stride, const RowNorm& nm, int in, int r0, int nr, int nb,
                            float* scratch, float* srs) {
    const int nchunks = in / kChunk, tid = threadIdx.x;
    for (int e = tid; e < nb * nchunks; e += NTHREADS) {
        const int r = e / nchunks, c = e % nchunks;
        float sq = 0.f;
        if (r < nr) {
            float v[kChunk];
            load32<KIND>(x, x_stride, nm, r0 + r, c * kChunk, v);
#pragma unroll
            for (int k = 0; k < kChunk; ++k) sq = fmaf(v[k], v[k], sq);
        }
        scratch[e] = sq;
    }
    __syncthreads();
    const int groups = KIND == 2 ? nm.groups : 1;
    const int cpg = nchunks / groups;
    for (int k = tid; k < nb * groups; k += NTHREADS) {
        const int r = k / groups, g = k % groups;
        float t = 0.f;
        for (int c = g * cpg; c < (g + 1) * cpg; ++c) t += scratch[r * nchunks + c];
        srs[k] = rsqrtf(t / (float)(cpg * kChunk) + nm.eps);
    }
    __syncthreads();
}

// The staged bf16 bits of inputs [i0, i0+32) of row r (of this pass), as 16
// words of natural pairs (x_{2j}, x_{2j+1}); zeros past the last row.
template <int KIND>
__device__ __forceinline__ void staged32(const void* x, long x_stride, const RowNorm& nm, int in, int r0, int r,
                                         int nr, int i0, const float* srs, uint32_t (&wd)[16]) {
    if (r >= nr) {
#pragma unroll
        for (int k = 0; k < 16; ++k) wd[k] = 0u;
        return;
    }
    if (KIND == 0) {
        const uint4* src =
            reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(x) + (size_t)(r0 + r) * x_stride + i0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 u = __ldg(src + k);
            wd[4 * k] = u.x;
            wd[4 * k + 1] = u.y;
            wd[4 * k + 2] = u.z;
            wd[4 * k + 3] = u.w;
        }
        return;
    }
    float v[kChunk];
    load32<KIND>(x, x_stride, nm, r0 + r, i0, v);
    const int groups = KIND == 2 ? nm.groups : 1;
    const float sc = srs[r * groups + i0 / (in / groups)];
    const float4* w4 = reinterpret_cast<const float4*>(nm.weight + i0);
#pragma unroll
    for (int k = 0; k < kChunk / 4; ++k) {
        const float4 w = __ldg(w4 + k);
        const uint32_t lo = (uint32_t)float_to_bf16_bits(v[4 * k] * sc * w.x) |
                            ((uint32_t)float_to_bf16_bits(v[4 * k + 1] * sc * w.y) << 16);
        const uint32_t hi = (uint32_t)float_to_bf16_bits(v[4 * k + 2] * sc * w.z) |
                            ((uint32_t)float_to_bf16_bits(v[4 * k + 3] * sc * w.w) << 16);
        wd[2 * k] = lo;
        wd[2 * k + 1] = hi;
    }
}

}  // namespace rowprep
}  // namespace m2
