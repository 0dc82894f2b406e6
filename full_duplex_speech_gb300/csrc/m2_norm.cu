// Gated RMSNorm of the mixer output (the standard Mamba-2 output norm; the
// VoiceChat issue "feat(nemotron_voicechat): load the VoiceChat checkpoint and
// run offline duplex inference", section config.json / text_config, gives its
// eps, rms_norm_eps 1e-5):
//     v   = y * silu(z)
//     out = weight * v / sqrt(mean over the channel group of v^2 + eps)
// over ngroups contiguous groups of H*P/ngroups channels per position.
//
// One CTA per (position, group), sized to the group: each thread issues all
// its 16-byte loads of y and z at once (at most four of each), keeps them in
// registers across a block reduction of sum(v^2), and writes its own
// elements, after every read of the group, so out may alias y or z. Bound by
// HBM: 6 bytes per channel for bf16 activations (y, z in; out).
#include "m2_common.cuh"
#include "m2_launch.h"

namespace m2 {

namespace {

template <typename TA> __device__ __forceinline__ void store8(void* base, size_t elem, const float (&v)[8]);
template <> __device__ __forceinline__ void store8<bf16_t>(void* base, size_t elem, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = (uint32_t)float_to_bf16_bits(v[2 * j]) | ((uint32_t)float_to_bf16_bits(v[2 * j + 1]) << 16);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + elem) = make_uint4(w[0], w[1], w[2], w[3]);
}
template <> __device__ __forceinline__ void store8<float>(void* base, size_t elem, const float (&v)[8]) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
}

constexpr int kMaxVecs = 4;  // 16-byte vectors per thread: groups of up to 4 * 1024 * 8 channels

// One CTA per (position, group) of blockDim.x >= vectors / VPT threads. VPT
// is the smallest of 1, 2, 4 that covers the group with at most 1024 threads
// (1 at the Nemotron-H shape); fewer registers keep more CTAs resident.
template <typename TA, int VPT>
__global__ void __launch_bounds__(1024) gated_norm_kernel(NormArgs a) {
    __shared__ float sPart[32];
    const long r = blockIdx.x;
    const int g = blockIdx.y;
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long width = a.s.HP(), gw = width / a.s.G;
    const int nvec = (int)(gw / 8);
    const size_t base = (size_t)r * width + (size_t)g * gw;
    pdl_wait();  // y and z may come from the previous kernel
    pdl_trigger();

    Act8<TA> yv[VPT], zv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = tid + nt * k;
        if (v < nvec) {
            yv[k].load_rw(a.y, base + (size_t)v * 8);
            zv[k].load_rw(a.z, base + (size_t)v * 8);
        }
    }
    float u[VPT][8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const bool live = tid + nt * k < nvec;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            u[k][j] = live ? yv[k].get(j) * silu_fast(zv[k].get(j)) : 0.f;
            ss = fmaf(u[k][j], u[k][j], ss);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) sPart[warp] = ss;
    __syncthreads();  // also: every read of the group precedes every write
    float tot = 0.f;
    for (int w = 0; w < (nt + 31) / 32; ++w) tot += sPart[w];
    const float inv = rsqrtf(tot / (float)gw + a.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = tid + nt * k;
        if (v < nvec) {
            const float4* w4 = reinterpret_cast<const float4*>(a.weight + (size_t)g * gw + (size_t)v * 8);
            const float4 w0 = __ldg(w4), w1 = __ldg(w4 + 1);
            float o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = (j < 4 ? (&w0.x)[j] : (&w1.x)[j - 4]) * u[k][j] * inv;
            store8<TA>(a.out, base + (size_t)v * 8, o);
        }
    }
}

template <int VPT>
cudaError_t launch_vpt(const NormArgs& a, int nvec, cudaStream_t st) {
    const int threads = ((nvec + VPT - 1) / VPT + 31) / 32 * 32;
    const dim3 grid((unsigned)a.rows, (unsigned)a.s.G);
    return a.s.bf16 ? launch_pdl(gated_norm_kernel<bf16_t, VPT>, grid, dim3(threads), 0, st, a)
                    : launch_pdl(gated_norm_kernel<float, VPT>, grid, dim3(threads), 0, st, a);
}

}  // namespace

cudaError_t launch_gated_norm(const NormArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    const int nvec = (int)(a.s.HP() / a.s.G / 8);
    if (nvec <= 1024) return launch_vpt<1>(a, nvec, st);
    if (nvec <= 2048) return launch_vpt<2>(a, nvec, st);
    if (nvec <= kMaxVecs * 1024) return launch_vpt<kMaxVecs>(a, nvec, st);
    return cudaErrorInvalidValue;
}

}  // namespace m2
