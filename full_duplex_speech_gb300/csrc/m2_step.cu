// Single-frame cached step of the Mamba2 mixer core (the per-position update
// of the persistent "Mamba2 state" that the VoiceChat online session keeps;
// "docs/nemotron-voicechat.md", section Online session).
//
// Two kernels per call, both bound by memory latency or bandwidth:
//  1. step_conv_kernel: for every (session, channel) the 4-tap causal conv of
//     the cached tail plus this frame, bias, SiLU -> fp32 scratch; the tail is
//     shifted in place. Each channel is owned by exactly one thread, so the
//     in-place update of a tail that 16 heads read (B and C channels are
//     shared by a group) cannot race. It also turns dt_raw into dt.
//  2. step_ssm_kernel: for every (session, head, block of head_dim rows) the
//     fp32 state update h <- exp(dt A) h + dt x (outer) B and y = h.C + D x.
//     The state is 98% of the bytes; it is read and written once with 16-byte
//     vector accesses, one row of N fp32 per N/4 lanes.
// Both are launched with programmatic dependent launch: the conv kernel waits
// for its predecessor before reading anything, then lets the state-update
// kernel start, which issues its state loads (data written before the conv
// kernel began) and only then waits for the conv kernel's outputs.
#include "m2_common.cuh"
#include "m2_launch.h"

namespace m2 {

namespace {

// u = SiLU(conv_b + sum_k w[k] * window[k]) for 8 consecutive channels from
// c; the window is the cached tail (t-3, t-2, t-1) and this frame. All weight
// loads are issued before any arithmetic, so they overlap one another.
template <typename TA>
__device__ __forceinline__ void conv_silu8(const StepArgs& a, long c, const Act8<TA> (&tail)[3],
                                           const Act8<TA>& cur, float (&out)[8]) {
    const float4* w4 = reinterpret_cast<const float4*>(a.conv_w + c * 4);
    float4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __ldg(w4 + j);
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(a.conv_b + c));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(a.conv_b + c) + 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float u = j < 4 ? (&b0.x)[j] : (&b1.x)[j - 4];
        u = fmaf(w[j].x, tail[0].get(j), u);
        u = fmaf(w[j].y, tail[1].get(j), u);
        u = fmaf(w[j].z, tail[2].get(j), u);
        u = fmaf(w[j].w, cur.get(j), u);
        out[j] = silu_fast(u);
    }
}

// The tail after this frame: the oldest frame drops out, this frame enters.
template <typename TA>
__device__ __forceinline__ void shift_tail(const StepArgs& a, int ses, long c, const Act8<TA> (&tail)[3],
                                           const Act8<TA>& cur) {
    const long CH = a.s.CH();
    tail[1].store(a.conv, ((size_t)ses * 3 + 0) * CH + c);
    tail[2].store(a.conv, ((size_t)ses * 3 + 1) * CH + c);
    cur.store(a.conv, ((size_t)ses * 3 + 2) * CH + c);
}

template <typename TA>
__device__ __forceinline__ void load_tail(const StepArgs& a, int ses, long c, Act8<TA> (&tail)[3]) {
    const long CH = a.s.CH();
#pragma unroll
    for (int k = 0; k < 3; ++k) tail[k].load_rw(a.conv, ((size_t)ses * 3 + k) * CH + c);
}

constexpr int kConvThreads = 64;

template <typename TA>
__global__ void __launch_bounds__(kConvThreads) step_conv_kernel(StepArgs a) {
    const Shape& s = a.s;
    const int ses = blockIdx.y;
    const long CH = s.CH(), HP = s.HP(), GN = s.GN();
    const long nvec = CH / 8;
    const long v = (long)blockIdx.x * blockDim.x + threadIdx.x;
    pdl_wait();     // inputs and the conv tail may come from the previous kernel
    pdl_trigger();  // the state-update kernel may start loading the state
    if (v < nvec) {
        const long c = v * 8;
        // this frame's pre-conv input for channels [c, c+8)
        Act8<TA> cur;
        if (c < HP)
            cur.load(a.x, (size_t)ses * a.sx + c);
        else if (c < HP + GN)
            cur.load(a.B, (size_t)ses * a.sbc + (c - HP));
        else
            cur.load(a.C, (size_t)ses * a.sbc + (c - HP - GN));
        Act8<TA> tail[3];
        load_tail<TA>(a, ses, c, tail);
        float out[8];
        conv_silu8<TA>(a, c, tail, cur, out);
        float4* dst = reinterpret_cast<float4*>(a.ws_u + (size_t)ses * CH + c);
        dst[0] = make_float4(out[0], out[1], out[2], out[3]);
        dst[1] = make_float4(out[4], out[5], out[6], out[7]);
        shift_tail<TA>(a, ses, c, tail, cur);
    } else if (v - nvec < s.H) {
        const int h = (int)(v - nvec);
        const float z = load_act<TA>(a.dt_raw, (size_t)ses * a.sdt + h) + __ldg(a.dt_bias + h);
        a.ws_dt[(size_t)ses * s.H + h] = softplus_f32(z);
    }
}

// Rows of head_dim handled by one CTA and rows per thread of the row loop.
constexpr int kSsmThreads = 128;

template <typename TA, int N, int ROWS>
__global__ void __launch_bounds__(kSsmThreads) step_ssm_kernel(StepArgs a) {
    constexpr int LPR = N / 4;        // lanes per state row (float4 each)
    constexpr int RPW = 32 / LPR;     // rows per warp per pass
    constexpr int WARPS = kSsmThreads / 32;
    constexpr int RPP = RPW * WARPS;  // rows per CTA pass
    constexpr int PASSES = (ROWS + RPP - 1) / RPP;
    const Shape& s = a.s;
    const int ses = blockIdx.z, h = blockIdx.y, p0 = blockIdx.x * ROWS;
    const int g = h / (s.H / s.G);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n4 = (lane % LPR) * 4, sub = lane / LPR;

    const float* u = a.ws_u + (size_t)ses * s.CH();
    float* state = a.ssm + (((size_t)ses * s.H + h) * s.P) * N;

    // issue the state loads first: they are the bytes that matter
    float4 hv[PASSES];
    int prow[PASSES];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const int r = i * RPP + warp * RPW + sub;
        prow[i] = (r < ROWS && p0 + r < s.P) ? p0 + r : -1;
        if (prow[i] >= 0) hv[i] = __ldcs(reinterpret_cast<const float4*>(state + (size_t)prow[i] * N + n4));
    }
    // the state was written before the conv kernel started; its outputs are not
    pdl_wait();
    pdl_trigger();
    const float dt = a.ws_dt[(size_t)ses * s.H + h];
    const float A = -expf(__ldg(a.A_log + h));
    const float dA = expf(dt * A);
    const float Dh = __ldg(a.D + h);
    const float4 Bn = *reinterpret_cast<const float4*>(u + s.HP() + (long)g * N + n4);
    const float4 Cn = *reinterpret_cast<const float4*>(u + s.HP() + s.GN() + (long)g * N + n4);
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const int p = prow[i];
        float part = 0.f, xv = 0.f;
        if (p >= 0) {
            xv = u[(long)h * s.P + p];
            const float dx = dt * xv;
            float4 v = hv[i];
            v.x = fmaf(dA, v.x, dx * Bn.x);
            v.y = fmaf(dA, v.y, dx * Bn.y);
            v.z = fmaf(dA, v.z, dx * Bn.z);
            v.w = fmaf(dA, v.w, dx * Bn.w);
            __stcs(reinterpret_cast<float4*>(state + (size_t)p * N + n4), v);
            part = Cn.x * v.x;
            part = fmaf(Cn.y, v.y, part);
            part = fmaf(Cn.z, v.z, part);
            part = fmaf(Cn.w, v.w, part);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (p >= 0 && (lane % LPR) == 0)
            store_act<TA>(a.y, ((size_t)ses * s.H + h) * s.P + p, fmaf(Dh, xv, part));
    }
}

template <typename TA, int N>
cudaError_t launch_ssm(const StepArgs& a, cudaStream_t st) {
    constexpr int ROWS = 16;
    dim3 grid((a.s.P + ROWS - 1) / ROWS, a.s.H, a.S);
    return launch_pdl(step_ssm_kernel<TA, N, ROWS>, grid, dim3(kSsmThreads), 0, st, a);
}

template <typename TA>
cudaError_t launch_typed(const StepArgs& a, cudaStream_t st) {
    const long nvec = a.s.CH() / 8 + a.s.H;
    dim3 g1((unsigned)((nvec + kConvThreads - 1) / kConvThreads), a.S);
    cudaError_t e = launch_pdl(step_conv_kernel<TA>, g1, dim3(kConvThreads), 0, st, a);
    if (e != cudaSuccess) return e;
    switch (a.s.N) {
        case 16: return launch_ssm<TA, 16>(a, st);
        case 32: return launch_ssm<TA, 32>(a, st);
        case 64: return launch_ssm<TA, 64>(a, st);
        case 128: return launch_ssm<TA, 128>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t step_workspace_bytes(const Shape& s, int S) {
    const size_t u = ((size_t)S * s.CH() * 4 + 255) / 256 * 256;
    const size_t dt = ((size_t)S * s.H * 4 + 255) / 256 * 256;
    return u + dt;
}

cudaError_t launch_step(const StepArgs& a, cudaStream_t st) {
    if (a.S == 0) return cudaSuccess;
    return a.s.bf16 ? launch_typed<bf16_t>(a, st) : launch_typed<float>(a, st);
}

}  // namespace m2
