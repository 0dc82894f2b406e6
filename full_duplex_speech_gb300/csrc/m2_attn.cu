// One cached decode position of the hybrid model's grouped-query attention
// layers with their KV caches: the Nemotron-H attention layers (40 query
// heads, 8 kv heads, head_dim 128, no bias, no positional rotation in the
// configuration; VoiceChat issue, section config.json / text_config), whose
// caches are part of the state a session keeps ("docs/nemotron-voicechat.md",
// section Online session, persistent-state table).
//
// For session s with len[s] positions cached, the new key and value of each
// kv head go to position len[s], and query head h (kv head g = h / R,
// R = Hq / Hkv) attends over positions 0 .. len[s]:
//     a_t = scale q_h . k_t,  out_h = sum_t softmax(a)_t v_t.
// Bound by HBM: every cached key and value is read once per position (the R
// query heads of a kv head share each read), at 2 x 256 B per position and
// kv head in bf16 against 4R flops per byte.
//
// Two kernels, both launched with programmatic dependent launch:
//  1. attn_split_kernel: one CTA per (chunk of kTc positions, kv head,
//     session). Two bulk copies (the TMA engine) bring the chunk's cached keys
//     and values into shared memory: each is one contiguous run of rows. The
//     chunk holding position len[s] takes the new key and value from the
//     inputs instead, and writes them into the cache there (no other CTA
//     reads that slot). Then scores (8 lanes per position, 16 dims a lane, the
//     R heads' dot products reduced over the 8 lanes), the chunk's softmax
//     statistics in the log2 domain (m = max, l = sum of 2^(a - m)) and
//     acc = sum_t 2^(a_t - m) v_t, written as the chunk's partial result.
//  2. attn_combine_kernel: per (kv head, session), merges the chunks:
//     M = max_i m_i, out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;

// Positions per chunk: 32 KB of keys and 32 KB of values per CTA.
template <typename TA>
struct AttnTile {
    static constexpr int kTc = sizeof(TA) == 2 ? 128 : 64;
    static constexpr int kRowBytes = kAttnD * (int)sizeof(TA);
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + kTc * kRowBytes;
    static constexpr uint32_t kS = kV + kTc * kRowBytes;           // float [kAttnMaxR][kTc]: scores, then 2^(a-m)
    static constexpr uint32_t kM = kS + kAttnMaxR * kTc * 4;       // float [kAttnMaxR]
    static constexpr uint32_t kL = kM + kAttnMaxR * 4;             // float [kAttnMaxR]
    static constexpr uint32_t kBar = kL + kAttnMaxR * 4;           // one mbarrier
    static constexpr uint32_t kFlag = kBar + 8;                    // a wait gave up
    static constexpr uint32_t kBytes = kBar + 16;
    static_assert(kAttnMaxR * kAttnD * 4 <= kTc * kRowBytes, "the key tile holds the half-sums of acc");
};

__host__ __device__ inline int attn_chunks(int Tmax, int tc) { return (Tmax + tc - 1) / tc; }

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// acc += q . k over two bf16 pairs held in 32-bit words: mixed-precision fmas
// (bf16 x bf16 products are exact in fp32), no unpacking.
__device__ __forceinline__ float dot2_bf16(uint32_t qw, uint32_t kw, float acc) {
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %1;\n\t"
        "mov.b32 {kl, kh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.bf16 %0, qh, kh, %0;\n\t}"
        : "+f"(acc)
        : "r"(qw), "r"(kw));
    return acc;
}

// The 16 dims of q (or k) a lane holds: the 16-byte chunks i and i + 8 of a
// bf16 row (8 dims each), or chunks i, i + 8, i + 16, i + 24 of an fp32 row
// (4 dims each). Lanes i = 0..7 of one position read chunks whose bank groups
// differ, so a row is read without bank conflicts.
template <typename TA>
struct Lane16 {
    static constexpr int kChunks = sizeof(TA) == 2 ? 2 : 4;
    uint4 w[kChunks];
    __device__ __forceinline__ void load_global(const void* row, int i) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) w[c] = __ldg(reinterpret_cast<const uint4*>(row) + i + 8 * c);
    }
    __device__ __forceinline__ void load_shared(const uint8_t* row, int i) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) w[c] = *reinterpret_cast<const uint4*>(row + 16 * (i + 8 * c));
    }
};

// q . k over the lane's 16 dims
template <typename TA>
__device__ __forceinline__ float lane_dot(const Lane16<TA>& q, const Lane16<TA>& k) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < Lane16<TA>::kChunks; ++c) {
        const uint32_t* qw = &q.w[c].x;
        const uint32_t* kw = &k.w[c].x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (sizeof(TA) == 2)
                acc = dot2_bf16(qw[j], kw[j], acc);
            else
                acc = fmaf(__uint_as_float(qw[j]), __uint_as_float(kw[j]), acc);
        }
    }
    return acc;
}

template <typename TA>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(AttnArgs a) {
    using L = AttnTile<TA>;
    constexpr int TC = L::kTc;
    constexpr int RB = L::kRowBytes;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    float* sS = reinterpret_cast<float*>(smem + L::kS);
    float* sM = reinterpret_cast<float*>(smem + L::kM);
    float* sL = reinterpret_cast<float*>(smem + L::kL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(smem + L::kFlag);

    const int chunk = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = a.Hq / a.Hkv;

    pdl_wait();  // the inputs and the caches may come from the previous kernel
    pdl_trigger();
    const int len = a.lens[s];
    if (len < 0 || len >= a.Tmax) return;  // refused; the combine kernel reports it
    const int t0 = chunk * TC;
    if (t0 > len) return;                  // past this session's positions
    const int n = min(TC, len + 1 - t0);   // positions of this chunk
    const int ncached = min(n, len - t0);  // of which come from the cache
    const bool has_new = len - t0 < TC;    // position len is in this chunk

    const size_t kvrow = ((size_t)s * a.Hkv + g) * a.Tmax;  // row of position 0
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(a.k_cache);
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(a.v_cache);
    if (tid == 0) {
        *sFlag = 0;
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
        if (ncached > 0) {
            const uint32_t bytes = (uint32_t)ncached * RB;
            tc::mbar_arrive_expect_tx(bar, 2 * bytes);
            tc::bulk_g2s(sK, kc + (kvrow + t0) * RB, bytes, bar);
            tc::bulk_g2s(sV, vc + (kvrow + t0) * RB, bytes, bar);
        }
    }
    // the new position: into its shared-memory row and into the cache
    if (has_new) {
        constexpr int V16 = RB / 16;  // 16-byte pieces of one row
        if (tid < 2 * V16) {
            const int which = tid / V16, piece = tid % V16;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(which ? a.v_new : a.k_new) +
                                 ((size_t)s * a.Hkv + g) * RB + piece * 16;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
            *reinterpret_cast<uint4*>((which ? sV : sK) + (size_t)(len - t0) * RB + piece * 16) = v;
            uint8_t* dst = reinterpret_cast<uint8_t*>(which ? a.v_cache : a.k_cache) + (kvrow + len) * RB + piece * 16;
            *reinterpret_cast<uint4*>(dst) = v;
        }
    }
    // this lane's 16 dims of the R query heads (lanes i = lane & 7)
    const int i8 = lane & 7, j4 = lane >> 3;
    Lane16<TA> q[kAttnMaxR];
#pragma unroll
    for (int r = 0; r < kAttnMaxR; ++r)
        if (r < R)
            q[r].load_global(reinterpret_cast<const uint8_t*>(a.q) + ((size_t)s * a.Hq + g * R + r) * RB, i8);
    const float sl2 = a.scale * kLog2e;
    __syncthreads();
    if (ncached > 0 && !tc::mbar_wait(bar, 0)) {
        atomicOr(a.err, ERR_MBAR_TIMEOUT_LOAD);
        *sFlag = 1;
    }
    __syncthreads();
    if (*sFlag) {
        // the whole CTA gives up; thread 0 lets the copies land before it exits
        if (tid == 0) tc::mbar_wait(bar, 0, 100000000ull);
        return;
    }

    // scores: warp w takes positions [w TC/4, (w+1) TC/4), four at a time
    // (8 lanes each); a2 = scale log2(e) q . k, -inf past the chunk's end
    constexpr int PW = TC / kAttnWarps;
#pragma unroll 2
    for (int it = 0; it < PW / 4; ++it) {
        const int t = warp * PW + it * 4 + j4;
        Lane16<TA> k;
        if (t < n) k.load_shared(sK + (size_t)t * RB, i8);
        float d[kAttnMaxR];
#pragma unroll
        for (int r = 0; r < kAttnMaxR; ++r) d[r] = (r < R && t < n) ? lane_dot<TA>(q[r], k) : 0.f;
#pragma unroll
        for (int off = 1; off < 8; off <<= 1)
#pragma unroll
            for (int r = 0; r < kAttnMaxR; ++r)
                if (r < R) d[r] += __shfl_xor_sync(0xffffffffu, d[r], off);
        // lane i of the position writes head i's score
#pragma unroll
        for (int r = 0; r < kAttnMaxR; ++r)
            if (r == i8 && r < R) sS[r * TC + t] = t < n ? d[r] * sl2 : -INFINITY;
    }
    __syncthreads();

    // softmax statistics per head: warp w takes heads w and w + 4
    for (int r = warp; r < R; r += kAttnWarps) {
        float v[TC / 32];
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < TC / 32; ++c) {
            v[c] = sS[r * TC + c * 32 + lane];
            m = fmaxf(m, v[c]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < TC / 32; ++c) {
            const float p = ex2_approx(v[c] - m);  // 0 for -inf
            sS[r * TC + c * 32 + lane] = p;
            l += p;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
            sM[r] = m;
            sL[r] = l;
        }
    }
    __syncthreads();

    // acc_r = sum_t p_r[t] v_t: thread = (dims pair dp, half of the positions)
    const int dp = tid & 63, hf = tid >> 6;
    float acc[kAttnMaxR][2];
#pragma unroll
    for (int r = 0; r < kAttnMaxR; ++r) acc[r][0] = acc[r][1] = 0.f;
    const int ta = hf * (TC / 2), tb = min(n, ta + TC / 2);
#pragma unroll 4
    for (int t = ta; t < tb; ++t) {
        float v0, v1;
        if constexpr (sizeof(TA) == 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(sV + (size_t)t * RB + 4 * dp);
            v0 = __uint_as_float(w << 16);
            v1 = __uint_as_float(w & 0xFFFF0000u);
        } else {
            const float2 w = *reinterpret_cast<const float2*>(sV + (size_t)t * RB + 8 * dp);
            v0 = w.x;
            v1 = w.y;
        }
#pragma unroll
        for (int r = 0; r < kAttnMaxR; ++r) {
            if (r < R) {
                const float p = sS[r * TC + t];
                acc[r][0] = fmaf(p, v0, acc[r][0]);
                acc[r][1] = fmaf(p, v1, acc[r][1]);
            }
        }
    }
    // the second half's sums through shared memory (the key tile is free now)
    float* sAcc = reinterpret_cast<float*>(sK);
    if (hf == 1) {
#pragma unroll
        for (int r = 0; r < kAttnMaxR; ++r)
            if (r < R) *reinterpret_cast<float2*>(sAcc + r * kAttnD + 2 * dp) = make_float2(acc[r][0], acc[r][1]);
    }
    __syncthreads();
    if (hf == 0) {
        const int nch = attn_chunks(a.Tmax, TC);
        const size_t part = ((size_t)s * a.Hkv + g) * nch + chunk;  // this chunk's partial result
        float* wacc = a.ws + part * R * kAttnD;
#pragma unroll
        for (int r = 0; r < kAttnMaxR; ++r) {
            if (r < R) {
                const float2 o = *reinterpret_cast<const float2*>(sAcc + r * kAttnD + 2 * dp);
                *reinterpret_cast<float2*>(wacc + r * kAttnD + 2 * dp) = make_float2(acc[r][0] + o.x, acc[r][1] + o.y);
            }
        }
        if (tid < R) {
            float* wml = a.ws + (size_t)a.S * a.Hkv * nch * R * kAttnD + part * R * 2;
            *reinterpret_cast<float2*>(wml + 2 * tid) = make_float2(sM[tid], sL[tid]);
        }
    }
}

// out_h = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i over the chunks of
// session s; thread = (query head r of kv head g, dims pair).
template <typename TA>
__global__ void attn_combine_kernel(AttnArgs a) {
    constexpr int TC = AttnTile<TA>::kTc;
    const int g = blockIdx.x, s = blockIdx.y;
    const int R = a.Hq / a.Hkv;
    const int r = threadIdx.x >> 6, dp = threadIdx.x & 63;
    pdl_wait();  // the split kernel's partial results
    pdl_trigger();
    const int len = a.lens[s];
    const size_t o = ((size_t)s * a.Hq + g * R + r) * kAttnD + 2 * dp;
    float v0 = 0.f, v1 = 0.f;
    if (len < 0 || len >= a.Tmax) {
        if (threadIdx.x == 0) atomicOr(a.err, ERR_ATTN_LENGTH);
    } else {
        const int nch = attn_chunks(a.Tmax, TC);
        const int nc = len / TC + 1;  // chunks holding positions 0..len
        const size_t part0 = ((size_t)s * a.Hkv + g) * nch;
        const float* wml = a.ws + (size_t)a.S * a.Hkv * nch * R * kAttnD;
        float M = -INFINITY;
        for (int c = 0; c < nc; ++c) M = fmaxf(M, wml[((part0 + c) * R + r) * 2]);
        float den = 0.f;
        for (int c = 0; c < nc; ++c) {
            const float2 ml = *reinterpret_cast<const float2*>(wml + ((part0 + c) * R + r) * 2);
            const float f = ex2_approx(ml.x - M);
            const float2 acc = *reinterpret_cast<const float2*>(a.ws + ((part0 + c) * R + r) * kAttnD + 2 * dp);
            v0 = fmaf(f, acc.x, v0);
            v1 = fmaf(f, acc.y, v1);
            den = fmaf(f, ml.y, den);
        }
        const float inv = 1.f / den;
        v0 *= inv;
        v1 *= inv;
    }
    if constexpr (sizeof(TA) == 2) {
        const uint32_t w = (uint32_t)float_to_bf16_bits(v0) | ((uint32_t)float_to_bf16_bits(v1) << 16);
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out) + o) = w;
    } else {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + o) = make_float2(v0, v1);
    }
}

template <typename TA>
cudaError_t launch_attn_typed(const AttnArgs& a, cudaStream_t st) {
    using L = AttnTile<TA>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(attn_split_kernel<TA>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int nch = attn_chunks(a.Tmax, L::kTc);
    e = launch_pdl(attn_split_kernel<TA>, dim3(nch, a.Hkv, a.S), dim3(kAttnThreads), L::kBytes, st, a);
    if (e != cudaSuccess) return e;
    const int R = a.Hq / a.Hkv;
    return launch_pdl(attn_combine_kernel<TA>, dim3(a.Hkv, a.S), dim3(R * (kAttnD / 2)), 0, st, a);
}

}  // namespace

size_t attn_workspace_bytes(int S, int Hq, int Hkv, int Tmax, bool bf16) {
    if (S <= 0 || Hq <= 0 || Hkv <= 0 || Tmax <= 0 || Hq % Hkv) return 0;
    const int tc = bf16 ? AttnTile<bf16_t>::kTc : AttnTile<float>::kTc;
    const size_t parts = (size_t)S * Hkv * attn_chunks(Tmax, tc) * (Hq / Hkv);
    return parts * (kAttnD + 2) * sizeof(float);
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st) {
    if (a.S == 0) return cudaSuccess;
    return a.bf16 ? launch_attn_typed<bf16_t>(a, st) : launch_attn_typed<float>(a, st);
}

}  // namespace m2
