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
//  1. attn_split_kernel: one CTA per (chunk of up to 128 positions, kv head,
//     session; shorter chunks where there would be too few CTAs to fill the
//     GPU). Two bulk copies (the TMA engine) bring the chunk's cached keys
//     and values into shared memory: each is one contiguous run of rows. The
//     chunk holding position len[s] takes the new key and value from the
//     inputs instead, and writes them into the cache there (no other CTA
//     reads that slot). Then scores (8 lanes per position, 16 dims a lane, the
//     R heads' dot products reduced over the 8 lanes, q held in fp32
//     registers), the chunk's softmax statistics in the log2 domain (m = max,
//     l = sum of 2^(a - m)) and acc = sum_t 2^(a_t - m) v_t (16 threads per
//     value row, 8 dims each, all R heads at once), written as the chunk's
//     partial result.
//  2. attn_combine_kernel: per (kv head, session), merges the chunks:
//     M = max_i m_i, out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;

// Positions per chunk: 32 KB of keys and 32 KB of values per CTA (chunks of
// 64 positions, four CTAs an SM, measured slower for one session).
template <typename TA>
struct AttnTile {
    static constexpr int kTc = sizeof(TA) == 2 ? 128 : 64;
    static constexpr int kRowBytes = kAttnD * (int)sizeof(TA);
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + kTc * kRowBytes;
    static constexpr uint32_t kS = kV + kTc * kRowBytes;           // float [kAttnMaxR][kTc]: scores
    static constexpr uint32_t kP = kS + kAttnMaxR * kTc * 4;       // float [kTc][kAttnMaxR]: 2^(a - m)
    static constexpr uint32_t kM = kP + kAttnMaxR * kTc * 4;       // float [kAttnMaxR]
    static constexpr uint32_t kL = kM + kAttnMaxR * 4;             // float [kAttnMaxR]
    static constexpr uint32_t kBar = kL + kAttnMaxR * 4;           // one mbarrier
    static constexpr uint32_t kFlag = kBar + 8;                    // a wait gave up
    static constexpr uint32_t kBytes = kBar + 16;
    static_assert(8 * kAttnMaxR * kAttnD * 4 <= 2 * kTc * kRowBytes, "the K and V tiles hold the 8 groups' sums");
    static_assert(kV == kK + kTc * kRowBytes, "the K and V tiles are adjacent");
    static_assert(kAttnThreads == kAttnD, "one thread per dim in the final sum");
};

__host__ __device__ inline int attn_chunks(int Tmax, int tc) { return (Tmax + tc - 1) / tc; }

// Positions per chunk: the most a CTA holds, halved (down to 32) while the
// grid would have fewer than two CTAs per SM of the 152-SM GB300, so that a
// short cache of few sessions still spreads over the GPU. A function of the
// sizes alone: the workspace query needs no device.
int attn_chunk_len(int S, int Hkv, int Tmax, bool bf16) {
    int tc = bf16 ? AttnTile<bf16_t>::kTc : AttnTile<float>::kTc;
    while (tc > 32 && (long)S * Hkv * attn_chunks(Tmax, tc) < 2 * 152) tc /= 2;
    return tc;
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
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
    // the 16 values in fp32, in the order they were loaded
    __device__ __forceinline__ void unpack(float (&f)[16]) const {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const uint32_t* u = &w[c].x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (sizeof(TA) == 2) {
                    f[c * 8 + 2 * j] = __uint_as_float(u[j] << 16);
                    f[c * 8 + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                } else {
                    f[c * 4 + j] = __uint_as_float(u[j]);
                }
            }
        }
    }
};

// Dims [8 dq, 8 dq + 8) of a shared-memory row in fp32 (one 16-byte read in
// bf16, two in fp32; 16 threads read a row's 256 or 512 bytes together).
template <typename TA>
struct Row8 {
    __device__ __forceinline__ static void load(const uint8_t* row, int dq, float (&f)[8]) {
        if constexpr (sizeof(TA) == 2) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * dq);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(u[j] << 16);
                f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
            }
        } else {
            const float4 a = *reinterpret_cast<const float4*>(row + 32 * dq);
            const float4 b = *reinterpret_cast<const float4*>(row + 32 * dq + 16);
            f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
            f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
    }
};

// RM: the most query heads per kv head this instantiation handles (registers
// for q and the sums are sized by it).
template <typename TA, int RM>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(AttnArgs a) {
    using L = AttnTile<TA>;
    constexpr int TCM = L::kTc;  // the most positions a chunk holds
    constexpr int RB = L::kRowBytes;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    float* sS = reinterpret_cast<float*>(smem + L::kS);  // [kAttnMaxR][TCM] scores
    float* sP = reinterpret_cast<float*>(smem + L::kP);  // [TCM][kAttnMaxR] 2^(a - m)
    float* sM = reinterpret_cast<float*>(smem + L::kM);
    float* sL = reinterpret_cast<float*>(smem + L::kL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(smem + L::kFlag);

    const int chunk = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = a.Hq / a.Hkv;
    const int tc = a.tc;  // positions per chunk, at most TCM

    pdl_wait();  // the inputs and the caches may come from the previous kernel
    pdl_trigger();
    const int len = a.lens[s] + a.len_add;
    if (len < 0 || len >= a.Tmax) return;  // refused; the combine kernel reports it
    const int t0 = chunk * tc;
    if (t0 > len) return;                  // past this session's positions
    const int n = min(tc, len + 1 - t0);   // positions of this chunk
    const int ncached = min(n, len - t0);  // of which come from the cache
    const bool has_new = len - t0 < tc;    // position len is in this chunk

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
                                 (size_t)s * a.kv_ss * sizeof(TA) + (size_t)g * RB + piece * 16;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
            *reinterpret_cast<uint4*>((which ? sV : sK) + (size_t)(len - t0) * RB + piece * 16) = v;
            uint8_t* dst = reinterpret_cast<uint8_t*>(which ? a.v_cache : a.k_cache) + (kvrow + len) * RB + piece * 16;
            *reinterpret_cast<uint4*>(dst) = v;
        }
    }
    // this lane's 16 dims of the R query heads, in fp32 (lanes i = lane & 7)
    const int i8 = lane & 7, j4 = lane >> 3;
    float qf[RM][16];
#pragma unroll
    for (int r = 0; r < RM; ++r) {
        if (r < R) {
            Lane16<TA> qr;
            qr.load_global(reinterpret_cast<const uint8_t*>(a.q) + (size_t)s * a.q_ss * sizeof(TA) +
                               (size_t)(g * R + r) * RB, i8);
            qr.unpack(qf[r]);
        }
    }
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

    // scores a2 = scale log2(e) q . k (-inf past the chunk's end): groups of
    // four positions (8 lanes each) dealt round-robin to the warps
#pragma unroll 2
    for (int base = 4 * warp; base < tc; base += 4 * kAttnWarps) {
        const int t = base + j4;
        float kf[16];
        if (t < n) {
            Lane16<TA> kr;
            kr.load_shared(sK + (size_t)t * RB, i8);
            kr.unpack(kf);
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) kf[e] = 0.f;
        }
        // two partial sums a head: shorter dependent chains
        float d[RM];
#pragma unroll
        for (int r = 0; r < RM; ++r) {
            d[r] = 0.f;
            if (r < R) {
                float d1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    d[r] = fmaf(qf[r][e], kf[e], d[r]);
                    d1 = fmaf(qf[r][e + 1], kf[e + 1], d1);
                }
                d[r] += d1;
            }
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1)
#pragma unroll
            for (int r = 0; r < RM; ++r)
                if (r < R) d[r] += __shfl_xor_sync(0xffffffffu, d[r], off);
        // lane i of the position writes head i's score
#pragma unroll
        for (int r = 0; r < RM; ++r)
            if (r == i8 && r < R && t < tc) sS[r * TCM + t] = t < n ? d[r] * sl2 : -INFINITY;
    }
    __syncthreads();

    // softmax statistics per head (warp w takes heads w and w + 4); the
    // weights go out position-major for the value pass
    for (int r = warp; r < R; r += kAttnWarps) {
        float v[TCM / 32];
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < TCM / 32; ++c) {
            const int t = c * 32 + lane;
            v[c] = t < tc ? sS[r * TCM + t] : -INFINITY;
            m = fmaxf(m, v[c]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < TCM / 32; ++c) {
            const int t = c * 32 + lane;
            const float p = ex2_approx(v[c] - m);  // 0 for -inf
            if (t < tc) sP[t * kAttnMaxR + r] = p;
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

    // acc_r = sum_t p_r[t] v_t: 16 threads per position (8 dims each), the 8
    // groups of 16 taking every 8th position
    const int grp = tid >> 4, dq = tid & 15;
    float acc[RM][8];
#pragma unroll
    for (int r = 0; r < RM; ++r)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;
#pragma unroll 2
    for (int t = grp; t < n; t += 8) {
        float vf[8];
        Row8<TA>::load(sV + (size_t)t * RB, dq, vf);
        const float4 p0 = *reinterpret_cast<const float4*>(sP + t * kAttnMaxR);
        const float4 p1 = *reinterpret_cast<const float4*>(sP + t * kAttnMaxR + 4);
        const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int r = 0; r < RM; ++r)
            if (r < R)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr[r], vf[e], acc[r][e]);
    }
    // the 8 groups' sums through shared memory (over the K and V tiles, once
    // every thread is done reading them)
    __syncthreads();
    float* red = reinterpret_cast<float*>(sK);  // [8][R][kAttnD]
#pragma unroll
    for (int r = 0; r < RM; ++r) {
        if (r < R) {
            float* dst = red + (grp * R + r) * kAttnD + 8 * dq;
            *reinterpret_cast<float4*>(dst) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
        }
    }
    __syncthreads();
    const int nch = attn_chunks(a.Tmax, tc);
    const size_t part = ((size_t)s * a.Hkv + g) * nch + chunk;  // this chunk's partial result
    float* wacc = a.ws + part * R * kAttnD;
    for (int r = 0; r < R; ++r) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += red[(q * R + r) * kAttnD + tid];
        wacc[r * kAttnD + tid] = sum;
    }
    if (tid < R) {
        float* wml = a.ws + (size_t)a.S * a.Hkv * nch * R * kAttnD + part * R * 2;
        *reinterpret_cast<float2*>(wml + 2 * tid) = make_float2(sM[tid], sL[tid]);
    }
}

// out_h = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i over the chunks of
// session s; thread = (query head r of kv head g, dims pair). The 64 threads
// of a head find M together (every 64th chunk each); the sum over chunks is
// unrolled so that its loads are in flight together.
template <typename TA>
__global__ void __launch_bounds__(kAttnMaxR * 64) attn_combine_kernel(AttnArgs a) {
    __shared__ float sMax[kAttnMaxR][2];
    const int g = blockIdx.x, s = blockIdx.y;
    const int tc = a.tc;
    const int R = a.Hq / a.Hkv;
    const int r = threadIdx.x >> 6, dp = threadIdx.x & 63, lane = threadIdx.x & 31;
    pdl_wait();  // the split kernel's partial results
    pdl_trigger();
    const int len = a.lens[s] + a.len_add;
    const bool bad = len < 0 || len >= a.Tmax;  // the same for the whole block
    const int nch = attn_chunks(a.Tmax, tc);
    const int nc = bad ? 0 : len / tc + 1;  // chunks holding positions 0..len
    const size_t part0 = ((size_t)s * a.Hkv + g) * nch;
    const float* wml = a.ws + (size_t)a.S * a.Hkv * nch * R * kAttnD;
    float m = -INFINITY;
    for (int c = dp; c < nc; c += 64) m = fmaxf(m, wml[((part0 + c) * R + r) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) sMax[r][dp >> 5] = m;
    __syncthreads();
    float v0 = 0.f, v1 = 0.f;
    if (!bad) {
        const float M = fmaxf(sMax[r][0], sMax[r][1]);
        float den = 0.f;
#pragma unroll 8
        for (int c = 0; c < nc; ++c) {
            const float2 ml = *reinterpret_cast<const float2*>(wml + ((part0 + c) * R + r) * 2);
            const float2 acc = *reinterpret_cast<const float2*>(a.ws + ((part0 + c) * R + r) * kAttnD + 2 * dp);
            const float f = ex2_approx(ml.x - M);
            v0 = fmaf(f, acc.x, v0);
            v1 = fmaf(f, acc.y, v1);
            den = fmaf(f, ml.y, den);
        }
        const float inv = 1.f / den;
        v0 *= inv;
        v1 *= inv;
    } else if (threadIdx.x == 0) {
        atomicOr(a.err, ERR_ATTN_LENGTH);
    }
    const size_t o = (size_t)s * a.out_ss + (size_t)(g * R + r) * kAttnD + 2 * dp;
    if constexpr (sizeof(TA) == 2) {
        const uint32_t w = (uint32_t)float_to_bf16_bits(v0) | ((uint32_t)float_to_bf16_bits(v1) << 16);
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out) + o) = w;
    } else {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + o) = make_float2(v0, v1);
    }
}

template <typename TA, int RM>
cudaError_t launch_split(const AttnArgs& a, cudaStream_t st) {
    using L = AttnTile<TA>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(attn_split_kernel<TA, RM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::kBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int nch = attn_chunks(a.Tmax, a.tc);
    return launch_pdl(attn_split_kernel<TA, RM>, dim3(nch, a.Hkv, a.S), dim3(kAttnThreads), L::kBytes, st, a);
}

template <typename TA>
cudaError_t launch_attn_typed(const AttnArgs& a, cudaStream_t st) {
    const int R = a.Hq / a.Hkv;
    // register sets for up to 2, 5 (the Nemotron-H layers) or 8 query heads per kv head
    cudaError_t e = R <= 2 ? launch_split<TA, 2>(a, st) : R <= 5 ? launch_split<TA, 5>(a, st)
                                                                 : launch_split<TA, 8>(a, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_combine_kernel<TA>, dim3(a.Hkv, a.S), dim3(R * (kAttnD / 2)), 0, st, a);
}

}  // namespace

size_t attn_workspace_bytes(int S, int Hq, int Hkv, int Tmax, bool bf16) {
    if (S <= 0 || Hq <= 0 || Hkv <= 0 || Tmax <= 0 || Hq % Hkv) return 0;
    const int tc = attn_chunk_len(S, Hkv, Tmax, bf16);
    const size_t parts = (size_t)S * Hkv * attn_chunks(Tmax, tc) * (Hq / Hkv);
    return parts * (kAttnD + 2) * sizeof(float);
}

cudaError_t launch_attn_decode(const AttnArgs& a0, cudaStream_t st) {
    if (a0.S == 0) return cudaSuccess;
    AttnArgs a = a0;
    a.tc = attn_chunk_len(a.S, a.Hkv, a.Tmax, a.bf16);
    return a.bf16 ? launch_attn_typed<bf16_t>(a, st) : launch_attn_typed<float>(a, st);
}

}  // namespace m2
