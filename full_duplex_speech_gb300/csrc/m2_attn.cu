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
//  1. a split kernel that computes partial results over runs of positions:
//     - bf16 caches: attn_walk_kernel, on the tensor cores. One CTA per
//       (walker, kv head, session): a walker takes a run of 64-position
//       chunks, brought into shared memory by 2-D TMA copies through a
//       3-stage ring; its four warps keep their own online softmax over 16
//       positions of every chunk, with the scores (query heads x positions)
//       and the weighted values (query heads x dims) as mma.sync products.
//     - fp32 caches: attn_split_kernel, on the CUDA cores. One CTA per (chunk
//       of up to 64 positions, kv head, session; shorter chunks where there
//       would be too few CTAs to fill the GPU). Two bulk copies (the TMA
//       engine) bring the chunk's cached keys and values into shared memory;
//       then scores (8 lanes per position, 16 dims a lane, the R heads' dot
//       products reduced over the 8 lanes, q held in fp32 registers), the
//       chunk's softmax statistics in the log2 domain (m = max, l = sum of
//       2^(a - m)) and acc = sum_t 2^(a_t - m) v_t (16 threads per value row,
//       8 dims each, all R heads at once), written as the chunk's partial result.
//     The run holding position len[s] takes the new key and value from the
//     inputs instead of the cache, and writes them into the cache there (no
//     other CTA reads that slot).
//  2. attn_combine_kernel: per (kv head, session), merges the partial results:
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
int attn_walk_chunks(int S, int Hkv, int Tmax);

// bf16 caches go to the tensor-core walkers, whose 2-D copies address the
// caches' rows (S x Hkv x Tmax of them) with 32-bit coordinates.
bool attn_use_walk(int S, int Hkv, int Tmax, bool bf16) {
    return bf16 && (long long)S * Hkv * Tmax < (1LL << 31) - 64;
}

int attn_chunk_len(int S, int Hkv, int Tmax, bool bf16) {
    if (attn_use_walk(S, Hkv, Tmax, bf16)) return attn_walk_chunks(S, Hkv, Tmax) * 64;  // a walker's run of 64-position chunks
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

// ---------------------------------------------------------------------------
// bf16 caches: the split kernel on the tensor cores. A CTA ("walker") takes a
// run of consecutive 64-position chunks of one (session, kv head); a 3-stage
// ring of 2-D TMA copies (128-byte swizzle) keeps the next chunks' keys and
// values in flight while it computes. Each of its four warps takes 16
// positions of every chunk and keeps its own online softmax, so the warps
// meet only at the chunk boundary where a stage is refilled:
//     scores  S (16 x 16) = Q (16 query rows, R real) . K^T      mma m16n8k16
//     P = 2^(S log2e scale - m), m the running max, l += sum P
//     acc (16 x 128) += P . V      (P as bf16 hi + lo: two MMAs)
// The scores' accumulator fragments are the P operand's fragments as they
// stand (row = query head, column = position). The four warps' (m, l, acc)
// are merged at the end into the walker's partial result, which the combine
// kernel merges with the other walkers' as it does the chunks'.
constexpr int kWalkTc = 64;                        // positions per chunk
constexpr int kWalkStages = 3;
constexpr int kWalkThreads = 128;
constexpr uint32_t kWalkBox = kWalkTc * 128;        // one box: 64 rows x 64 dims of bf16 (8 KiB)
constexpr uint32_t kWalkStage = 4 * kWalkBox;       // K (2 boxes) + V (2 boxes)
constexpr uint32_t kWalkBar = kWalkStages * kWalkStage;
constexpr uint32_t kWalkSmem = kWalkBar + 64 + 1024;  // + barriers, + slack to align to 1024

// Byte offset of (row r, dim d) in a stage's K or V tile: two 64-dim boxes,
// 128-byte rows, the 16-byte pieces of a row XOR-ed with r % 8.
__device__ __forceinline__ uint32_t walk_off(int r, int d) {
    return (uint32_t)(d >> 6) * kWalkBox + (uint32_t)r * 128u + ((((uint32_t)(d & 63) >> 3) ^ (uint32_t)(r & 7)) << 4) +
           ((uint32_t)(d & 7) << 1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += A B, m16n8k16, bf16 in, fp32 accumulate; A's rows 8..15 are zero here
__device__ __forceinline__ void mma_rows8(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kWalkThreads, 2) attn_walk_kernel(AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                                                                    const __grid_constant__ CUtensorMap tmv, int cpw) {
    extern __shared__ uint8_t walk_smem_raw[];
    uint8_t* sm = walk_smem_raw + ((1024u - (tc::smem_u32(walk_smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kWalkBar);  // one per stage: its copies landed
    const int wk = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, t = lane & 3;  // fragment row (query head) and lane in its quad
    const int R = a.Hq / a.Hkv;
    constexpr int RB = kAttnD * 2;  // bytes of one cached row

    pdl_wait();  // the inputs and the caches may come from the previous kernel
    pdl_trigger();
    const int len = a.lens[s] + a.len_add;
    if (len < 0 || len >= a.Tmax) return;  // refused; the combine kernel reports it
    const int nch = len / kWalkTc + 1;     // chunks holding positions 0 .. len
    const int cb = wk * cpw, ce = min(cb + cpw, nch);
    if (cb >= ce) return;                  // past this session's positions
    const int row0 = (s * a.Hkv + g) * a.Tmax;  // tensor row of position 0

    auto issue = [&](int c) {  // one thread: chunk c's keys and values into its stage
        const int st = (c - cb) % kWalkStages;
        uint8_t* dst = sm + st * kWalkStage;
        tc::mbar_arrive_expect_tx(bar + st, kWalkStage);
        const int y = row0 + c * kWalkTc;
        tc::tma_load_2d(dst, &tmk, 0, y, bar + st);
        tc::tma_load_2d(dst + kWalkBox, &tmk, 64, y, bar + st);
        tc::tma_load_2d(dst + 2 * kWalkBox, &tmv, 0, y, bar + st);
        tc::tma_load_2d(dst + 3 * kWalkBox, &tmv, 64, y, bar + st);
    };
    if (tid == 0) {
        for (int i = 0; i < kWalkStages; ++i) tc::mbar_init(bar + i, 1);
        tc::fence_mbar_init();
        for (int c = cb; c < min(ce, cb + kWalkStages); ++c) issue(c);
    }
    // the query rows as the A operand (row = query head gq of this kv head;
    // rows past R, and rows 8..15, zero): per 16-dim K-step two bf16 pairs
    uint32_t qa[8][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                                 (size_t)s * a.q_ss + (size_t)(g * R + min(gq, R - 1)) * kAttnD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qa[kk][0] = gq < R ? __ldg(qrow + 8 * kk + t) : 0u;
            qa[kk][1] = gq < R ? __ldg(qrow + 8 * kk + 4 + t) : 0u;
        }
    }
    const float sl2 = a.scale * kLog2e;
    float m = -1e30f, l = 0.f;  // running max (finite: a fully masked row stays harmless) and sum
    float acc[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[dt][e] = 0.f;
    __syncthreads();  // the barriers are initialised

    bool ok = true;
    for (int c = cb; c < ce; ++c) {
        const int st = (c - cb) % kWalkStages;
        const uint32_t phase = ((c - cb) / kWalkStages) & 1;
        uint8_t* sK = sm + st * kWalkStage;
        uint8_t* sV = sK + 2 * kWalkBox;
        if (!tc::mbar_wait(bar + st, phase)) {
            atomicOr(a.err, ERR_MBAR_TIMEOUT_LOAD);
            ok = false;
        }
        if (c == nch - 1) {
            // the chunk holding position len: the new key and value go into
            // their rows here and into the caches; the value rows past len
            // (whatever the cache holds there) become zeros
            const int pl = len - c * kWalkTc;
            if (tid < 32) {
                const int which = tid >> 4, piece = tid & 15;
                const uint8_t* src = reinterpret_cast<const uint8_t*>(which ? a.v_new : a.k_new) +
                                     ((size_t)s * a.kv_ss + (size_t)g * kAttnD) * 2 + piece * 16;
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
                *reinterpret_cast<uint4*>((which ? sV : sK) + walk_off(pl, piece * 8)) = v;
                uint8_t* dst = reinterpret_cast<uint8_t*>(which ? a.v_cache : a.k_cache) + ((size_t)row0 + len) * RB +
                               piece * 16;
                *reinterpret_cast<uint4*>(dst) = v;
            }
            for (int e = tid; e < (kWalkTc - 1 - pl) * 16; e += kWalkThreads) {
                const int r = pl + 1 + e / 16, piece = e % 16;
                *reinterpret_cast<uint4*>(sV + walk_off(r, piece * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
        }
        const uint32_t kb = tc::smem_u32(sK), vb = tc::smem_u32(sV);
        // scores of this warp's positions 16 warp .. +15 (two 8-position tiles)
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
            const int r = 16 * warp + 8 * nt + (lane & 7);
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) {
                uint32_t b[4];
                ldsm_x4(kb + walk_off(r, 32 * kk2 + 8 * (lane >> 3)), b);
                mma_rows8(sc[nt], qa[2 * kk2][0], qa[2 * kk2][1], b[0], b[1]);
                mma_rows8(sc[nt], qa[2 * kk2 + 1][0], qa[2 * kk2 + 1][1], b[2], b[3]);
            }
        }
        // online softmax of row gq over these 16 positions (-inf past len)
        float sv[2][2], mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int pos = c * kWalkTc + 16 * warp + 8 * nt + 2 * t + e;
                sv[nt][e] = (pos <= len && gq < R) ? sc[nt][e] * sl2 : -INFINITY;
                mx = fmaxf(mx, sv[nt][e]);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m, mx);
        const float corr = ex2_approx(m - mn);
        m = mn;
        float p[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) p[nt][e] = ex2_approx(sv[nt][e] - mn);  // 0 for -inf
        l = fmaf(l, corr, (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            acc[dt][0] *= corr;
            acc[dt][1] *= corr;
        }
        // P as bf16 hi + lo (p = hi + lo to ~2^-16): row gq, positions 2t, 2t+1 and 8+2t, 8+2t+1
        const uint32_t h0 = pack_bf16x2(p[0][0], p[0][1]), h1 = pack_bf16x2(p[1][0], p[1][1]);
        const uint32_t l0 = pack_bf16x2(p[0][0] - __uint_as_float(h0 << 16), p[0][1] - __uint_as_float(h0 & 0xFFFF0000u));
        const uint32_t l1 = pack_bf16x2(p[1][0] - __uint_as_float(h1 << 16), p[1][1] - __uint_as_float(h1 & 0xFFFF0000u));
        // acc += P V: 16 tiles of 8 dims, two per transposed 4-matrix load
        const int vr = 16 * warp + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
        for (int dt2 = 0; dt2 < 8; ++dt2) {
            uint32_t b[4];
            ldsm_x4_trans(vb + walk_off(vr, 16 * dt2 + 8 * (lane >> 4)), b);
            mma_rows8(acc[2 * dt2], h0, h1, b[0], b[1]);
            mma_rows8(acc[2 * dt2], l0, l1, b[0], b[1]);
            mma_rows8(acc[2 * dt2 + 1], h0, h1, b[2], b[3]);
            mma_rows8(acc[2 * dt2 + 1], l0, l1, b[2], b[3]);
        }
        __syncthreads();  // every warp is done with this stage
        if (tid == 0 && ok && c + kWalkStages < ce) issue(c + kWalkStages);
    }
    if (!ok) {
        // a copy did not land in time: let the copies still in flight land
        // (bounded), leave no partial result (the combine kernel would read
        // garbage: the error word is set)
        if (tid == 0)
            for (int i = 0; i < kWalkStages; ++i) tc::mbar_wait(bar + i, 0, 100000000ull), tc::mbar_wait(bar + i, 1, 100000000ull);
        return;
    }
    // merge the four warps: the quad's sum of l, then (m, l, acc) through
    // shared memory (over the stages, no longer read)
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    float* sml = reinterpret_cast<float*>(sm);                 // [4 warps][8 rows][2]
    float* sacc = sml + 4 * 8 * 2;                             // [4 warps][8 rows][128]
    if (t == 0) {
        sml[(warp * 8 + gq) * 2] = m;
        sml[(warp * 8 + gq) * 2 + 1] = l;
    }
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
        *reinterpret_cast<float2*>(sacc + (warp * 8 + gq) * kAttnD + 8 * dt + 2 * t) = make_float2(acc[dt][0], acc[dt][1]);
    __syncthreads();
    const size_t part = ((size_t)s * a.Hkv + g) * attn_chunks(a.Tmax, cpw * kWalkTc) + wk;
    float* wacc = a.ws + part * R * kAttnD;
    float* wml = a.ws + (size_t)a.S * a.Hkv * attn_chunks(a.Tmax, cpw * kWalkTc) * R * kAttnD + part * R * 2;
    for (int r = 0; r < R; ++r) {
        float M = -1e30f;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sml[(w * 8 + r) * 2]);
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = ex2_approx(sml[(w * 8 + r) * 2] - M);
            o = fmaf(f, sacc[(w * 8 + r) * kAttnD + tid], o);
            L = fmaf(f, sml[(w * 8 + r) * 2 + 1], L);
        }
        wacc[r * kAttnD + tid] = o;
        if (tid == 0) *reinterpret_cast<float2*>(wml + 2 * r) = make_float2(M, L);
    }
}

// Chunks per walker for bf16 caches: enough walkers that sessions x kv heads
// x walkers fill two CTAs an SM of the 152-SM GB300 (a function of the sizes
// alone, like the workspace query that depends on it).
int attn_walk_chunks(int S, int Hkv, int Tmax) {
    const long nchunks = (Tmax + kWalkTc - 1) / kWalkTc;
    const long pairs = (long)S * Hkv;
    const long walkers = pairs >= 2 * 152 ? 1 : (2 * 152 + pairs - 1) / pairs;
    return (int)((nchunks + walkers - 1) / walkers);
}

cudaError_t make_cache_map(const void* cache, const AttnArgs& a, CUtensorMap* map) {
    tc::EncodeTiledFn enc = tc::encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)kAttnD, (cuuint64_t)a.S * a.Hkv * a.Tmax};
    const cuuint64_t strides[1] = {(cuuint64_t)kAttnD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kWalkTc};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_walk(const AttnArgs& a, cudaStream_t st) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(attn_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWalkSmem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CUtensorMap tmk, tmv;
    e = make_cache_map(a.k_cache, a, &tmk);
    if (e == cudaSuccess) e = make_cache_map(a.v_cache, a, &tmv);
    if (e != cudaSuccess) return e;
    const int cpw = a.tc / kWalkTc;
    const int nwalk = attn_chunks(a.Tmax, a.tc);
    return launch_pdl(attn_walk_kernel, dim3(nwalk, a.Hkv, a.S), dim3(kWalkThreads), kWalkSmem, st, a, tmk, tmv, cpw);
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
    // bf16: the tensor-core walkers; fp32: register sets for up to 2, 5 (the
    // Nemotron-H layers) or 8 query heads per kv head
    cudaError_t e = attn_use_walk(a.S, a.Hkv, a.Tmax, sizeof(TA) == 2) ? launch_walk(a, st)
                    : R <= 2        ? launch_split<TA, 2>(a, st)
                    : R <= 5        ? launch_split<TA, 5>(a, st)
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
