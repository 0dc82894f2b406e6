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
// Launched with programmatic dependent launch:
//  - bf16 caches: attn_walk_kernel alone, on the tensor cores. One CTA
//    ("walker") per (walker, kv head, session) takes a run of 64-position
//    chunks, brought into shared memory by 2-D TMA copies through a 3-stage
//    ring; its four warps keep their own online softmax over 16
//    positions of every chunk, with the scores (query heads x positions) and
//    the weighted values (query heads x dims) as mma.sync products. The
//    walkers of one (session, kv head) form a thread-block cluster and merge
//    their results through distributed shared memory:
//        M = max_w m_w, out = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w.
//  - fp32 caches: two kernels.
//    1. attn_split_kernel, on the CUDA cores. One CTA per (chunk of up to 64
//       positions, kv head, session; shorter chunks where there would be too
//       few CTAs to fill the GPU). Two bulk copies (the TMA engine) bring the
//       chunk's cached keys and values into shared memory; then scores (8
//       lanes per position, 16 dims a lane, the R heads' dot products reduced
//       over the 8 lanes, q held in fp32 registers), the chunk's softmax
//       statistics in the log2 domain (m = max, l = sum of 2^(a - m)) and
//       acc = sum_t 2^(a_t - m) v_t (16 threads per value row, 8 dims each,
//       all R heads at once), written as the chunk's partial result.
//    2. attn_combine_kernel: per (kv head, session), merges the chunks'
//       partial results with the same formula.
// The run holding position len[s] takes the new key and value from the
// inputs instead of the cache, and writes them into the cache there (no other
// CTA reads that slot).
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

// bf16 caches go to the tensor-core walkers, whose 2-D copies address the
// caches' rows (S x Hkv x Tmax of them) with 32-bit coordinates.
bool attn_use_walk(int S, int Hkv, int Tmax, bool bf16) {
    return bf16 && (long long)S * Hkv * Tmax < (1LL << 31) - 64;
}

// Positions per chunk of the split kernel: the most a CTA holds, halved (down
// to 32) while the grid would have fewer than two CTAs per SM of the 152-SM
// GB300, so that a short cache of few sessions still spreads over the GPU. A
// function of the sizes alone: the workspace query needs no device.
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

// ---------------------------------------------------------------------------
// bf16 caches on the tensor cores. A CTA ("walker") takes a run of
// consecutive 64-position chunks of one (session, kv head); a ring of 2-D TMA
// copies (128-byte swizzle) keeps the next chunks' keys and values in flight
// while it computes. Each of its four warps takes 16 positions of every chunk
// and keeps its own online softmax, so the warps meet only at the chunk
// boundary where a stage is refilled:
//     scores  S^T (16 positions x 8 heads, R real) = K . Q^T     mma m16n8k16
//     P = 2^(S log2e scale - m), m the running max per head, l += sum P
//     acc^T (128 dims x 8 heads) += V^T . P^T   (P as bf16 hi + lo: two MMAs)
// Positions are the products' M (or K) side and the R <= 8 heads their N
// side, so no MMA works on rows of zeros. The scores' accumulator fragments
// become the B operand of the second product by an in-register transpose of
// each 8 x 8 block (movmatrix). At the end the four warps' (m, l, acc) merge
// into the walker's own in shared memory. The W walkers of
// one (session, kv head) form one thread-block cluster: walker w owns query
// heads w, w + W, ...; every walker stores its (m, l, acc) of each head into
// the owner's shared memory (distributed shared memory), and after one
// cluster barrier each owner merges what it received and writes out, so one
// launch computes the whole decode position.
constexpr int kWalkTc = 64;                   // positions per chunk
constexpr int kWalkStages = 3;
constexpr int kWalkThreads = 128;
constexpr int kWalkMaxW = 16;                 // walkers per cluster, at most
constexpr uint32_t kWalkBox = kWalkTc * 128;  // one box: 64 rows x 64 dims of bf16 (8 KiB)
constexpr uint32_t kWalkStage = 4 * kWalkBox; // K (2 boxes) + V (2 boxes)
// After the ring: the slots an owner receives, [head / W][walker], each a
// walker's acc (128 floats relative to its max) then (max, sum); then the
// ring's barriers.
constexpr int kWalkSlots = kAttnMaxR + kWalkMaxW - 1;  // ceil(R / W) W, at most
constexpr uint32_t kWalkSlotF = kAttnD + 2;
constexpr uint32_t kWalkRecv = kWalkStages * kWalkStage;
constexpr uint32_t kWalkBar = kWalkRecv + kWalkSlots * kWalkSlotF * 4;
constexpr uint32_t kWalkSmem = kWalkBar + kWalkStages * 8 + 1024;  // + barriers, + slack to align to 1024
static_assert(2 * (kWalkSmem + 1024) <= 228 * 1024, "two CTAs an SM");
// The four warps' merge, over the first stage (no longer read): their
// (m, l) and acc.
constexpr uint32_t kWalkMl = 0;                                  // float [4][8][2]
constexpr uint32_t kWalkAcc = kWalkMl + 4 * 8 * 2 * 4;           // float [4][8][128]
static_assert(kWalkAcc + 4 * 8 * kAttnD * 4 <= kWalkStage, "the warps' merge fits in one stage");
static_assert(kWalkThreads == kAttnD, "one thread per dim in the merge");

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
// d += A B, m16n8k16, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The warp's 8 x 8 matrix of 16-bit elements (lane l holding row l / 4,
// columns 2 (l % 4) and + 1), transposed, in the same layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// grid (W, Hkv, S), a cluster of W walkers per (session, kv head) when W > 1;
// walker w takes chunks [w cpw, (w + 1) cpw) of those holding positions
// 0 .. len. Two CTAs an SM.
__global__ void __launch_bounds__(kWalkThreads, 2)
    attn_walk_kernel(AttnArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     int cpw) {
    extern __shared__ uint8_t walk_smem_raw[];
    uint8_t* sm = walk_smem_raw + ((1024u - (tc::smem_u32(walk_smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kWalkBar);  // one per stage: its copies landed
    const int W = gridDim.x, wk = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, t = lane & 3;  // fragment row and lane in its quad
    const int R = a.Hq / a.Hkv;
    constexpr int RB = kAttnD * 2;  // bytes of one cached row

    if (W > 1) tc::cluster_arrive_relaxed();  // waited on before the first remote store: every walker has started
    const int row0 = (s * a.Hkv + g) * a.Tmax;  // tensor row of position 0
    const int cb = wk * cpw;
    pdl_wait();  // the inputs and the caches may come from the previous kernel
    pdl_trigger();
    const int len = a.lens[s] + a.len_add;
    const bool bad = len < 0 || len >= a.Tmax;  // the same for the whole cluster
    const int nch = bad ? 0 : len / kWalkTc + 1;  // chunks holding positions 0 .. len
    const int ce = min(cb + cpw, nch);           // empty past this session's positions

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
    // Q^T as the B operand (k = dims, n = query head gq of this kv head;
    // heads past R zero): per 16-dim K-step two bf16 pairs
    uint32_t qb[8][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.q) +
                                                                 (size_t)s * a.q_ss + (size_t)(g * R + min(gq, R - 1)) * kAttnD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qb[kk][0] = gq < R ? __ldg(qrow + 8 * kk + t) : 0u;
            qb[kk][1] = gq < R ? __ldg(qrow + 8 * kk + 4 + t) : 0u;
        }
    }
    const float sl2 = a.scale * kLog2e;
    const bool h0ok = 2 * t < R, h1ok = 2 * t + 1 < R;  // this lane's heads 2t, 2t + 1
    // per head 2t and 2t + 1: running max (finite: a fully masked head stays
    // harmless), this lane's part of the sum, and acc^T (dims 16 dt + gq and
    // + 8)
    float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;
    float acc[8][4];
#pragma unroll
    for (int dt = 0; dt < 8; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[dt][e] = 0.f;
    __syncthreads();  // the barriers are initialised

    bool ok = true;  // the same in every thread: the end-of-chunk barrier votes on it
    for (int c = cb; c < ce; ++c) {
        const int st = (c - cb) % kWalkStages;
        const uint32_t phase = ((c - cb) / kWalkStages) & 1;
        uint8_t* sK = sm + st * kWalkStage;
        uint8_t* sV = sK + 2 * kWalkBox;
        bool landed = tc::mbar_wait(bar + st, phase);
        if (!landed) atomicOr(a.err, ERR_MBAR_TIMEOUT_LOAD);
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
        // S^T of this warp's positions 16 warp .. + 15: the A operand from K
        // (lanes 8j .. 8j + 7 address 8x8 piece j: positions + 8 (j & 1),
        // dims + 8 (j >> 1)), two accumulation chains over the 8 K-steps
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int kr = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), kc = 8 * (lane >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                uint32_t ka[4], kn[4];
                ldsm_x4(kb + walk_off(kr, 16 * kk + kc), ka);
                ldsm_x4(kb + walk_off(kr, 16 * kk + 16 + kc), kn);
                mma16816(sa, ka, qb[kk][0], qb[kk][1]);
                mma16816(sb, kn, qb[kk + 1][0], qb[kk + 1][1]);
            }
        }
        // online softmax per head over these 16 positions (-inf past len):
        // this lane holds positions gq and gq + 8 of heads 2t and 2t + 1
        const int pos = c * kWalkTc + 16 * warp + gq;
        const bool p0ok = pos <= len, p1ok = pos + 8 <= len;
        const float v00 = (p0ok && h0ok) ? (sa[0] + sb[0]) * sl2 : -INFINITY;
        const float v01 = (p0ok && h1ok) ? (sa[1] + sb[1]) * sl2 : -INFINITY;
        const float v10 = (p1ok && h0ok) ? (sa[2] + sb[2]) * sl2 : -INFINITY;
        const float v11 = (p1ok && h1ok) ? (sa[3] + sb[3]) * sl2 : -INFINITY;
        float mx0 = fmaxf(v00, v10), mx1 = fmaxf(v01, v11);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float c0 = ex2_approx(m0 - mn0), c1 = ex2_approx(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float p00 = ex2_approx(v00 - mn0), p01 = ex2_approx(v01 - mn1);  // 0 for -inf
        const float p10 = ex2_approx(v10 - mn0), p11 = ex2_approx(v11 - mn1);
        l0 = fmaf(l0, c0, p00 + p10);
        l1 = fmaf(l1, c1, p01 + p11);
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            acc[dt][0] *= c0;
            acc[dt][1] *= c1;
            acc[dt][2] *= c0;
            acc[dt][3] *= c1;
        }
        // P^T as the B operand (k = positions, n = head gq): bf16 hi + lo
        // (p = hi + lo to ~2^-16), each 8x8 block of the accumulator layout
        // transposed
        const uint32_t ha = pack_bf16x2(p00, p01), hb = pack_bf16x2(p10, p11);
        const uint32_t la = pack_bf16x2(p00 - __uint_as_float(ha << 16), p01 - __uint_as_float(ha & 0xFFFF0000u));
        const uint32_t lb = pack_bf16x2(p10 - __uint_as_float(hb << 16), p11 - __uint_as_float(hb & 0xFFFF0000u));
        const uint32_t bh0 = movmatrix_t(ha), bh1 = movmatrix_t(hb);
        const uint32_t bl0 = movmatrix_t(la), bl1 = movmatrix_t(lb);
        // acc^T += V^T P^T: the A operand V^T by transposed loads (piece j:
        // positions + 8 (j >> 1), dims + 8 (j & 1)), 8 tiles of 16 dims
        {
            const int vr = 16 * warp + (lane & 7) + 8 * (lane >> 4), vc = 8 * ((lane >> 3) & 1);
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                uint32_t va[4];
                ldsm_x4_trans(vb + walk_off(vr, 16 * dt + vc), va);
                mma16816(acc[dt], va, bh0, bh1);
                mma16816(acc[dt], va, bl0, bl1);
            }
        }
        ok = __syncthreads_and(landed) != 0;  // every warp is done with this stage
        if (!ok) break;
        if (tid == 0 && c + kWalkStages < ce) issue(c + kWalkStages);
    }
    if (!ok) {
        // a copy did not land in time: let the copies still in flight land
        // (bounded) and contribute nothing (the error word is set)
        if (tid == 0)
            for (int i = 0; i < kWalkStages; ++i)
                tc::mbar_wait(bar + i, 0, 100000000ull), tc::mbar_wait(bar + i, 1, 100000000ull);
        m0 = m1 = -1e30f;
        l0 = l1 = 0.f;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[dt][e] = 0.f;
    }
    __syncthreads();  // the stages are free for the merge
    // the four warps: each head's sum over the warp's 8 lanes of it, then
    // (m, l, acc) through shared memory
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* sml = reinterpret_cast<float*>(sm + kWalkMl);
    float* sacc = reinterpret_cast<float*>(sm + kWalkAcc);
    float* recv = reinterpret_cast<float*>(sm + kWalkRecv);
    if (gq == 0) {
        *reinterpret_cast<float2*>(sml + (warp * 8 + 2 * t) * 2) = make_float2(m0, l0);
        *reinterpret_cast<float2*>(sml + (warp * 8 + 2 * t + 1) * 2) = make_float2(m1, l1);
    }
    {
        float* a0 = sacc + (warp * 8 + 2 * t) * kAttnD + gq;  // head 2t, dim gq
        float* a1 = a0 + kAttnD;                              // head 2t + 1
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            a0[16 * dt] = acc[dt][0];
            a1[16 * dt] = acc[dt][1];
            a0[16 * dt + 8] = acc[dt][2];
            a1[16 * dt + 8] = acc[dt][3];
        }
    }
    __syncthreads();
    if (W > 1) tc::cluster_wait();  // every walker of the cluster has started: its shared memory is there
    // this walker's (max, sum, acc) per query head, acc relative to its max
    // (a walker without positions: max -1e30, sum 0, acc 0), to the head's
    // owner: slot (r / W) W + wk of walker r % W
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
        if (W == 1) {
            const float v = L > 0.f ? o / L : 0.f;  // a refused length (or a failed copy): zeros
            reinterpret_cast<uint16_t*>(a.out)[(size_t)s * a.out_ss + (size_t)(g * R + r) * kAttnD + tid] =
                float_to_bf16_bits(v);
        } else {
            const uint32_t slot = tc::smem_u32(recv + ((r / W) * W + wk) * kWalkSlotF);
            const uint32_t owner = (uint32_t)(r % W);
            tc::st_cluster_f32(tc::cluster_map(slot + 4u * tid, owner), o);
            if (tid == 0) tc::st_cluster_f32x2(tc::cluster_map(slot + 4u * kAttnD, owner), make_float2(M, L));
        }
    }
    if (bad && wk == 0 && g == 0 && tid == 0) atomicOr(a.err, ERR_ATTN_LENGTH);
    if (W == 1) return;
    tc::cluster_arrive();  // the stores into the owners' slots are visible ...
    tc::cluster_wait();    // ... once every walker has made them
    // out for the heads this walker owns: M = max_w m_w,
    // out = sum_w 2^(m_w - M) acc_w / sum_w 2^(m_w - M) l_w
    for (int r = wk; r < R; r += W) {
        const float* sl = recv + (r / W) * W * kWalkSlotF;
        float M = -1e30f;
        for (int w = 0; w < W; ++w) M = fmaxf(M, sl[w * kWalkSlotF + kAttnD]);
        float o = 0.f, L = 0.f;
        for (int w = 0; w < W; ++w) {
            const float f = ex2_approx(sl[w * kWalkSlotF + kAttnD] - M);
            o = fmaf(f, sl[w * kWalkSlotF + tid], o);
            L = fmaf(f, sl[w * kWalkSlotF + kAttnD + 1], L);
        }
        const float v = L > 0.f ? o / L : 0.f;  // a refused length (or a failed copy): zeros
        reinterpret_cast<uint16_t*>(a.out)[(size_t)s * a.out_ss + (size_t)(g * R + r) * kAttnD + tid] =
            float_to_bf16_bits(v);
    }
}

// Walkers per (session, kv head), a power of two, and 64-position chunks per
// walker. The walkers double while the grid stays within two CTAs an SM of
// the 152-SM GB300, every walker still gets a chunk, and the device runs one
// cluster per (session, kv head) at once (`clusters[k]`: clusters of 2^k
// walkers the device holds together, 0 where it runs none).
struct WalkPlan {
    int W, cpw;
};
WalkPlan walk_plan(int S, int Hkv, int Tmax, const int (&clusters)[5]) {
    const long nchunks = (Tmax + kWalkTc - 1) / kWalkTc;
    const long pairs = (long)S * Hkv;
    int W = 1, k = 0;
    while (k + 1 < 5 && pairs * 2 * W <= 2 * 152 && 2 * W <= nchunks && pairs <= clusters[k + 1]) W *= 2, ++k;
    WalkPlan p;
    p.W = W;
    p.cpw = (int)((nchunks + W - 1) / W);
    return p;
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

// Per device, once: the kernel's shared-memory and cluster-size attributes,
// and how many clusters of 2, 4, 8 and 16 walkers the device holds at once.
cudaError_t walk_setup(const int (**clusters)[5]) {
    static int configured_device = -1;
    static int cached[5];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(attn_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWalkSmem);
        if (e != cudaSuccess) return e;
        const bool wide = cudaFuncSetAttribute(attn_walk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                          cudaSuccess;
        cached[0] = 1 << 30;
        for (int k = 1; k < 5; ++k) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1u << k, 1, 1);
            cfg.blockDim = dim3(kWalkThreads);
            cfg.dynamicSmemBytes = kWalkSmem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1u << k;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if ((k == 4 && !wide) || cudaOccupancyMaxActiveClusters(&n, attn_walk_kernel, &cfg) != cudaSuccess) n = 0;
            cached[k] = n;
        }
        (void)cudaGetLastError();  // a refused query leaves no sticky error
        configured_device = dev;
    }
    *clusters = &cached;
    return cudaSuccess;
}

cudaError_t launch_walk(const AttnArgs& a, cudaStream_t st) {
    const int (*clusters)[5] = nullptr;
    cudaError_t e = walk_setup(&clusters);
    if (e != cudaSuccess) return e;
    CUtensorMap tmk, tmv;
    e = make_cache_map(a.k_cache, a, &tmk);
    if (e == cudaSuccess) e = make_cache_map(a.v_cache, a, &tmv);
    if (e != cudaSuccess) return e;
    const WalkPlan p = walk_plan(a.S, a.Hkv, a.Tmax, *clusters);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.W, a.Hkv, a.S);
    cfg.blockDim = dim3(kWalkThreads);
    cfg.dynamicSmemBytes = kWalkSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.W;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.W > 1 ? 2 : 1;
    const int cpw = p.cpw;
    return cudaLaunchKernelEx(&cfg, attn_walk_kernel, a, tmk, tmv, cpw);
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

// fp32 caches (and bf16 caches past the walkers' 32-bit row coordinates): the
// split kernel over chunks, then the combine kernel
template <typename TA>
cudaError_t launch_split_combine(const AttnArgs& a, cudaStream_t st) {
    const int R = a.Hq / a.Hkv;
    cudaError_t e = R <= 2   ? launch_split<TA, 2>(a, st)
                    : R <= 5 ? launch_split<TA, 5>(a, st)
                             : launch_split<TA, 8>(a, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_combine_kernel<TA>, dim3(a.Hkv, a.S), dim3(R * (kAttnD / 2)), 0, st, a);
}

}  // namespace

size_t attn_workspace_bytes(int S, int Hq, int Hkv, int Tmax, bool bf16) {
    if (S <= 0 || Hq <= 0 || Hkv <= 0 || Tmax <= 0 || Hq % Hkv) return 0;
    if (attn_use_walk(S, Hkv, Tmax, bf16)) return 0;  // the walkers merge in shared memory
    const int tc = attn_chunk_len(S, Hkv, Tmax, bf16);
    const size_t parts = (size_t)S * Hkv * attn_chunks(Tmax, tc) * (Hq / Hkv);
    return parts * (kAttnD + 2) * sizeof(float);
}

cudaError_t launch_attn_decode(const AttnArgs& a0, cudaStream_t st) {
    if (a0.S == 0) return cudaSuccess;
    if (attn_use_walk(a0.S, a0.Hkv, a0.Tmax, a0.bf16)) return launch_walk(a0, st);
    AttnArgs a = a0;
    a.tc = attn_chunk_len(a.S, a.Hkv, a.Tmax, a.bf16);
    return a.bf16 ? launch_split_combine<bf16_t>(a, st) : launch_split_combine<float>(a, st);
}

}  // namespace m2
