// Chunked (SSD) scan of the Mamba2 mixer core: full-history recompute and
// prefill. Two kernels per call, on the caller's stream:
//
//  1. scan_bc_kernel  — causal conv + SiLU of the B and C channels (shared by
//     the H/G heads of a group), written once per (sequence, chunk, group) as
//     ready-to-copy tensor-core operand tiles: B~ as a bf16 hi + lo pair
//     (B~ = hi + lo to ~2^-16), C~ as bf16. Rows past the end of the sequence
//     and state columns past N are zero.
//  2. scan_ssd_kernel — one CTA per (sequence, head) walks the chunks in order
//     with the fp32 state h [N x P] resident in tensor memory. Per chunk of L
//     frames with in-chunk cumulative log-decay S_i = sum_{s<=i} dt_s A:
//        G       = C~ B~^T                                   (tcgen05, bf16)
//        Y_off   = C~ h_prev^T, scaled by exp(S_i) later     (tcgen05, bf16)
//        h       = exp(S_last) h + B~^T (w o x~),  w_j = exp(S_last-S_j) dt_j
//                  as three bf16 products hi*hi + hi*lo + lo*hi (fp32-grade)
//        M_ij    = G_ij exp(S_i - S_j) dt_j  for j <= i, else 0
//        y       = M x~ + exp(S_i) Y_off + D x~              (tcgen05, bf16)
//     The conv + SiLU of the head's own x channels, softplus(dt) and the
//     cumulative sums run on the CUDA cores between the tensor-core phases.
//     Each CTA also writes its share of the final conv tail (the last K-1
//     pre-conv frames).
//
// The chunked form is the state-space-duality (SSD) evaluation of the Mamba-2
// recurrence (Dao & Gu 2024): the intra-chunk part is a masked quadratic form,
// the carried state enters through C~ h_prev.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kTR = 128;                       // tile rows: the maximum chunk length
constexpr int kNP = 128;                       // state dimension padded to the MMA M extent
constexpr uint32_t kTileBytes = kTR * kNP * 2;  // one bf16 operand tile, 32 KiB
constexpr uint32_t kPanel = kTR * 128;          // one 64-column panel of a tile, 16 KiB

// Frames used by sequence b: its entry of the lengths array clamped to
// [0, T], or T. Strides always use T.
__device__ __forceinline__ int seq_len(const ScanArgs& a, int b) {
    return a.lens ? min(max(__ldg(a.lens + b), 0), a.T) : a.T;
}

// ----------------------------------------------------------------- kernel 1
// This kernel lets the SSD kernel launch as soon as every CTA here has passed its
// griddepcontrol.wait: SSD CTAs then start at once on SMs without a CTA of
// this kernel, and on each other SM as soon as its CTA here exits. (An SSD
// CTA cannot share an SM with these CTAs: three of its nine warps, at 160
// registers, nearly fill one sub-partition's register file.) Two rows per
// thread keep each CTA short.
constexpr int kBcThreads = 256;
constexpr int kBcRows = 2;                                   // rows per thread
constexpr int kBcCtaRows = (kBcThreads / 32) * kBcRows;      // rows per CTA of one (chunk, group)
constexpr int kBcParts = kTR / kBcCtaRows;                   // CTAs per (chunk, group)
static_assert(kBcParts * kBcCtaRows == kTR, "a chunk's rows split evenly over its CTAs");

// conv + SiLU of one B/C value from its four pre-conv frames, oldest first
__device__ __forceinline__ float bc_conv_silu(float4 w, float bias, float f0, float f1, float f2, float f3) {
    float u = bias;
    u = fmaf(w.x, f0, u);
    u = fmaf(w.y, f1, u);
    u = fmaf(w.z, f2, u);
    u = fmaf(w.w, f3, u);
    return silu_fast(u);
}

// Stores row `row` of 8 channels [n0, n0+8) of the (B or C) operand tiles of
// one (sequence, chunk, group): B~ as bf16 hi + lo, C~ as bf16 hi; zeros when
// the row is not live (past the sequence end, or channels past N).
__device__ __forceinline__ void bc_store_row(uint8_t* tiles, int row, int n0, int which, bool live,
                                             const float (&out)[8]) {
    uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
    if (live) {
        // each 32-bit word: two channels rounded to bf16 (nearest even) with one
        // paired conversion, then their residuals the same way
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hw[j]) : "f"(out[2 * j + 1]), "f"(out[2 * j]));
            const float r0 = out[2 * j] - __uint_as_float(hw[j] << 16);
            const float r1 = out[2 * j + 1] - __uint_as_float(hw[j] & 0xFFFF0000u);
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lw[j]) : "f"(r1), "f"(r0));
        }
        hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    const uint32_t off = tc::sw128_off(row, n0, kTR);
    if (which == 0) {
        *reinterpret_cast<uint4*>(tiles + off) = hi;
        *reinterpret_cast<uint4*>(tiles + kTileBytes + off) = lo;
    } else {
        *reinterpret_cast<uint4*>(tiles + 2 * kTileBytes + off) = hi;
    }
}

template <typename TA>
__global__ void __launch_bounds__(kBcThreads) scan_bc_kernel(ScanArgs a, int nchunks) {
    // the conv weights and bias of the CTA's 32 columns of 8 channels, read
    // from global memory by its first warp only: the 24 CTAs of a group and
    // the 8 warps of each would otherwise ask L2 for the same lines at once
    __shared__ float4 sW[32][10];
    const Shape& s = a.s;
    const int c = blockIdx.x / kBcParts, part = blockIdx.x % kBcParts, g = blockIdx.y, b = blockIdx.z;
    const int T = a.T, Q = a.chunk;
    const int c0 = c * Q;
    const long HP = s.HP(), GN = s.GN(), CH = s.CH();
    uint8_t* tiles = reinterpret_cast<uint8_t*>(a.ws) + (((size_t)b * nchunks + c) * s.G + g) * 3 * kTileBytes;

    // 32 columns of 8 channels (16 for B, 16 for C) x (threads / 32) groups of kBcRows rows.
    const int cc = threadIdx.x & 31, rs = threadIdx.x >> 5;
    const int which = cc >> 4;  // 0: B, 1: C
    const int n0 = (cc & 15) * 8;
    const int r0 = part * kBcCtaRows + rs * kBcRows;
    const bool real = n0 < s.N;
    const long ch0 = HP + which * GN + (long)g * s.N + n0;  // conv channel of n0
    const void* src = which ? a.C : a.B;
    pdl_wait();     // B, C and the lengths may come from the previous kernel
    pdl_trigger();  // the SSD kernel may launch: its early reads are of data written before this kernel
    const int L = min(Q, seq_len(a, b) - c0);  // rows of this chunk in the sequence
    if (L <= 0) return;                        // past the sequence end: no tile is read

    // pre-conv rows r0-3 .. r0+kBcRows-1, and (first warp) the weights and
    // bias: every load is issued before any use, so all are in flight
    // together. A row outside the sequence (and not in the initial tail) reads
    // the chunk's first row, a valid address, and counts as zero.
    Act8<TA> v[kBcRows + 3];
    bool have[kBcRows + 3];
    float4 w[8], b0 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = b0;
    if (rs == 0 && real) {
#pragma unroll
        for (int j = 0; j < 8; ++j) sW[cc][j] = ldg_pinned_f4(reinterpret_cast<const float4*>(a.conv_w) + ch0 + j);
        sW[cc][8] = ldg_pinned_f4(reinterpret_cast<const float4*>(a.conv_b + ch0));
        sW[cc][9] = ldg_pinned_f4(reinterpret_cast<const float4*>(a.conv_b + ch0) + 1);
    }
    const bool any = real && r0 < L;
    if (any) {
#pragma unroll
        for (int k = 0; k < kBcRows + 3; ++k) {
            const int t = c0 + r0 - 3 + k;
            const bool in_seq = t >= 0 && t < c0 + L;
            const bool from_tail = t < 0 && a.init_conv != nullptr;
            have[k] = in_seq || from_tail;
            const void* base = from_tail ? a.init_conv : src;
            const size_t elem = from_tail ? ((size_t)b * (s.K - 1) + (s.K - 1 + t)) * CH + ch0
                                          : ((size_t)b * T + (in_seq ? t : c0)) * a.fbc + (size_t)g * s.N + n0;
            v[k].load_pinned(base, elem);
        }
    }
    __syncthreads();
    if (any) {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = sW[cc][j];
        b0 = sW[cc][8];
        b1 = sW[cc][9];
    }
#pragma unroll
    for (int r = 0; r < kBcRows; ++r) {
        float out[8];
        if (any) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float f[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) f[k] = have[r + k] ? v[r + k].get(j) : 0.f;
                out[j] = bc_conv_silu(w[j], j < 4 ? (&b0.x)[j] : (&b1.x)[j - 4], f[0], f[1], f[2], f[3]);
            }
        }
        bc_store_row(tiles, r0 + r, n0, which, real && r0 + r < L, out);
    }
}

// The final conv tail of 8 channels [c, c+8) of sequence b: frames Tb-3..Tb-1
// (Tb = its length), taken from the initial tail (or zeros) where Tb < 3.
// Every source slot is read before any is written, so final_conv may alias
// init_conv.
template <typename TA>
__device__ void write_tail(const ScanArgs& a, int b, long c) {
    const Shape& s = a.s;
    const long CH = s.CH(), HP = s.HP(), GN = s.GN();
    const int T = a.T, Tb = seq_len(a, b);
    // source of each frame chosen first, so the three loads go out together
    Act8<TA> vals[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int t = Tb - 3 + k;
        const void* base;
        size_t elem;
        if (t >= 0) {
            base = c < HP ? a.x : (c < HP + GN ? a.B : a.C);
            elem = c < HP ? ((size_t)b * T + t) * a.fx + c
                          : ((size_t)b * T + t) * a.fbc + (c < HP + GN ? c - HP : c - HP - GN);
        } else {
            base = a.init_conv;
            elem = ((size_t)b * 3 + (3 + t)) * CH + c;
        }
        if (base)
            vals[k].load_rw(base, elem);
        else
            memset(&vals[k], 0, sizeof(vals[k]));
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) vals[k].store(a.final_conv, ((size_t)b * 3 + k) * CH + c);
}

// ----------------------------------------------------------------- kernel 2
// kComputeWarps compute warps and one control warp whose elected thread
// issues every TMA copy and tcgen05 instruction. The issuing thread stalls
// while the tensor cores work through its MMAs, so it is kept out of the
// CUDA-core phases. Compute warp w works on TMEM lane quarter w % 4 (rows
// 32(w % 4) .. +31 of a chunk, or of the state's n) and on column part w / 4:
// the P columns, in units of 8, are split over the parts as evenly as they
// go, and the 128 columns j of the decay mask go to the parts with fewer P
// columns (to every part alike when the units split evenly).
constexpr int kComputeWarps = 16;
constexpr int kParts = kComputeWarps / 4;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kSsdThreads = kComputeThreads + 32;
constexpr int kCtrl = kComputeThreads;  // the control thread
constexpr int kDtPart = kParts - 1;     // the column part that also computes dt and S
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRawRows = kTR + 3;  // pre-conv rows of one chunk plus the 3-frame halo
static_assert(kComputeWarps == 8 || kComputeWarps == 16, "two or four column parts");
// TMEM columns
// M, the masked G in bf16, is the A operand of Y_diag straight from TMEM:
// row i on lane i, two columns j per 32-bit TMEM column. A part writes the M
// of its mask columns over the first half of the G columns it has just read
// (SsdParts::m_col). Y_off is double-buffered by chunk parity: a chunk's
// Y_off MMAs run while the previous chunk's y is still being read.
constexpr uint32_t kColG = 0, kColState = 128, kColYd = 224, kColYo0 = 320, kColYo1 = 416, kTmemCols = 512;
static_assert(kColYo1 + 80 <= kTmemCols, "accumulators of up to 80 columns fit the allocation");

// How the column work of one head is split over the column parts.
template <int P>
struct SsdParts {
    static constexpr int U = P / 8;                          // 8-column units of P
    static constexpr int kBase = U / kParts, kRem = U % kParts;
    static constexpr int kMaxUnits = kBase + (kRem ? 1 : 0);
    // parts below kRem carry one unit more; the mask then goes to the others
    static constexpr int kMaskParts = kRem ? kParts - kRem : kParts;
    static constexpr int kMaskSteps = 8 / kMaskParts;        // K-steps of 16 mask columns per mask part
    static_assert(kMaskSteps * kMaskParts == 8, "the mask's 8 K-steps split evenly");
    __device__ static int units(int part) { return kBase + (part < kRem ? 1 : 0); }
    __device__ static int first_unit(int part) { return part * kBase + min(part, kRem); }
    __device__ static int mask_steps(int part) { return (kRem && part < kRem) ? 0 : kMaskSteps; }
    __device__ static int first_mask_step(int part) { return (kRem ? part - kRem : part) * kMaskSteps; }
    // TMEM column (from kColG) of the M of K-step ks: the part that owns ks
    // writes 8 columns per step from the start of the G columns it read
    __host__ __device__ static constexpr uint32_t m_col(int ks) {
        return (uint32_t)((ks / kMaskSteps) * kMaskSteps * 16 + (ks % kMaskSteps) * 8);
    }
};

template <typename TA, int P>
struct SsdSmem {
    static constexpr uint32_t kC = 0;                     // C~ hi           (K-major SW128)
    static constexpr uint32_t kBh = kTileBytes;           // B~ hi           (K-major / MN-major SW128)
    static constexpr uint32_t kBl = 2 * kTileBytes;       // B~ lo           (SW128)
    static constexpr uint32_t kPT = kTR * P * 2;          // one [128 x P] bf16 interleaved tile
    static constexpr uint32_t kX = 3 * kTileBytes;        // x~ hi           (MN-major interleave, K = j)
    static constexpr uint32_t kWh = kX + kPT;             // (w o x~) hi
    static constexpr uint32_t kWl = kWh + kPT;            // (w o x~) lo
    static constexpr uint32_t kH = kWl + kPT;             // h hi            (MN-major interleave, K = n)
    static constexpr uint32_t kRaw = kH + kPT;            // pre-conv x rows [kRawRows][P + pad] (act dtype)
    // bf16 rows carry 8 channels of padding (the next head's, or zeros past the
    // last): an odd number of 16-byte units per row, so the 32 rows a warp reads
    // at once fall on distinct bank groups
    static constexpr int kRawPad = sizeof(TA) == 2 ? 8 : 0;
    static constexpr uint32_t kRowBytes = (P + kRawPad) * sizeof(TA);
    static constexpr uint32_t kRowData = P * sizeof(TA);  // the head's own channels
    static constexpr uint32_t kS = kRaw + kRawRows * kRowBytes;  // float S[128]
    static constexpr uint32_t kDt = kS + 512;             // float dt[128]
    static constexpr uint32_t kTj = kDt + 512;            // float exp(S_j1 - S_j) dt_j, j1 = j | 7 [128]
    static constexpr uint32_t kWsum = kTj + 512;          // float warp sums[4]
    static constexpr uint32_t kCw = kWsum + 64;           // float conv_w[4][P] (tap-major)
    static constexpr uint32_t kCb = kCw + P * 16;         // float conv_b[P]
    static constexpr uint32_t kBar = (kCb + P * 4 + 15) / 16 * 16;  // 9 mbarriers
    static constexpr uint32_t kTmem = kBar + 72;          // TMEM base address
    static constexpr uint32_t kFlag = kTmem + 4;          // abort flag
    static constexpr uint32_t kBytes = kFlag + 4 + 1024;  // + slack to align the base to 1024
};

// Two fp32 -> packed bf16x2 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack2(v.x, v.y); }

// 2^x on the special-function unit (ex2.approx: relative error ~2^-22, ftz).
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// 1/x on the special-function unit (rcp.approx, ftz: 0 for |x| above 2^126).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Paired fp32 arithmetic: one instruction for two lanes of values, each
// rounded exactly as its scalar counterpart.
__device__ __forceinline__ uint64_t f2_bits(float2 v) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
    return r;
}
__device__ __forceinline__ float2 f2_of(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return f2_of(r);
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_of(r);
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_of(r);
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_of(r);
}
__device__ __forceinline__ float2 f2_splat(float v) { return make_float2(v, v); }
// a bf16 pair (low half first) as two fp32 values
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// SiLU(u) = u / (1 + 2^(-u log2 e)) on a pair, with the special-function
// unit's exponential and reciprocal. Where the divisor is huge (u below about
// -87) the reciprocal is 0, and so is the result (exactly: below 1e-36).
__device__ __forceinline__ float2 silu2(float2 u) {
    const float2 t = f2_mul(u, f2_splat(-kLog2e));
    const float2 d = f2_add(make_float2(ex2_approx(t.x), ex2_approx(t.y)), f2_splat(1.f));
    return f2_mul(u, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Eight consecutive activations of one staged row as four fp32 pairs.
template <typename TA>
__device__ __forceinline__ void load8_pairs(const uint8_t* p, float2 (&v)[4]) {
    if constexpr (sizeof(TA) == 2) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        v[0] = bf2_to_f2(r.x);
        v[1] = bf2_to_f2(r.y);
        v[2] = bf2_to_f2(r.z);
        v[3] = bf2_to_f2(r.w);
    } else {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        v[0] = make_float2(a.x, a.y);
        v[1] = make_float2(a.z, a.w);
        v[2] = make_float2(b.x, b.y);
        v[3] = make_float2(b.z, b.w);
    }
}

// Barrier among the compute warps only (the control warp never joins).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory"); }

// Stages the pre-conv x rows of chunk c (frames c0-3 .. c0+kTR-1) of this head
// into shared memory with one 3-D TMA box copy of [kRawRows frames x P
// channels]; frames outside [0, T) read as zero (the caller patches the three
// frames before the sequence from the initial conv tail, when there is one).
template <typename TA, int P>
__device__ __forceinline__ void stage_raw_x(const CUtensorMap* tmx, uint8_t* raw, uint64_t* bar, int b, int h,
                                            int c0) {
    using Lay = SsdSmem<TA, P>;
    tc::mbar_arrive_expect_tx(bar, (uint32_t)kRawRows * Lay::kRowBytes);
    tc::tma_load_3d(raw, tmx, h * P, c0 - 3, b, bar);
}

template <typename TA, int P>
// Seventeen warps put five on one SM sub-partition, whose register file then
// allows at most 96 registers a thread: the bound below (20 warps' worth) asks
// the compiler for that.
__global__ void __launch_bounds__(kComputeWarps == 16 ? 640 : kSsdThreads, 1) scan_ssd_kernel(ScanArgs a, int nchunks,
                                                                  const __grid_constant__ CUtensorMap tmx) {
    using L = SsdSmem<TA, P>;
    using Parts = SsdParts<P>;
    constexpr int NU = Parts::kMaxUnits;       // 8-column units of a part, at most
    constexpr int NK = Parts::kMaskSteps;      // mask K-steps of a mask part
    constexpr uint32_t LBO_I = (P / 8) * 128;  // K-group stride of the interleaved tiles
    extern __shared__ uint8_t smem_raw[];
    // offset from the shared array itself, so that the compiler keeps the shared address space
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);

    const Shape& s = a.s;
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / (s.H / s.G);
    const int T = a.T, Q = a.chunk;
    const long HP = s.HP();
    const int tid = threadIdx.x, row = tid & 127, part = tid >> 7, warp = tid >> 5, lane = tid & 31;
    const bool compute = tid < kComputeThreads;
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int nu = compute ? Parts::units(part) : 0, u0 = Parts::first_unit(part);

    float* sS = reinterpret_cast<float*>(sm + L::kS);
    float* sDt = reinterpret_cast<float*>(sm + L::kDt);
    float* sEb = reinterpret_cast<float*>(sm + L::kTj);
    float* sWsum = reinterpret_cast<float*>(sm + L::kWsum);
    float* sCw = reinterpret_cast<float*>(sm + L::kCw);
    float* sCb = reinterpret_cast<float*>(sm + L::kCb);
    uint8_t* sRaw = sm + L::kRaw;
    uint64_t* bar_a = reinterpret_cast<uint64_t*>(sm + L::kBar);  // C~ hi + B~ hi tiles landed
    uint64_t* bar_b = bar_a + 1;                                   // B~ lo tile landed
    uint64_t* bar_x = bar_a + 2;                                   // pre-conv x rows landed
    uint64_t* bar_g = bar_a + 3;                                   // G done
    uint64_t* bar_op0 = bar_a + 4;                                 // h_prev tile written (all compute threads)
    uint64_t* bar_y = bar_a + 5;                                   // every MMA of the chunk done
    uint64_t* bar_op1 = bar_a + 6;                                 // phase-1 operands written (all compute threads)
    uint64_t* bar_op2 = bar_a + 7;                                 // phase-2 operands written (all compute threads)
    uint64_t* bar_end = bar_a + 8;                                 // MMAs of an abandoned chunk done
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::kTmem);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(sm + L::kFlag);

    // Bounded wait that gives up at once after any earlier timeout in the CTA,
    // so a failure cannot turn into a hang; it records `code` when it runs out.
    auto wait_ok = [&](uint64_t* bar, uint32_t parity, unsigned code) -> bool {
        if (*sFlag) return false;
        if (tc::mbar_wait(bar, parity)) return true;
        atomicOr(a.err, code);
        *sFlag = 1;
        return false;
    };

    // setup that reads no input: barriers, TMEM
    if (tid == kCtrl) {
        for (int i = 0; i < 4; ++i) tc::mbar_init(bar_a + i, 1);
        tc::mbar_init(bar_op0, kComputeThreads);
        tc::mbar_init(bar_y, 1);
        tc::mbar_init(bar_op1, kComputeThreads);
        tc::mbar_init(bar_op2, kComputeThreads);
        tc::mbar_init(bar_end, 1);
        tc::fence_mbar_init();
        *sFlag = 0;
    }
    if (!compute) {
        tc::tmem_alloc(sTmem, kTmemCols);
        tc::tmem_relinquish();
    }
    // Every input read before the control thread's wait for the prologue's
    // tiles was written before the prologue kernel started: this launch
    // directly follows it, and may start early only once each prologue CTA has
    // passed its own wait for its predecessor.

    // this sequence's frames and chunks (the workspace is laid out for nchunks)
    const int Tb = seq_len(a, b);
    const int nchb = (Tb + Q - 1) / Q;
    // the first chunk's x rows (the barrier is the control thread's own; the
    // other threads wait on it only after the block sync)
    if (tid == kCtrl && nchb > 0) stage_raw_x<TA, P>(&tmx, sRaw, bar_x, b, h, 0);
    // The other global loads of the setup, issued before any is used so that
    // all are in flight together: this head's conv weights, its scalars, and
    // dt_raw of this thread's row of the first chunk (kept raw, hence no stall
    // before the block sync; from then on dt_raw is loaded one chunk ahead of
    // the dt phase that uses it, and kept raw until then, so that its latency
    // passes under the wait for the chunk's MMAs).
    static_assert(P <= kSsdThreads, "one conv weight row per thread");
    float4 cw = make_float4(0.f, 0.f, 0.f, 0.f);
    float cb = 0.f;
    if (tid < P) {
        cw = ldg_pinned_f4(reinterpret_cast<const float4*>(a.conv_w) + (long)h * P + tid);
        cb = ldg_pinned_f32(a.conv_b + (long)h * P + tid);
    }
    const float A_log_h = ldg_pinned_f32(a.A_log + h);
    const float Dh = ldg_pinned_f32(a.D + h);
    const float dtb = ldg_pinned_f32(a.dt_bias + h);
    const bool dt_part = compute && part == kDtPart;
    ActRaw<TA> dt_raw_bits = 0;
    if (dt_part && nchb > 0 && row < min(Q, Tb))
        dt_raw_bits = load_raw_pinned<TA>(a.dt_raw, ((size_t)b * T + row) * a.fdt + h);
    if (tid < P) {
        // tap-major, so that one 16-byte load gives a tap's weights of four channels
        sCw[0 * P + tid] = cw.x;
        sCw[1 * P + tid] = cw.y;
        sCw[2 * P + tid] = cw.z;
        sCw[3 * P + tid] = cw.w;
        sCb[tid] = cb;
    }
    const float A = -expf(A_log_h);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *sTmem;

    const uint32_t sbase = tc::smem_u32(sm);
    const uint8_t* ws = reinterpret_cast<const uint8_t*>(a.ws);
    auto tiles_of = [&](int c) { return ws + (((size_t)b * nchunks + c) * s.G + g) * 3 * kTileBytes; };

    if (!compute) {
        // ================================================================ control
        // The whole warp runs the loop (so that the descriptor arithmetic stays
        // warp-uniform); one elected lane issues every copy and MMA.
        if (nchb > 0) {
            const bool leader = tc::elect_one();
            pdl_wait();  // the operand tiles are the prologue kernel's output
            const uint8_t* src = tiles_of(0);
            if (leader) {
                tc::mbar_arrive_expect_tx(bar_a, 2 * kTileBytes);
                tc::bulk_g2s(sm + L::kBh, src, kTileBytes, bar_a);
                tc::bulk_g2s(sm + L::kC, src + 2 * kTileBytes, kTileBytes, bar_a);
                tc::mbar_arrive_expect_tx(bar_b, kTileBytes);
                tc::bulk_g2s(sm + L::kBl, src + kTileBytes, kTileBytes, bar_b);
            }
            __syncwarp();
            // Matrix descriptors of every operand at K-step 0; a K-step's
            // descriptor adds its byte offset / 16 to the start-address field.
            const uint64_t dCk = tc::sdesc(sbase + L::kC, 0, 1024, 2);    // C~, K-major (K = n)
            const uint64_t dBk = tc::sdesc(sbase + L::kBh, 0, 1024, 2);   // B~ hi, K-major (K = n)
            const uint64_t dBhm = tc::sdesc(sbase + L::kBh, kPanel, 1024, 2);  // B~ hi as B~^T, MN-major (K = j)
            const uint64_t dBlm = tc::sdesc(sbase + L::kBl, kPanel, 1024, 2);  // B~ lo as B~^T
            const uint64_t dH = tc::sdesc(sbase + L::kH, LBO_I, 128, 0);   // h_prev, MN-major interleave (K = n)
            const uint64_t dWh = tc::sdesc(sbase + L::kWh, LBO_I, 128, 0);  // (w o x~) hi (K = j)
            const uint64_t dWl = tc::sdesc(sbase + L::kWl, LBO_I, 128, 0);  // (w o x~) lo
            const uint64_t dX = tc::sdesc(sbase + L::kX, LBO_I, 128, 0);    // x~ hi (K = j)
            auto koff_k = [](int ks) { return (uint64_t)(((ks >> 2) * kPanel + (ks & 3) * 32) >> 4); };
            auto koff_m = [](int ks) { return (uint64_t)((ks * 2048) >> 4); };
            auto koff_i = [](int ks) { return (uint64_t)((ks * 2 * LBO_I) >> 4); };
            const uint32_t idG = tc::idesc_bf16(128, 128, 0, 0);
            const uint32_t idS = tc::idesc_bf16(128, P, 1, 1);
            const uint32_t idY = tc::idesc_bf16(128, P, 0, 1);
            for (int c = 0; c < nchb; ++c) {
                const int c0 = c * Q;
                const int ksteps = (min(Q, Tb - c0) + 15) / 16;
                const uint32_t par = c & 1;
                const bool has_next = c + 1 < nchb;
                // G = C~ B~^T as soon as the tiles are in: it needs nothing from the
                // compute warps, and its TMEM columns (which also held the previous
                // chunk's M) were last read by the previous chunk's Y_diag MMAs,
                // done before these tiles were fetched
                const bool okt = wait_ok(bar_a, par, ERR_MBAR_TIMEOUT_LOAD);
                if (okt) {
                    tc::tc_fence_after();
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + kColG, dCk + koff_k(ks), dBk + koff_k(ks), idG, ks > 0);
                        tc::mma_commit(bar_g);
                    }
                    __syncwarp();
                }
                // Y_off = C~ h_prev^T as soon as the h_prev tile is written: it runs
                // under the compute warps' conv (into the Y_off buffer of this
                // chunk's parity; the other one holds the previous chunk's, still
                // to be read)
                const bool ok0 = wait_ok(bar_op0, par, ERR_MBAR_TIMEOUT_MMA);
                tc::tc_fence_after();
                const uint32_t colYo = par ? kColYo1 : kColYo0;
                if (ok0 && okt) {
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_bf16(tm + colYo, dCk + koff_k(ks), dH + koff_i(ks), idY, ks > 0);
                    }
                    __syncwarp();
                }
                const bool ok1 = wait_ok(bar_op1, par, ERR_MBAR_TIMEOUT_MMA);
                tc::tc_fence_after();
                const bool okb = wait_ok(bar_b, par, ERR_MBAR_TIMEOUT_LOAD);
                if (ok0 && ok1 && okt && okb) {
                    // phase 1: state += B~^T (w o x~) as hi*hi + hi*lo + lo*hi. A
                    // fresh sequence's state is not in TMEM before its first chunk:
                    // that chunk's first product overwrites the accumulator.
                    const uint32_t acc0 = (c > 0 || a.init_ssm != nullptr) ? 1u : 0u;
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            if (ks < ksteps) {
                                tc::mma_bf16(tm + kColState, dBlm + koff_m(ks), dWh + koff_i(ks), idS,
                                             ks > 0 ? 1u : acc0);
                                tc::mma_bf16(tm + kColState, dBhm + koff_m(ks), dWh + koff_i(ks), idS, 1);
                                tc::mma_bf16(tm + kColState, dBhm + koff_m(ks), dWl + koff_i(ks), idS, 1);
                            }
                        }
                    }
                    __syncwarp();
                }
                // the staged rows are consumed: stage the next chunk's (needed only
                // at the next chunk's conv, so after this chunk's MMAs are queued)
                if (has_next && ok1 && leader) stage_raw_x<TA, P>(&tmx, sRaw, bar_x, b, h, c0 + Q);
                __syncwarp();
                if (wait_ok(bar_op2, par, ERR_MBAR_TIMEOUT_MMA)) {
                    tc::tc_fence_after();
                    // phase 2: Y_diag += M x~ (onto D x~, M from TMEM)
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            if (ks < ksteps)
                                tc::mma_bf16_tmem_a(tm + kColYd, tm + kColG + Parts::m_col(ks), dX + koff_i(ks), idY,
                                                    1);
                        tc::mma_commit(bar_y);
                    }
                    __syncwarp();
                }
                // every operand tile of this chunk is consumed: fetch the next chunk's
                if (wait_ok(bar_y, par, ERR_MBAR_TIMEOUT_MMA) && has_next) {
                    if (leader) {
                        const uint8_t* nsrc = tiles_of(c + 1);
                        tc::mbar_arrive_expect_tx(bar_a, 2 * kTileBytes);
                        tc::bulk_g2s(sm + L::kBh, nsrc, kTileBytes, bar_a);
                        tc::bulk_g2s(sm + L::kC, nsrc + 2 * kTileBytes, kTileBytes, bar_a);
                        tc::mbar_arrive_expect_tx(bar_b, kTileBytes);
                        tc::bulk_g2s(sm + L::kBl, nsrc + kTileBytes, kTileBytes, bar_b);
                    }
                    __syncwarp();
                }
            }
            if (*sFlag && leader) {
                // A wait gave up. Before the CTA frees TMEM and exits: every MMA
                // this lane issued must be done (the commit arrives on bar_end
                // once all of them have completed; some, such as Y_off and the
                // state terms, are covered by no other commit), and the copies
                // still in flight must land. Every wait here is bounded.
                tc::mma_commit(bar_end);
                tc::mbar_wait(bar_end, 0, 100000000ull);
                for (int i = 0; i < 3; ++i) {
                    tc::mbar_wait(bar_a + i, 0, 100000000ull);
                    tc::mbar_wait(bar_a + i, 1, 100000000ull);
                }
            }
        }
        __syncwarp();
        // Final conv tail (the last K-1 pre-conv frames), written by this warp
        // while the compute warps finish the last chunk's y. This CTA owns the
        // tail of its head's x channels: their initial frames are read only by
        // this CTA, in chunk 0, before the phase-1 handoff the loop above
        // waited for. The first head of each group also owns the group's B and
        // C channels, whose initial frames only the prologue kernel reads, and
        // that kernel has finished once griddepcontrol.wait returns. So
        // final_conv may alias init_conv.
        pdl_wait();
        const int R = s.H / s.G;
        const int nx = P / 8, nbc = (h % R == 0) ? 2 * s.N / 8 : 0;
        // (skipped if a wait gave up: chunk 0 may not have read the initial tail)
        const int nt = *sFlag ? 0 : nx + nbc;
        for (int v = lane; v < nt; v += 32) {
            long ch;
            if (v < nx)
                ch = (long)h * P + v * 8;
            else if (v - nx < s.N / 8)
                ch = HP + (long)g * s.N + (v - nx) * 8;
            else
                ch = HP + s.GN() + (long)g * s.N + (v - nx - s.N / 8) * 8;
            write_tail<TA>(a, b, ch);
        }
    } else {
        // ================================================================ compute
        // Initial state -> TMEM [n lanes][p columns]; rows n >= N stay zero.
        // Without one (a fresh sequence) the first chunk's state step takes the
        // old state as zero instead of reading TMEM, so nothing is stored here:
        // TMEM stores right after the allocation were measured to take ~1 us.
        // With no chunk at all the final state is read back from here.
        const bool state_in_tmem = a.init_ssm != nullptr || nchb == 0;
        if (state_in_tmem) {
            const int n = row;
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                if (k < nu) {
                    const int p0 = (u0 + k) * 8;
                    float v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        v[q] = (a.init_ssm && n < s.N)
                                   ? __ldg(a.init_ssm + (((size_t)b * s.H + h) * P + p0 + q) * s.N + n)
                                   : 0.f;
                    tc::tmem_st8(tm + lane_base + kColState + p0, v);
                }
            }
            tc::tmem_wait_st();
        }

        // dt = softplus(dt_raw + dt_bias), a = dt A, inclusive cumulative sum S over
        // a chunk of Lx rows, and the column factor of the decay mask,
        // Eb_j = exp(S_j1 - S_j) dt_j with j1 = j | 7 the last column of j's
        // 8-column block (0 past the chunk end, where dt_j = 0), all into shared
        // memory by the dt part. S does not increase, so Eb_j <= dt_j. Every
        // compute thread must call it (it holds barriers).
        auto dt_phase = [&](int Lx, float raw) {
            float v = 0.f, dt = 0.f;
            if (dt_part) {
                dt = row < Lx ? softplus_f32(raw + dtb) : 0.f;
                v = dt * A;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v += o;
                }
                if (lane == 31) sWsum[quarter] = v;
            }
            compute_sync();
            if (dt_part) {
                float add = 0.f;
                for (int w = 0; w < quarter; ++w) add += sWsum[w];
                const float S = v + add;
                const float S1 = __shfl_sync(0xffffffffu, S, lane | 7);  // same warp: 8 | 32
                sS[row] = S;
                sDt[row] = dt;
                sEb[row] = ex2_approx((S1 - S) * kLog2e) * dt;
            }
            compute_sync();
        };

        // y = (D x~ + M x~) + exp(S_i) Y_off for the chunk whose results sit in TMEM.
        // The TMEM loads are warp-collective (.sync.aligned): every lane issues
        // them; only the stores are predicated.
        auto y_epilogue = [&](int c0y, int Ly, float eSy, uint32_t colYo) {
            const bool live = row < Ly;
            const size_t ybase = (((size_t)b * T + c0y + row) * s.H + h) * P;
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                if (k < nu) {
                    const int p0 = (u0 + k) * 8;
                    float yd[8], yo[8];
                    tc::tmem_ld8(tm + lane_base + kColYd + p0, yd);
                    tc::tmem_ld8(tm + lane_base + colYo + p0, yo);
                    tc::tmem_wait_ld();
                    float2 out[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        out[m] = f2_fma(f2_splat(eSy), make_float2(yo[2 * m], yo[2 * m + 1]),
                                        make_float2(yd[2 * m], yd[2 * m + 1]));
                    if (live) {
                        if constexpr (sizeof(TA) == 2) {
                            *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.y) + ybase + p0) =
                                make_uint4(pack2(out[0]), pack2(out[1]), pack2(out[2]), pack2(out[3]));
                        } else {
                            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + ybase + p0);
                            dst[0] = make_float4(out[0].x, out[0].y, out[1].x, out[1].y);
                            dst[1] = make_float4(out[2].x, out[2].y, out[3].x, out[3].y);
                        }
                    }
                }
            }
        };

        if (nchb > 0) {
            dt_phase(min(Q, Tb), raw_to_f32<TA>(dt_raw_bits));
            dt_raw_bits = 0;
            if (dt_part && nchb > 1 && row < min(Q, Tb - Q))
                dt_raw_bits = load_raw_pinned<TA>(a.dt_raw, ((size_t)b * T + Q + row) * a.fdt + h);
        }

        // The chunk loop is skewed so that CUDA-core work overlaps the tensor
        // cores: the y epilogue of chunk c-1 and the D x~ preload run under
        // chunk c's phase-1 MMAs, the dt phase of chunk c+1 under its phase 2.
        float eS_prev = 0.f;
        int L_prev = 0, c0_prev = 0;
        for (int c = 0; c < nchb; ++c) {
            const int c0 = c * Q;
            const int Lc = min(Q, Tb - c0);
            const uint32_t par = c & 1;
            const bool has_next = c + 1 < nchb;
            const int Ln = has_next ? min(Q, Tb - c0 - Q) : 0;
            const int Lnn = c + 2 < nchb ? min(Q, Tb - c0 - 2 * Q) : 0;

            // 1. state: h_prev (bf16) into shared memory for Y_off, then
            //    h <- exp(S_last) h in TMEM (its dt phase ran one step earlier;
            //    the previous chunk's MMAs are done). A fresh sequence's first
            //    chunk has h_prev = 0 and leaves TMEM alone: the first state MMA
            //    overwrites the accumulator.
            const float Slast = sS[Lc - 1];
            {
                const float2 decay = f2_splat(__expf(Slast));
                const int n = row;
                const bool in_tmem = c > 0 || state_in_tmem;
                float v[NU][8];
                if (in_tmem) {
#pragma unroll
                    for (int k = 0; k < NU; ++k)
                        if (k < nu) tc::tmem_ld8(tm + lane_base + kColState + (u0 + k) * 8, v[k]);
                    tc::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < NU; ++k)
#pragma unroll
                        for (int q = 0; q < 8; ++q) v[k][q] = 0.f;
                }
#pragma unroll
                for (int k = 0; k < NU; ++k) {
                    if (k < nu) {
                        const int p0 = (u0 + k) * 8;
                        *reinterpret_cast<uint4*>(sm + L::kH + tc::mn_inter_off(p0, n, P)) =
                            make_uint4(pack2(v[k][0], v[k][1]), pack2(v[k][2], v[k][3]), pack2(v[k][4], v[k][5]),
                                       pack2(v[k][6], v[k][7]));
                        if (in_tmem) {
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float2 sc = f2_mul(make_float2(v[k][2 * m], v[k][2 * m + 1]), decay);
                                v[k][2 * m] = sc.x;
                                v[k][2 * m + 1] = sc.y;
                            }
                            tc::tmem_st8(tm + lane_base + kColState + p0, v[k]);
                        }
                    }
                }
                if (in_tmem) tc::tmem_wait_st();
            }
            // hand the h_prev tile (and the scaled state) to the control warp
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::mbar_arrive(bar_op0);

            // 2a. this chunk's staged x rows
            wait_ok(bar_x, par, ERR_MBAR_TIMEOUT_LOAD);
            if (c == 0 && a.init_conv) {
                // frames -3..-1 (zero-filled by the copy) come from the initial conv tail
                constexpr int V = L::kRowData / 16;
                for (int e = tid; e < 3 * V; e += kComputeThreads) {
                    const int r = e / V, q = e % V;
                    *reinterpret_cast<uint4*>(sRaw + (size_t)r * L::kRowBytes + q * 16) =
                        *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.init_conv) +
                                                        (((size_t)b * 3 + r) * s.CH() + (size_t)h * P) * sizeof(TA) +
                                                        q * 16);
                }
                compute_sync();
            }
            const float Si = sS[row];
            const float wi = row < Lc ? __expf(Slast - Si) * sDt[row] : 0.f;

            // 2. conv + SiLU of this part's x channels for row i (staged rows
            //    i..i+3), on channel pairs
            float2 xf[NU][4];
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                if (k < nu) {
                    const int p0 = (u0 + k) * 8;
                    float2 o[4];
                    if (row < Lc) {
                        const float4 b0 = *reinterpret_cast<const float4*>(sCb + p0);
                        const float4 b1 = *reinterpret_cast<const float4*>(sCb + p0 + 4);
                        float2 acc[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                         make_float2(b1.z, b1.w)};
#pragma unroll
                        for (int tap = 0; tap < 4; ++tap) {
                            float2 xv[4];
                            load8_pairs<TA>(sRaw + (size_t)(row + tap) * L::kRowBytes + p0 * sizeof(TA), xv);
                            const float4 w0 = *reinterpret_cast<const float4*>(sCw + tap * P + p0);
                            const float4 w1 = *reinterpret_cast<const float4*>(sCw + tap * P + p0 + 4);
                            acc[0] = f2_fma(make_float2(w0.x, w0.y), xv[0], acc[0]);
                            acc[1] = f2_fma(make_float2(w0.z, w0.w), xv[1], acc[1]);
                            acc[2] = f2_fma(make_float2(w1.x, w1.y), xv[2], acc[2]);
                            acc[3] = f2_fma(make_float2(w1.z, w1.w), xv[3], acc[3]);
                        }
#pragma unroll
                        for (int m = 0; m < 4; ++m) o[m] = silu2(acc[m]);
                    } else {
#pragma unroll
                        for (int m = 0; m < 4; ++m) o[m] = make_float2(0.f, 0.f);
                    }
                    uint32_t xh[4], wh[4], wl[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        xf[k][m] = o[m];
                        xh[m] = pack2(o[m]);
                        const float2 w = f2_mul(o[m], f2_splat(wi));
                        wh[m] = pack2(w);
                        wl[m] = pack2(f2_sub(w, bf2_to_f2(wh[m])));
                    }
                    const uint32_t off = tc::mn_inter_off(p0, row, P);
                    *reinterpret_cast<uint4*>(sm + L::kX + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
                    *reinterpret_cast<uint4*>(sm + L::kWh + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    *reinterpret_cast<uint4*>(sm + L::kWl + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            }

            // hand the phase-1 operands (x~ and w o x~ tiles) to the control warp
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::mbar_arrive(bar_op1);

            // 3. meanwhile: the previous chunk's y (this chunk's MMAs so far write
            //    G, the state and the other Y_off buffer), then this chunk's D x~
            //    preloaded into the Y_diag accumulator that phase 2 adds M x~ onto
            if (c > 0) y_epilogue(c0_prev, L_prev, eS_prev, par ? kColYo0 : kColYo1);
#pragma unroll
            for (int k = 0; k < NU; ++k) {
                if (k < nu) {
                    float dx[8];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float2 d = f2_mul(xf[k][m], f2_splat(Dh));
                        dx[2 * m] = d.x;
                        dx[2 * m + 1] = d.y;
                    }
                    tc::tmem_st8(tm + lane_base + kColYd + (u0 + k) * 8, dx);
                }
            }
            tc::tmem_wait_st();

            // 4. M = G o exp(S_i - S_j) dt_j (j <= i) -> bf16 into TMEM, the A
            //    operand of Y_diag (the state MMAs run meanwhile), by the parts
            //    that own mask columns, 16 columns j (one K-step) at a time. Each
            //    K-step is, for the whole warp (rows 32 quarter .. +31), either
            //    left of every row's diagonal block, holding some row's
            //    diagonal block, or right of every row's diagonal (zero).
            //    An 8-column block [j0, j1] wholly left of row i factors as
            //    exp(S_i - S_j1) * Eb_j, both factors <= 1 (S does not
            //    increase); the block holding the diagonal takes one exponential
            //    per entry.
            const int nks = Parts::mask_steps(part);
            if (nks > 0) {
                wait_ok(bar_g, par, ERR_MBAR_TIMEOUT_MMA);
                tc::tc_fence_after();
                const int fks = Parts::first_mask_step(part);
                const int i = row;
                const bool live = i < Lc;
                const int jd = i & ~7;  // this row's diagonal block
#pragma unroll
                for (int q = 0; q < NK; ++q) {
                    const int j0 = 16 * (fks + q);
                    float mv[8];
                    if (j0 >= 32 * quarter + 32) {
                        // right of every row's diagonal: zero
#pragma unroll
                        for (int e = 0; e < 8; ++e) mv[e] = 0.f;
                    } else {
                        float gv[16];
                        tc::tmem_ld16(tm + lane_base + kColG + j0, gv);
                        const bool left = j0 + 16 <= 32 * quarter;  // uniform across the warp
                        // this row's diagonal block, when it lies in this K-step
                        float dg[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) dg[e] = 0.f;
                        if (!left && live && jd >= j0 && jd < j0 + 16) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (jd + e <= i) dg[e] = ex2_approx((Si - sS[jd + e]) * kLog2e) * sDt[jd + e];
                        }
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e8 = 0; e8 < 16; e8 += 8) {
                            const int jb = j0 + e8;
                            // row factor of a block left of the diagonal (0 for dead rows)
                            const float ea = (live && jb < jd) ? ex2_approx((Si - sS[jb + 7]) * kLog2e) : 0.f;
                            const float4 c0v = *reinterpret_cast<const float4*>(sEb + jb);
                            const float4 c1v = *reinterpret_cast<const float4*>(sEb + jb + 4);
                            float2 f[4] = {make_float2(c0v.x, c0v.y), make_float2(c0v.z, c0v.w),
                                           make_float2(c1v.x, c1v.y), make_float2(c1v.z, c1v.w)};
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                f[m] = f2_mul(f[m], f2_splat(ea));
                                if (!left && jb == jd) f[m] = make_float2(dg[2 * m], dg[2 * m + 1]);
                                const float2 mm = f2_mul(make_float2(gv[e8 + 2 * m], gv[e8 + 2 * m + 1]), f[m]);
                                mv[e8 / 2 + m] = __uint_as_float(pack2(mm));
                            }
                        }
                    }
                    tc::tmem_st8(tm + lane_base + kColG + Parts::m_col(fks + q), mv);
                }
                tc::tmem_wait_st();
            }
            // hand the phase-2 operands (M and D x~ in TMEM) to the control warp
            tc::tc_fence_before();
            tc::mbar_arrive(bar_op2);

            // 5. meanwhile: the next chunk's dt phase (its first barrier orders this
            //    chunk's reads of S, dt and Eb before its writes; S_i is kept in a
            //    register)
            if (has_next) {
                dt_phase(Ln, raw_to_f32<TA>(dt_raw_bits));
                dt_raw_bits = 0;
                if (dt_part && row < Lnn)
                    dt_raw_bits = load_raw_pinned<TA>(a.dt_raw, ((size_t)b * T + c0 + 2 * Q + row) * a.fdt + h);
            }
            wait_ok(bar_y, par, ERR_MBAR_TIMEOUT_MMA);
            tc::tc_fence_after();
            eS_prev = __expf(Si);
            L_prev = Lc;
            c0_prev = c0;
        }
        // the last chunk's y
        compute_sync();
        if (!*sFlag && nchb > 0) y_epilogue(c0_prev, L_prev, eS_prev, ((nchb - 1) & 1) ? kColYo1 : kColYo0);
    }

    pdl_trigger();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const bool ok = !*sFlag;
    // final state: TMEM [n][p] -> final_ssm [b,h,p,n]
    if (ok && compute) {
        const int n = row;
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            if (k < nu) {
                const int p0 = (u0 + k) * 8;
                float v[8];
                tc::tmem_ld8(tm + lane_base + kColState + p0, v);
                tc::tmem_wait_ld();
                if (n < s.N) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        a.final_ssm[(((size_t)b * s.H + h) * P + p0 + q) * s.N + n] = v[q];
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (!compute) tc::tmem_dealloc(tm, kTmemCols);
}

// x viewed as a 3-D tensor [b][T][H*P] (innermost last; rows fx elements
// apart, which is H*P for a dense x and wider for x inside the rows of a
// projection output); a box is the
// [kRawRows x (P + pad)] pre-conv rows of one head for one chunk (the pad
// channels belong to the next head, or lie past the end and read as zero).
template <typename TA, int P>
cudaError_t make_x_map(const ScanArgs& a, CUtensorMap* map) {
    tc::EncodeTiledFn enc = tc::encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t HP = (cuuint64_t)a.s.H * P;
    const cuuint64_t dims[3] = {HP, (cuuint64_t)a.T, (cuuint64_t)a.batch};
    const cuuint64_t fx = (cuuint64_t)a.fx;
    const cuuint64_t strides[2] = {fx * sizeof(TA), fx * (cuuint64_t)a.T * sizeof(TA)};
    const cuuint32_t box[3] = {(cuuint32_t)(P + SsdSmem<TA, P>::kRawPad), (cuuint32_t)kRawRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = sizeof(TA) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = enc(map, dt, 3, const_cast<void*>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// after_prologue: the launch directly follows this call's prologue kernel on
// the stream. Only then may the SSD kernel start early (programmatic
// dependent launch): its reads before griddepcontrol.wait (x, dt_raw, the
// initial state, the weights) are of data written before the prologue began.
// Otherwise it is an ordinary launch.
template <typename TA, int P>
cudaError_t launch_ssd(const ScanArgs& a, int nchunks, bool after_prologue, cudaStream_t st) {
    CUtensorMap tmx;
    memset(&tmx, 0, sizeof(tmx));
    if (nchunks > 0) {
        cudaError_t me = make_x_map<TA, P>(a, &tmx);
        if (me != cudaSuccess) return me;
    }
    const int smem = SsdSmem<TA, P>::kBytes;
    // once per process and instantiation (kept out of graph captures after the first call)
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(scan_ssd_kernel<TA, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    if (after_prologue && nchunks > 0)
        return launch_pdl(scan_ssd_kernel<TA, P>, dim3(a.s.H, a.batch), dim3(kSsdThreads), smem, st, a, nchunks, tmx);
    scan_ssd_kernel<TA, P><<<dim3(a.s.H, a.batch), kSsdThreads, smem, st>>>(a, nchunks, tmx);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_bc_typed(const ScanArgs& a, cudaStream_t st) {
    const int nchunks = (a.T + a.chunk - 1) / a.chunk;
    if (nchunks == 0) return cudaSuccess;
    return launch_pdl(scan_bc_kernel<TA>, dim3(nchunks * kBcParts, a.s.G, a.batch), dim3(kBcThreads), 0, st, a, nchunks);
}

template <typename TA>
cudaError_t launch_chunks_typed(const ScanArgs& a, bool after_prologue, cudaStream_t st) {
    const int nchunks = (a.T + a.chunk - 1) / a.chunk;
    switch (a.s.P) {
        case 16: return launch_ssd<TA, 16>(a, nchunks, after_prologue, st);
        case 32: return launch_ssd<TA, 32>(a, nchunks, after_prologue, st);
        case 48: return launch_ssd<TA, 48>(a, nchunks, after_prologue, st);
        case 64: return launch_ssd<TA, 64>(a, nchunks, after_prologue, st);
        case 80: return launch_ssd<TA, 80>(a, nchunks, after_prologue, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t scan_workspace_bytes(const Shape& s, int batch, int T, int chunk) {
    if (chunk < 1 || batch <= 0 || T <= 0) return 0;
    const size_t nchunks = ((size_t)T + chunk - 1) / chunk;
    return (size_t)batch * nchunks * s.G * 3 * kTileBytes;
}

cudaError_t launch_scan_prepare(const ScanArgs& a, cudaStream_t st) {
    if (a.batch == 0) return cudaSuccess;
    return a.s.bf16 ? launch_bc_typed<bf16_t>(a, st) : launch_bc_typed<float>(a, st);
}

cudaError_t launch_scan_chunks(const ScanArgs& a, bool after_prologue, cudaStream_t st) {
    if (a.batch == 0) return cudaSuccess;
    return a.s.bf16 ? launch_chunks_typed<bf16_t>(a, after_prologue, st)
                    : launch_chunks_typed<float>(a, after_prologue, st);
}

}  // namespace m2
