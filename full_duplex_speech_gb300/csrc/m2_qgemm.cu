// 4-bit group-64 affine-quantized linear layer for many rows of x (a
// prefill of T positions, many sessions at once): y = x W^T (+ residual) as
// a tensor-core GEMM. The weight format is that of m2_qlinear.cu (MLX's
// affine group quantization, the VoiceChat checkpoint's 4-bit mixer
// projections: group_size 64, bits 4): W[o][i] = scale[o][i/64] q + bias[o][i/64].
//
// One CTA computes a tile of 128 rows of x by 64 outputs, one 64-input group
// at a time:
//   A = x[rows][group]          bf16, by TMA (128-byte swizzle)
//   B = (128 + q)[outputs][group] as bf16 (exact), decoded by the CTA's
//       threads into the same layout, plus one row of ones (so that the
//       product also gives sum_i x_i over the group) and zero rows up to 80
//   D_g = A B^T                 tcgen05.mma, fp32 in tensor memory (4 K-steps)
// and, while the next group's products run, every thread takes its row of
// D_g out of tensor memory and accumulates in fp32
//   y += scale * D_g[o] + (bias - 128 scale) * D_g[ones]
// which is the decode kernel's arithmetic (exact bf16 products, fp32 sums,
// the group's scale and bias applied once per output), summed in a different
// order. The x tiles run two groups ahead in three buffers, the weights'
// fields and scales three groups ahead in registers; two buffers of B and D
// alternate between groups.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kGmThreads = 256;
constexpr int kGmRows = 128;       // rows of x per tile (the MMA's M, one per TMEM lane)
constexpr int kGmOut = 64;         // outputs per tile
constexpr int kGmN = 80;           // MMA N: 64 outputs, the ones row, 15 zero rows
constexpr int kGroup = 64;         // inputs per quantization group (one K panel of 128 B)
constexpr uint32_t kATile = kGmRows * 128;  // 16 KB
constexpr uint32_t kBTile = kGmN * 128;     // 10 KB
constexpr uint32_t kColD1 = 128;            // TMEM columns of the second D buffer
constexpr uint32_t kTmemCols = 256;

constexpr int kAStages = 3;  // x tiles in flight: groups g .. g + 2
struct GmSmem {
    static constexpr uint32_t kA = 0;                      // kAStages x A tile (1024-byte aligned)
    static constexpr uint32_t kB = kAStages * kATile;      // 2 x B tile
    static constexpr uint32_t kS = kB + 2 * kBTile;        // 2 x float2 (scale, bias - 128 scale) [64]
    static constexpr uint32_t kBar = kS + 2 * kGmOut * 8;  // xbar[3], mbar[2], end
    static constexpr uint32_t kTmem = kBar + 6 * 8;
    static constexpr uint32_t kFlag = kTmem + 4;
    // + slack to align the base to 1024; at least 80 KB, so that at most two
    // CTAs share an SM and their TMEM allocations (256 columns each) fit
    static constexpr uint32_t kBytes = (kFlag + 4 + 1024) > 80 * 1024 ? (kFlag + 4 + 1024) : 80 * 1024;
};

// The bf16 pair (128 + q_{2j}, 128 + q_{2j+1}) of the inputs 2j, 2j+1 of a
// 32-bit word of eight 4-bit fields (the first input lowest).
__device__ __forceinline__ uint32_t nat_pair(uint32_t w, int j) {
    const uint32_t lo = (w >> (8 * j)) & 0xFu;
    const uint32_t hi = (j < 2 ? (w << (12 - 8 * j)) : (w >> (8 * j - 12))) & 0xF0000u;
    return lo | hi | 0x43004300u;
}

template <bool RES>
__global__ void __launch_bounds__(kGmThreads) qgemm_kernel(QLinearArgs a, const __grid_constant__ CUtensorMap tmx) {
    using L = GmSmem;
    extern __shared__ uint8_t gm_raw[];
    uint8_t* sm = gm_raw + ((1024u - (tc::smem_u32(gm_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int o0 = blockIdx.x * kGmOut, t0 = blockIdx.y * kGmRows;
    const int in = a.in, ngroups = in / kGroup;
    float2* sS = reinterpret_cast<float2*>(sm + L::kS);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(sm + L::kBar);  // x tile landed, by A buffer
    uint64_t* mbar = xbar + kAStages;                             // products done, by D buffer
    uint64_t* endbar = mbar + 2;                                  // every product done (abort path)
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::kTmem);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(sm + L::kFlag);

    if (tid == 0) {
        for (int i = 0; i < kAStages + 3; ++i) tc::mbar_init(xbar + i, 1);
        tc::fence_mbar_init();
        *sFlag = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(sTmem, kTmemCols);
        tc::tmem_relinquish();
    }
    // the constant rows of both B tiles: the ones row (64) and zero rows 65..79
    for (int e = tid; e < 2 * (kGmN - kGmOut) * 8; e += kGmThreads) {
        const int buf = e / ((kGmN - kGmOut) * 8), r = kGmOut + (e / 8) % (kGmN - kGmOut), c = e % 8;
        const uint32_t v = r == kGmOut ? 0x3F803F80u : 0u;  // bf16 1.0 pairs
        *reinterpret_cast<uint4*>(sm + L::kB + buf * kBTile + tc::sw128_off(r, c * 8, kGmN)) = make_uint4(v, v, v, v);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *sTmem;

    // A bounded wait; the first that runs out stops the CTA's work.
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (*sFlag) return false;
        if (tc::mbar_wait(bar, parity)) return true;
        atomicOr(a.err, ERR_MBAR_TIMEOUT_LOAD);
        *sFlag = 1;
        return false;
    };

    // decode work of this thread: weight row dr (0..63), inputs 16 dq .. 16 dq + 15 of a group
    const int dr = tid >> 2, dq = tid & 3;
    const bool drow_live = o0 + dr < a.out;
    const uint2* wrow = reinterpret_cast<const uint2*>(a.wq + (size_t)(drow_live ? o0 + dr : 0) * (uint32_t)(in / 8));
    // epilogue work: row 32 (warp % 4) + lane of the tile, outputs 32 (warp / 4) .. + 31
    const int eq = warp & 3, eh = warp >> 2;
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;

    pdl_wait();  // x (and the residual) may come from the previous kernel
    // x tile of group gx into its A buffer (thread 0); the buffer was last read
    // by group gx - 3's products, complete before this is called
    auto issue_x = [&](int gx) {
        if (gx < ngroups && !*sFlag) {
            uint64_t* bar = xbar + gx % kAStages;
            tc::mbar_arrive_expect_tx(bar, kATile);
            tc::tma_load_2d(sm + L::kA + (gx % kAStages) * kATile, &tmx, gx * kGroup, t0, bar);
        }
    };
    if (tid == 0) {
        issue_x(0);
        issue_x(1);
        issue_x(2);
    }
    // this thread's weight fields (and, for tid < 64, its output's scale and
    // bias) of groups g, g + 1, g + 2, rotated each group
    // (pinned loads: issued where they stand, three groups before their use)
    auto load_w = [&](int gw) -> uint2 {
        return (gw < ngroups && drow_live) ? ldg_pinned_u2(wrow + (size_t)gw * 4 + dq) : make_uint2(0u, 0u);
    };
    const bool srow_live = tid < kGmOut && o0 + tid < a.out;
    const size_t srow = (size_t)(srow_live ? o0 + tid : 0) * ngroups;
    auto load_s = [&](int gs) -> uint32_t {
        return (gs < ngroups && srow_live)
                   ? (uint32_t)ldg_pinned_u16(a.scales + srow + gs) | ((uint32_t)ldg_pinned_u16(a.biases + srow + gs) << 16)
                   : 0u;
    };
    uint2 w0 = load_w(0), w1 = load_w(1), w2 = load_w(2);
    uint32_t s0 = load_s(0), s1 = load_s(1), s2 = load_s(2);

    const uint32_t sbase = tc::smem_u32(sm);
    const uint32_t idesc = tc::idesc_bf16(kGmRows, kGmN, 0, 0);
    for (int g = 0; g <= ngroups; ++g) {
        const int p = g & 1;
        if (g < ngroups && !*sFlag) {
            // the weights of group g -> B[p] rows 0..63 (zeros past the last output);
            // B[p] was last read by group g - 2's products, done (waited for in
            // every thread's epilogue of that group)
            const uint32_t ws[2] = {w0.x, w0.y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 v;
                v.x = nat_pair(ws[h], 0);
                v.y = nat_pair(ws[h], 1);
                v.z = nat_pair(ws[h], 2);
                v.w = nat_pair(ws[h], 3);
                if (!drow_live) v = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + L::kB + p * kBTile + tc::sw128_off(dr, dq * 16 + h * 8, kGmN)) = v;
            }
            // the group's scale and bias - 128 scale of each output
            if (tid < kGmOut) {
                const float sc = bf16_bits_to_float(s0 & 0xFFFFu), bi = bf16_bits_to_float(s0 >> 16);
                sS[p * kGmOut + tid] = make_float2(sc, bi - 128.f * sc);
            }
            tc::fence_proxy_async_smem();
            w0 = w1;
            w1 = w2;
            w2 = load_w(g + 3);
            s0 = s1;
            s1 = s2;
            s2 = load_s(g + 3);
        }
        tc::tc_fence_before();
        __syncthreads();  // B[p], S[p] written; every epilogue of group g - 2 finished
        tc::tc_fence_after();
        if (g < ngroups && tid == 0 && !*sFlag) {
            const int ab = g % kAStages;
            if (wait_ok(xbar + ab, (g / kAStages) & 1)) {
                tc::tc_fence_after();
                const uint64_t ad = tc::sdesc(sbase + L::kA + ab * kATile, 0, 1024, 2);
                const uint64_t bd = tc::sdesc(sbase + L::kB + p * kBTile, 0, 1024, 2);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tm + (p ? kColD1 : 0u), ad + 2 * ks, bd + 2 * ks, idesc, ks > 0 ? 1u : 0u);
                tc::mma_commit(mbar + p);
            }
        }
        if (g > 0) {
            // epilogue of group g - 1: D row -> fp32 accumulators
            const int pp = (g - 1) & 1;
            if (wait_ok(mbar + pp, ((g - 1) >> 1) & 1)) {
                tc::tc_fence_after();
                // group g - 1's products are done: its A buffer takes group g + 2
                if (tid == 0) issue_x(g + 2);
                const uint32_t ta = tm + ((uint32_t)(eq * 32) << 16) + (pp ? kColD1 : 0u);
                float d0[16], d1[16], dx[8];
                tc::tmem_ld16(ta + eh * 32, d0);
                tc::tmem_ld16(ta + eh * 32 + 16, d1);
                tc::tmem_ld8(ta + kGmOut, dx);  // column 64: sum of x over the group
                tc::tmem_wait_ld();
                const float2* sc = sS + pp * kGmOut + eh * 32;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 c0 = sc[j], c1 = sc[16 + j];
                    acc[j] = fmaf(c0.x, d0[j], fmaf(c0.y, dx[0], acc[j]));
                    acc[16 + j] = fmaf(c1.x, d1[j], fmaf(c1.y, dx[0], acc[16 + j]));
                }
            }
            tc::tc_fence_before();
            __syncthreads();  // S[pp] and D[pp] read by all before group g + 1 refills them
            tc::tc_fence_after();
        }
    }

    // the tile of y: row t, outputs o0 + 32 eh + j, plus the residual, rounded once
    const int t = t0 + eq * 32 + lane;
    if (!*sFlag && t < a.rows) {
        const int ob = o0 + eh * 32;
        uint16_t* yrow = reinterpret_cast<uint16_t*>(a.y) + (size_t)t * a.out;
        const uint16_t* rrow = reinterpret_cast<const uint16_t*>(a.residual) + (size_t)t * a.out;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (ob + j < a.out) {
                const float res = RES ? bf16_bits_to_float(rrow[ob + j]) : 0.f;
                yrow[ob + j] = float_to_bf16_bits(acc[j] + res);
            }
        }
    }
    pdl_trigger();
    if (*sFlag && tid == 0) {
        // A wait gave up. Every product issued must be done, and the x copies
        // in flight must land, before the tensor memory is freed and the CTA
        // exits (all waits bounded).
        tc::mma_commit(endbar);
        tc::mbar_wait(endbar, 0, 100000000ull);
        for (int i = 0; i < kAStages; ++i) {
            tc::mbar_wait(xbar + i, 0, 100000000ull);
            tc::mbar_wait(xbar + i, 1, 100000000ull);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, kTmemCols);
}

// x viewed as a 2-D tensor [rows][in] (innermost last; rows x_stride
// elements apart); a box is the [128 rows x 64 inputs] of one tile and group,
// 128-byte swizzled; rows past the last read as zero.
cudaError_t make_gm_x_map(const QLinearArgs& a, CUtensorMap* map) {
    tc::EncodeTiledFn enc = tc::encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)a.in, (cuuint64_t)a.rows};
    const cuuint64_t strides[1] = {(cuuint64_t)a.x_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGroup, (cuuint32_t)kGmRows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool RES>
cudaError_t launch_gm(const QLinearArgs& a, cudaStream_t st) {
    CUtensorMap tmx;
    memset(&tmx, 0, sizeof(tmx));
    cudaError_t e = make_gm_x_map(a, &tmx);
    if (e != cudaSuccess) return e;
    static int configured_device = -1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(qgemm_kernel<RES>, cudaFuncAttributeMaxDynamicSharedMemorySize, GmSmem::kBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const dim3 grid((unsigned)((a.out + kGmOut - 1) / kGmOut), (unsigned)((a.rows + kGmRows - 1) / kGmRows));
    return launch_pdl(qgemm_kernel<RES>, grid, dim3(kGmThreads), GmSmem::kBytes, st, a, tmx);
}

}  // namespace

cudaError_t launch_qgemm(const QLinearArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    return a.residual ? launch_gm<true>(a, st) : launch_gm<false>(a, st);
}

}  // namespace m2
