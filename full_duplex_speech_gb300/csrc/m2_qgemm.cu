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
// and the epilogue warps take their rows of D_g out of tensor memory and
// accumulate in fp32
//   y += scale * D_g[o] + (bias - 128 scale) * D_g[ones]
// which is the decode kernel's arithmetic (exact bf16 products, fp32 sums,
// the group's scale and bias applied once per output), summed in a different
// order. Decode, products and epilogue run in warps of their own, on
// different groups at once, through rings of three stages.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kGmThreads = 288;    // warps 0-3: epilogue (one TMEM lane quarter each); 4-7: decode; 8: copies and products
constexpr int kGmRows = 128;       // rows of x per tile (the MMA's M, one per TMEM lane)
constexpr int kGmOut = 64;         // outputs per tile
constexpr int kGmN = 80;           // MMA N: 64 outputs, the ones row, 15 zero rows
constexpr int kGroup = 64;         // inputs per quantization group (one K panel of 128 B)
constexpr int kStages = 3;         // groups in flight: B tile, scales and accumulator of each
constexpr int kAStages = 3;        // x tiles in flight (copies run kAStages - 2 groups ahead of the products)
constexpr uint32_t kATile = kGmRows * 128;  // 16 KB
constexpr uint32_t kBTile = kGmN * 128;     // 10 KB
constexpr uint32_t kTmemCols = 256;         // kStages accumulators of kGmN columns

struct GmSmem {
    static constexpr uint32_t kA = 0;                             // kAStages x A tile (1024-byte aligned)
    static constexpr uint32_t kB = kAStages * kATile;             // kStages x B tile
    static constexpr uint32_t kS = kB + kStages * kBTile;         // kStages x float2 (scale, bias - 128 scale) [64]
    static constexpr uint32_t kBar = kS + kStages * kGmOut * 8;   // xfull [kAStages], bfull, dfull, empty [kStages], end
    static constexpr uint32_t kTmem = kBar + (kAStages + 3 * kStages + 1) * 8;
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

// Warp roles, handing groups over through rings of kStages buffers (stage
// s = g mod kStages for group g):
//   decode (warps 4-7): wait until the epilogue has released stage s, write
//     group g's weights into B[s] and its scales into S[s], arrive on bfull[s];
//   issue (warp 8, one thread): copy x of group g + kAStages - 2 into its A
//     buffer once the products that last read it are done; once bfull[s]
//     and the x tile of group g are complete, issue group g's four products
//     into accumulator s and commit them to dfull[s];
//   epilogue (warps 0-3, one row of the tile per thread): wait on dfull[s],
//     add the group into its 64 fp32 accumulators, arrive on empty[s].
template <bool RES>
__global__ void __launch_bounds__(kGmThreads) qgemm_kernel(QLinearArgs a, const __grid_constant__ CUtensorMap tmx) {
    using L = GmSmem;
    extern __shared__ uint8_t gm_raw[];
    uint8_t* sm = gm_raw + ((1024u - (tc::smem_u32(gm_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int o0 = blockIdx.x * kGmOut, t0 = blockIdx.y * kGmRows;
    const int in = a.in, ngroups = in / kGroup;
    float2* sS = reinterpret_cast<float2*>(sm + L::kS);
    uint64_t* xfull = reinterpret_cast<uint64_t*>(sm + L::kBar);  // x tile landed
    uint64_t* bfull = xfull + kAStages;                           // B tile and scales written (128 producers)
    uint64_t* dfull = bfull + kStages;                            // products done
    uint64_t* empty = dfull + kStages;                            // accumulator and scales read (128 epilogue threads)
    uint64_t* endbar = empty + kStages;                           // every product done (abort path)
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::kTmem);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(sm + L::kFlag);

    if (tid == 0) {
        for (int i = 0; i < kAStages; ++i) tc::mbar_init(xfull + i, 1);
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(bfull + i, 128);
            tc::mbar_init(dfull + i, 1);
            tc::mbar_init(empty + i, 128);
        }
        tc::mbar_init(endbar, 1);
        tc::fence_mbar_init();
        *sFlag = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(sTmem, kTmemCols);
        tc::tmem_relinquish();
    }
    // the constant rows of every B tile: the ones row (64) and zero rows 65..79
    for (int e = tid; e < kStages * (kGmN - kGmOut) * 8; e += kGmThreads) {
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

    pdl_wait();  // x (and the residual) may come from the previous kernel
    if (warp == 8) {
        // ============================================================ issue
        if (tid == 256) {
            constexpr int kLead = kAStages - 2;  // x of group g + kLead is copied before group g's products
            auto issue_x = [&](int gx) {
                uint64_t* bar = xfull + gx % kAStages;
                tc::mbar_arrive_expect_tx(bar, kATile);
                tc::tma_load_2d(sm + L::kA + (gx % kAStages) * kATile, &tmx, gx * kGroup, t0, bar);
            };
            for (int gx = 0; gx < kLead && gx < ngroups; ++gx) issue_x(gx);
            const uint32_t sbase = tc::smem_u32(sm);
            const uint32_t idesc = tc::idesc_bf16(kGmRows, kGmN, 0, 0);
            for (int g = 0; g < ngroups; ++g) {
                const int st = g % kStages;
                const uint32_t rnd = (uint32_t)(g / kStages);
                if (g + kLead < ngroups) {
                    // A of group g + kLead last served group g - 2, whose products
                    // were committed to dfull two groups ago
                    if (g + kLead >= kAStages && !wait_ok(dfull + (g - 2) % kStages, (uint32_t)((g - 2) / kStages) & 1))
                        break;
                    issue_x(g + kLead);
                }
                const int ab = g % kAStages;
                if (!wait_ok(bfull + st, rnd & 1) || !wait_ok(xfull + ab, (uint32_t)(g / kAStages) & 1)) break;
                tc::tc_fence_after();
                const uint64_t ad = tc::sdesc(sbase + L::kA + ab * kATile, 0, 1024, 2);
                const uint64_t bd = tc::sdesc(sbase + L::kB + st * kBTile, 0, 1024, 2);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tm + st * kGmN, ad + 2 * ks, bd + 2 * ks, idesc, ks > 0 ? 1u : 0u);
                tc::mma_commit(dfull + st);
            }
        }
    } else if (warp >= 4) {
        // ============================================================ decode
        const int pt = tid - 128;
        const int dr = pt >> 1, dh = pt & 1;  // weight row; inputs 32 dh .. 32 dh + 31 of a group
        const bool drow_live = o0 + dr < a.out;
        const uint4* wrow =
            reinterpret_cast<const uint4*>(a.wq + (size_t)(drow_live ? o0 + dr : 0) * (uint32_t)(in / 8));
        const bool srow_live = pt < kGmOut && o0 + pt < a.out;
        const size_t srow = (size_t)(srow_live ? o0 + pt : 0) * ngroups;
        // this thread's weight fields (and, for pt < 64, its output's scale and
        // bias) of groups g .. g + kStages - 1: pinned loads, issued where they stand
        auto load_w = [&](int gw) -> uint4 {
            return (gw < ngroups && drow_live) ? ldg_pinned_u4(wrow + (size_t)gw * 2 + dh) : make_uint4(0u, 0u, 0u, 0u);
        };
        auto load_s = [&](int gs) -> uint32_t {
            return (gs < ngroups && srow_live)
                       ? (uint32_t)ldg_pinned_u16(a.scales + srow + gs) |
                             ((uint32_t)ldg_pinned_u16(a.biases + srow + gs) << 16)
                       : 0u;
        };
        // the ring is indexed by the stage, so the loop runs kStages groups per
        // pass with every index fixed: a rotated ring would copy each load's
        // register one group after issuing it, waiting for it there
        uint4 wr[kStages];
        uint32_t sr[kStages];
#pragma unroll
        for (int k = 0; k < kStages; ++k) {
            wr[k] = load_w(k);
            sr[k] = load_s(k);
        }
        bool stop = false;
        for (int g0 = 0; g0 < ngroups && !stop; g0 += kStages) {
#pragma unroll
            for (int st = 0; st < kStages; ++st) {
                const int g = g0 + st;
                // stage st is free once the epilogue has finished group g - kStages
                // (its accumulator and scales read, the products that read B[st] done)
                if (g >= ngroups || stop ||
                    (g0 > 0 && !wait_ok(empty + st, ((uint32_t)(g0 / kStages) - 1) & 1))) {
                    stop = true;
                    continue;
                }
                // the weights of group g -> B[st] rows 0..63 (zeros past the last output)
                const uint32_t ws[4] = {wr[st].x, wr[st].y, wr[st].z, wr[st].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint4 v;
                    v.x = nat_pair(ws[k], 0);
                    v.y = nat_pair(ws[k], 1);
                    v.z = nat_pair(ws[k], 2);
                    v.w = nat_pair(ws[k], 3);
                    if (!drow_live) v = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sm + L::kB + st * kBTile + tc::sw128_off(dr, dh * 32 + k * 8, kGmN)) = v;
                }
                if (pt < kGmOut) {
                    const float sc = bf16_bits_to_float(sr[st] & 0xFFFFu), bi = bf16_bits_to_float(sr[st] >> 16);
                    sS[st * kGmOut + pt] = make_float2(sc, bi - 128.f * sc);
                }
                wr[st] = load_w(g + kStages);
                sr[st] = load_s(g + kStages);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(bfull + st);
            }
        }
    } else {
        // ============================================================ epilogue
        float acc[kGmOut];
#pragma unroll
        for (int j = 0; j < kGmOut; ++j) acc[j] = 0.f;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int g = 0; g < ngroups; ++g) {
            const int st = g % kStages;
            // bfull orders the decode warps' scales before these reads
            if (!wait_ok(bfull + st, (uint32_t)(g / kStages) & 1) || !wait_ok(dfull + st, (uint32_t)(g / kStages) & 1))
                break;
            tc::tc_fence_after();
            const uint32_t ta = tm + lane_base + st * kGmN;
            float dx[8];
            tc::tmem_ld8(ta + kGmOut, dx);  // column 64: sum of x over the group
            tc::tmem_wait_ld();
            const float2* sc = sS + st * kGmOut;
#pragma unroll
            for (int q = 0; q < kGmOut / 16; ++q) {
                float d[16];
                tc::tmem_ld16(ta + q * 16, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 c = sc[q * 16 + j];
                    acc[q * 16 + j] = fmaf(c.x, d[j], fmaf(c.y, dx[0], acc[q * 16 + j]));
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(empty + st);
        }
        // the tile of y: row t, outputs o0 .. o0 + 63, plus the residual, rounded once
        const int t = t0 + tid;
        if (!*sFlag && t < a.rows) {
            uint16_t* yrow = reinterpret_cast<uint16_t*>(a.y) + (size_t)t * a.out;
            const uint16_t* rrow = reinterpret_cast<const uint16_t*>(a.residual) + (size_t)t * a.out;
#pragma unroll
            for (int j = 0; j < kGmOut; ++j) {
                if (o0 + j < a.out) {
                    const float res = RES ? bf16_bits_to_float(rrow[o0 + j]) : 0.f;
                    yrow[o0 + j] = float_to_bf16_bits(acc[j] + res);
                }
            }
        }
    }
    pdl_trigger();
    if (*sFlag && tid == 256) {
        // A wait gave up. Every product issued must be done, and the x copies
        // in flight must land, before the tensor memory is freed and the CTA
        // exits (all waits bounded).
        tc::mma_commit(endbar);
        tc::mbar_wait(endbar, 0, 100000000ull);
        for (int i = 0; i < kAStages; ++i) {
            tc::mbar_wait(xfull + i, 0, 100000000ull);
            tc::mbar_wait(xfull + i, 1, 100000000ull);
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
