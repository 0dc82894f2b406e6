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
//     At its end each CTA also writes its share of the final conv tail (the
//     last K-1 pre-conv frames).
//
// The chunked form is the state-space-duality (SSD) evaluation of the Mamba-2
// recurrence (Dao & Gu 2024): the intra-chunk part is a masked quadratic form,
// the carried state enters through C~ h_prev.
#include <math.h>

#include "m2_common.cuh"
#include "m2_launch.h"
#include "m2_tc.cuh"

namespace m2 {

namespace {

constexpr int kTR = 128;                       // tile rows: the maximum chunk length
constexpr int kNP = 128;                       // state dimension padded to the MMA M extent
constexpr uint32_t kTileBytes = kTR * kNP * 2;  // one bf16 operand tile, 32 KiB
constexpr uint32_t kPanel = kTR * 128;          // one 64-column panel of a tile, 16 KiB

// ----------------------------------------------------------------- kernel 1
constexpr int kBcThreads = 256;

template <typename TA>
__global__ void __launch_bounds__(kBcThreads) scan_bc_kernel(ScanArgs a, int nchunks) {
    const Shape& s = a.s;
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int T = a.T, Q = a.chunk;
    const int c0 = c * Q;
    const int L = min(Q, T - c0);
    const long HP = s.HP(), GN = s.GN(), CH = s.CH();
    uint8_t* tiles = reinterpret_cast<uint8_t*>(a.ws) + (((size_t)b * nchunks + c) * s.G + g) * 3 * kTileBytes;
    uint8_t* tBh = tiles;
    uint8_t* tBl = tiles + kTileBytes;
    uint8_t* tCh = tiles + 2 * kTileBytes;

    // 32 columns of 8 channels: 16 for B (n = 0..127), 16 for C; 8 row segments of 16.
    const int cc = threadIdx.x & 31, rs = threadIdx.x >> 5;
    const int which = cc >> 4;  // 0: B, 1: C
    const int n0 = (cc & 15) * 8;
    const int r0 = rs * 16;
    const bool real = n0 < s.N;
    const long ch0 = HP + which * GN + (long)g * s.N + n0;  // conv channel of n0
    const void* src = which ? a.C : a.B;

    float w[8][4], bias[8];
    if (real) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 wj = __ldg(reinterpret_cast<const float4*>(a.conv_w) + ch0 + j);
            w[j][0] = wj.x; w[j][1] = wj.y; w[j][2] = wj.z; w[j][3] = wj.w;
            bias[j] = __ldg(a.conv_b + ch0 + j);
        }
    }
    // sliding window of pre-conv rows t-3, t-2, t-1
    float win[3][8];
    auto load_row = [&](int t, float (&out)[8]) {
        if (t >= 0 && t < T) {
            Act8<TA> v;
            v.load(src, (((size_t)b * T + t) * s.G + g) * s.N + n0);
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = v.get(j);
        } else if (t < 0 && a.init_conv) {
            Act8<TA> v;
            v.load(a.init_conv, ((size_t)b * (s.K - 1) + (s.K - 1 + t)) * CH + ch0);
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = v.get(j);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = 0.f;
        }
    };
    if (real && r0 < L) {
#pragma unroll
        for (int k = 0; k < 3; ++k) load_row(c0 + r0 - 3 + k, win[k]);
    }
    for (int r = r0; r < r0 + 16; ++r) {
        uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
        if (real && r < L) {
            float cur[8];
            load_row(c0 + r, cur);
            uint32_t hb[8], lb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float u = bias[j];
                u = fmaf(w[j][0], win[0][j], u);
                u = fmaf(w[j][1], win[1][j], u);
                u = fmaf(w[j][2], win[2][j], u);
                u = fmaf(w[j][3], cur[j], u);
                const float v = silu_f32(u);
                hb[j] = float_to_bf16_bits(v);
                lb[j] = float_to_bf16_bits(v - bf16_bits_to_float(hb[j]));
                win[0][j] = win[1][j];
                win[1][j] = win[2][j];
                win[2][j] = cur[j];
            }
            hi = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16), hb[6] | (hb[7] << 16));
            lo = make_uint4(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16), lb[4] | (lb[5] << 16), lb[6] | (lb[7] << 16));
        }
        const uint32_t off = tc::sw128_off(r, n0, kTR);
        if (which == 0) {
            *reinterpret_cast<uint4*>(tBh + off) = hi;
            *reinterpret_cast<uint4*>(tBl + off) = lo;
        } else {
            *reinterpret_cast<uint4*>(tCh + off) = hi;
        }
    }
}

// The final conv tail of 8 channels [c, c+8) of sequence b: frames T-3..T-1,
// taken from the initial tail (or zeros) where T < 3. Every source slot is
// read before any is written, so final_conv may alias init_conv.
template <typename TA>
__device__ void write_tail(const ScanArgs& a, int b, long c) {
    const Shape& s = a.s;
    const long CH = s.CH(), HP = s.HP(), GN = s.GN();
    const int T = a.T;
    Act8<TA> vals[3];
    bool zero[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int t = T - 3 + k;
        zero[k] = false;
        if (t >= 0) {
            if (c < HP)
                vals[k].load(a.x, ((size_t)b * T + t) * HP + c);
            else if (c < HP + GN)
                vals[k].load(a.B, ((size_t)b * T + t) * GN + (c - HP));
            else
                vals[k].load(a.C, ((size_t)b * T + t) * GN + (c - HP - GN));
        } else if (a.init_conv) {
            vals[k].load_rw(a.init_conv, ((size_t)b * 3 + (3 + t)) * CH + c);
        } else {
            zero[k] = true;
        }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        if (zero[k]) memset(&vals[k], 0, sizeof(vals[k]));
        vals[k].store(a.final_conv, ((size_t)b * 3 + k) * CH + c);
    }
}

// ----------------------------------------------------------------- kernel 2
constexpr int kSsdThreads = 256;
// TMEM columns
constexpr uint32_t kColG = 0, kColState = 128, kColYd = 256, kColYo = 384, kTmemCols = 512;

template <int P>
struct SsdSmem {
    static constexpr uint32_t kC = 0;                     // C~ hi           (K-major SW128)
    static constexpr uint32_t kBh = kTileBytes;           // B~ hi           (K-major / MN-major SW128)
    static constexpr uint32_t kBl = 2 * kTileBytes;       // B~ lo, then M   (SW128)
    static constexpr uint32_t kPT = kTR * P * 2;          // one [128 x P] bf16 interleaved tile
    static constexpr uint32_t kX = 3 * kTileBytes;        // x~ hi           (MN-major interleave, K = j)
    static constexpr uint32_t kWh = kX + kPT;             // (w o x~) hi
    static constexpr uint32_t kWl = kWh + kPT;            // (w o x~) lo
    static constexpr uint32_t kH = kWl + kPT;             // h hi            (MN-major interleave, K = n)
    static constexpr uint32_t kS = kH + kPT;              // float S[128]
    static constexpr uint32_t kDt = kS + 512;             // float dt[128]
    static constexpr uint32_t kWsum = kDt + 512;          // float warp sums[8]
    static constexpr uint32_t kCw = kWsum + 64;           // float conv_w[P][4]
    static constexpr uint32_t kCb = kCw + P * 16;         // float conv_b[P]
    static constexpr uint32_t kBar = (kCb + P * 4 + 15) / 16 * 16;  // 3 mbarriers
    static constexpr uint32_t kTmem = kBar + 24;          // TMEM base address
    static constexpr uint32_t kFlag = kTmem + 4;          // abort flag
    static constexpr uint32_t kBytes = kFlag + 4 + 1024;  // + slack to align the base to 1024
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    return (uint32_t)float_to_bf16_bits(a) | ((uint32_t)float_to_bf16_bits(b) << 16);
}

template <typename TA, int P>
__global__ void __launch_bounds__(kSsdThreads, 1) scan_ssd_kernel(ScanArgs a, int nchunks) {
    using L = SsdSmem<P>;
    constexpr int PH = P / 2;  // columns handled by each half of the CTA
    constexpr uint32_t LBO_I = (P / 8) * 128;  // K-group stride of the interleaved tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const Shape& s = a.s;
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / (s.H / s.G);
    const int T = a.T, Q = a.chunk;
    const long HP = s.HP(), CH = s.CH();
    const int tid = threadIdx.x, row = tid & 127, half = tid >> 7, warp = tid >> 5;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    float* sS = reinterpret_cast<float*>(sm + L::kS);
    float* sDt = reinterpret_cast<float*>(sm + L::kDt);
    float* sWsum = reinterpret_cast<float*>(sm + L::kWsum);
    float* sCw = reinterpret_cast<float*>(sm + L::kCw);
    float* sCb = reinterpret_cast<float*>(sm + L::kCb);
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + L::kBar);
    uint64_t* bar_m1 = bar_ld + 1;
    uint64_t* bar_m2 = bar_ld + 2;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::kTmem);
    volatile uint32_t* sFlag = reinterpret_cast<uint32_t*>(sm + L::kFlag);

    if (tid == 0) {
        tc::mbar_init(bar_ld, 1);
        tc::mbar_init(bar_m1, 1);
        tc::mbar_init(bar_m2, 1);
        tc::fence_mbar_init();
        *sFlag = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(sTmem, kTmemCols);
        tc::tmem_relinquish();
    }
    for (int i = tid; i < P; i += kSsdThreads) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(a.conv_w) + (long)h * P + i);
        sCw[i * 4 + 0] = wv.x; sCw[i * 4 + 1] = wv.y; sCw[i * 4 + 2] = wv.z; sCw[i * 4 + 3] = wv.w;
        sCb[i] = __ldg(a.conv_b + (long)h * P + i);
    }
    const float A = -expf(__ldg(a.A_log + h));
    const float Dh = __ldg(a.D + h);
    const float dtb = __ldg(a.dt_bias + h);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tm = *sTmem;

    // initial state -> TMEM [n lanes][p columns]; rows n >= N stay zero
    {
        const int n = row;
        for (int p0 = half * PH; p0 < (half + 1) * PH; p0 += 8) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                v[q] = (a.init_ssm && n < s.N)
                           ? __ldg(a.init_ssm + (((size_t)b * s.H + h) * P + p0 + q) * s.N + n)
                           : 0.f;
            tc::tmem_st8(tm + lane_base + kColState + p0, v);
        }
        tc::tmem_wait_st();
    }

    const uint32_t sbase = tc::smem_u32(sm);
    const uint8_t* ws = reinterpret_cast<const uint8_t*>(a.ws);
    bool ok = true;

    for (int c = 0; c < nchunks; ++c) {
        const int c0 = c * Q;
        const int Lc = min(Q, T - c0);
        const int ksteps = (Lc + 15) / 16;
        const uint32_t par = c & 1;

        // 1. B~/C~ tiles of this chunk and group: bulk copy into shared memory
        if (tid == 0) {
            const uint8_t* src = ws + (((size_t)b * nchunks + c) * s.G + g) * 3 * kTileBytes;
            tc::mbar_arrive_expect_tx(bar_ld, 3 * kTileBytes);
            tc::bulk_g2s(sm + L::kBh, src, kTileBytes, bar_ld);
            tc::bulk_g2s(sm + L::kBl, src + kTileBytes, kTileBytes, bar_ld);
            tc::bulk_g2s(sm + L::kC, src + 2 * kTileBytes, kTileBytes, bar_ld);
        }

        // 2. dt, a = dt A, inclusive cumulative sum S over the chunk
        if (half == 0) {
            float dt = 0.f;
            if (row < Lc) dt = softplus_f32(load_act<TA>(a.dt_raw, ((size_t)b * T + c0 + row) * s.H + h) + dtb);
            float v = dt * A;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, v, off);
                if ((tid & 31) >= off) v += o;
            }
            if ((tid & 31) == 31) sWsum[warp] = v;
            sDt[row] = dt;
            sS[row] = v;  // warp-local prefix for now
        }
        __syncthreads();
        if (half == 0) {
            float add = 0.f;
            for (int w = 0; w < (row >> 5); ++w) add += sWsum[w];
            sS[row] += add;
        }
        __syncthreads();
        const float Slast = sS[Lc - 1];
        const float Si = sS[row];
        const float wi = row < Lc ? expf(Slast - Si) * sDt[row] : 0.f;

        // 3. conv + SiLU of this head's x channels for row i, columns of this half
        float xf[PH];
        {
            const int t = c0 + row;
#pragma unroll
            for (int q8 = 0; q8 < PH / 8; ++q8) {
                const int p0 = half * PH + q8 * 8;
                float o[8];
                if (row < Lc) {
                    float acc[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = sCb[p0 + j];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int tt = t - 3 + k;
                        Act8<TA> v;
                        bool have = true;
                        if (tt >= 0)
                            v.load(a.x, (((size_t)b * T + tt) * s.H + h) * P + p0);
                        else if (a.init_conv)
                            v.load(a.init_conv, ((size_t)b * (s.K - 1) + (s.K - 1 + tt)) * CH + (long)h * P + p0);
                        else
                            have = false;
                        if (have) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[j] = fmaf(sCw[(p0 + j) * 4 + k], v.get(j), acc[j]);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = silu_f32(acc[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = 0.f;
                }
                uint32_t xh[4], wh[4], wl[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    xf[q8 * 8 + j] = o[j];
                    xf[q8 * 8 + j + 1] = o[j + 1];
                    xh[j / 2] = pack2(o[j], o[j + 1]);
                    const float w0 = wi * o[j], w1 = wi * o[j + 1];
                    const uint32_t h0 = float_to_bf16_bits(w0), h1 = float_to_bf16_bits(w1);
                    wh[j / 2] = h0 | (h1 << 16);
                    wl[j / 2] = pack2(w0 - bf16_bits_to_float(h0), w1 - bf16_bits_to_float(h1));
                }
                const uint32_t off = tc::mn_inter_off(p0, row, P);
                *reinterpret_cast<uint4*>(sm + L::kX + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
                *reinterpret_cast<uint4*>(sm + L::kWh + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4*>(sm + L::kWl + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }

        // 4. state: h_prev (bf16) into shared memory for Y_off, then h <- exp(S_last) h in TMEM
        {
            const float decay = expf(Slast);
            const int n = row;
#pragma unroll
            for (int q8 = 0; q8 < PH / 8; ++q8) {
                const int p0 = half * PH + q8 * 8;
                float v[8];
                tc::tmem_ld8(tm + lane_base + kColState + p0, v);
                tc::tmem_wait_ld();
                *reinterpret_cast<uint4*>(sm + L::kH + tc::mn_inter_off(p0, n, P)) =
                    make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] *= decay;
                tc::tmem_st8(tm + lane_base + kColState + p0, v);
            }
            tc::tmem_wait_st();
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();

        // 5. tensor-core phase 1: G, Y_off, state update
        if (tid == 0) {
            tc::tc_fence_after();
            if (!tc::mbar_wait(bar_ld, par)) {
                atomicOr(a.err, ERR_MBAR_TIMEOUT_LOAD);
                *sFlag = 1;
            } else {
                const uint32_t sC = sbase + L::kC, sBh = sbase + L::kBh, sBl = sbase + L::kBl;
                const uint32_t sX = sbase + L::kX, sWh = sbase + L::kWh, sWl = sbase + L::kWl, sH = sbase + L::kH;
                (void)sX;
                const uint32_t idG = tc::idesc_bf16(128, 128, 0, 0);
                const uint32_t idY = tc::idesc_bf16(128, P, 0, 1);
                const uint32_t idS = tc::idesc_bf16(128, P, 1, 1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t koff = (ks >> 2) * kPanel + (ks & 3) * 32;
                    tc::mma_bf16(tm + kColG, tc::sdesc(sC + koff, 0, 1024, 2), tc::sdesc(sBh + koff, 0, 1024, 2), idG,
                                 ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t koff = (ks >> 2) * kPanel + (ks & 3) * 32;
                    tc::mma_bf16(tm + kColYo, tc::sdesc(sC + koff, 0, 1024, 2),
                                 tc::sdesc(sH + ks * 2 * LBO_I, LBO_I, 128, 0), idY, ks > 0);
                }
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint64_t dBh = tc::sdesc(sBh + ks * 2048, kPanel, 1024, 2);
                    const uint64_t dBl = tc::sdesc(sBl + ks * 2048, kPanel, 1024, 2);
                    const uint64_t dWh = tc::sdesc(sWh + ks * 2 * LBO_I, LBO_I, 128, 0);
                    const uint64_t dWl = tc::sdesc(sWl + ks * 2 * LBO_I, LBO_I, 128, 0);
                    tc::mma_bf16(tm + kColState, dBh, dWh, idS, 1);
                    tc::mma_bf16(tm + kColState, dBh, dWl, idS, 1);
                    tc::mma_bf16(tm + kColState, dBl, dWh, idS, 1);
                }
                tc::mma_commit(bar_m1);
            }
        }
        __syncthreads();
        if (*sFlag) { ok = false; break; }
        if (!tc::mbar_wait(bar_m1, par)) {
            atomicOr(a.err, ERR_MBAR_TIMEOUT_MMA);
            *sFlag = 1;
        }
        if (__syncthreads_or(*sFlag)) { ok = false; break; }
        tc::tc_fence_after();

        // 6. M = G o exp(S_i - S_j) dt_j (j <= i) -> bf16, K-major SW128 over the B~ lo tile
        {
            const int i = row;
#pragma unroll 1
            for (int j0 = half * 64; j0 < half * 64 + 64; j0 += 16) {
                float gv[16];
                tc::tmem_ld16(tm + lane_base + kColG + j0, gv);
                tc::tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int q = 0; q < 16; q += 2) {
                    float m0 = 0.f, m1 = 0.f;
                    const int j = j0 + q;
                    if (i < Lc && j <= i) m0 = gv[q] * expf(Si - sS[j]) * sDt[j];
                    if (i < Lc && j + 1 <= i) m1 = gv[q + 1] * expf(Si - sS[j + 1]) * sDt[j + 1];
                    pk[q / 2] = pack2(m0, m1);
                }
                *reinterpret_cast<uint4*>(sm + L::kBl + tc::sw128_off(i, j0, kTR)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(sm + L::kBl + tc::sw128_off(i, j0 + 8, kTR)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();

        // 7. tensor-core phase 2: Y_diag = M x~
        if (tid == 0) {
            tc::tc_fence_after();
            const uint32_t sM = sbase + L::kBl, sX = sbase + L::kX;
            const uint32_t idY = tc::idesc_bf16(128, P, 0, 1);
            for (int ks = 0; ks < ksteps; ++ks) {
                const uint32_t koff = (ks >> 2) * kPanel + (ks & 3) * 32;
                tc::mma_bf16(tm + kColYd, tc::sdesc(sM + koff, 0, 1024, 2), tc::sdesc(sX + ks * 2 * LBO_I, LBO_I, 128, 0),
                             idY, ks > 0);
            }
            tc::mma_commit(bar_m2);
        }
        __syncwarp();
        if (!tc::mbar_wait(bar_m2, par)) {
            atomicOr(a.err, ERR_MBAR_TIMEOUT_MMA);
            *sFlag = 1;
        }
        if (__syncthreads_or(*sFlag)) { ok = false; break; }
        tc::tc_fence_after();

        // 8. y = Y_diag + exp(S_i) Y_off + D x~. The TMEM loads are warp-collective
        //    (.sync.aligned): every lane issues them; only the stores are predicated.
        {
            const float eS = expf(Si);
            const bool live = row < Lc;
            const size_t ybase = (((size_t)b * T + c0 + row) * s.H + h) * P;
#pragma unroll
            for (int q8 = 0; q8 < PH / 8; ++q8) {
                const int p0 = half * PH + q8 * 8;
                float yd[8], yo[8];
                tc::tmem_ld8(tm + lane_base + kColYd + p0, yd);
                tc::tmem_ld8(tm + lane_base + kColYo + p0, yo);
                tc::tmem_wait_ld();
                float out[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) out[q] = fmaf(eS, yo[q], yd[q]) + Dh * xf[q8 * 8 + q];
                if (live) {
                    if constexpr (sizeof(TA) == 2) {
                        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.y) + ybase + p0) =
                            make_uint4(pack2(out[0], out[1]), pack2(out[2], out[3]), pack2(out[4], out[5]),
                                       pack2(out[6], out[7]));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + ybase + p0);
                        dst[0] = make_float4(out[0], out[1], out[2], out[3]);
                        dst[1] = make_float4(out[4], out[5], out[6], out[7]);
                    }
                }
            }
        }
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    }

    // final state: TMEM [n][p] -> final_ssm [b,h,p,n]
    if (ok) {
        const int n = row;
        for (int p0 = half * PH; p0 < (half + 1) * PH; p0 += 8) {
            float v[8];
            tc::tmem_ld8(tm + lane_base + kColState + p0, v);
            tc::tmem_wait_ld();
            if (n < s.N) {
#pragma unroll
                for (int q = 0; q < 8; ++q) a.final_ssm[(((size_t)b * s.H + h) * P + p0 + q) * s.N + n] = v[q];
            }
        }
    } else if (tid == 0) {
        // a wait gave up: let any bulk copy still in flight land before the CTA exits
        tc::mbar_wait(bar_ld, 0, 100000000ull);
        tc::mbar_wait(bar_ld, 1, 100000000ull);
    }
    // final conv tail (the last K-1 pre-conv frames). This CTA owns the tail of
    // its head's x channels (whose initial frames only it has read); the first
    // head of each group also owns the group's B and C channels (whose initial
    // frames only the prologue kernel read). So in-place updates are safe.
    {
        const int R = s.H / s.G;
        const int nx = P / 8, nbc = (h % R == 0) ? 2 * s.N / 8 : 0;
        for (int v = tid; v < nx + nbc; v += kSsdThreads) {
            long c;
            if (v < nx)
                c = (long)h * P + v * 8;
            else if (v - nx < s.N / 8)
                c = HP + (long)g * s.N + (v - nx) * 8;
            else
                c = HP + s.GN() + (long)g * s.N + (v - nx - s.N / 8) * 8;
            write_tail<TA>(a, b, c);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, kTmemCols);
}

template <typename TA, int P>
cudaError_t launch_ssd(const ScanArgs& a, int nchunks, cudaStream_t st) {
    const int smem = SsdSmem<P>::kBytes;
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
    scan_ssd_kernel<TA, P><<<dim3(a.s.H, a.batch), kSsdThreads, smem, st>>>(a, nchunks);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_bc_typed(const ScanArgs& a, cudaStream_t st) {
    const int nchunks = (a.T + a.chunk - 1) / a.chunk;
    if (nchunks == 0) return cudaSuccess;
    scan_bc_kernel<TA><<<dim3(nchunks, a.s.G, a.batch), kBcThreads, 0, st>>>(a, nchunks);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_chunks_typed(const ScanArgs& a, cudaStream_t st) {
    const int nchunks = (a.T + a.chunk - 1) / a.chunk;
    switch (a.s.P) {
        case 16: return launch_ssd<TA, 16>(a, nchunks, st);
        case 32: return launch_ssd<TA, 32>(a, nchunks, st);
        case 48: return launch_ssd<TA, 48>(a, nchunks, st);
        case 64: return launch_ssd<TA, 64>(a, nchunks, st);
        case 80: return launch_ssd<TA, 80>(a, nchunks, st);
        case 96: return launch_ssd<TA, 96>(a, nchunks, st);
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

cudaError_t launch_scan_chunks(const ScanArgs& a, cudaStream_t st) {
    if (a.batch == 0) return cudaSuccess;
    return a.s.bf16 ? launch_chunks_typed<bf16_t>(a, st) : launch_chunks_typed<float>(a, st);
}

}  // namespace m2
