// One cached position of the hybrid language model (mamba2_lm_step) and its
// full-history recompute (mamba2_lm_prefill): host code that walks the blocks
// in order and enqueues their kernels on one stream. Per 'M' block: the 4-bit
// in_proj with the block's RMSNorm fused into its staging, the mixer core on
// the strided z | x | B | C | dt rows of its output, the 4-bit out_proj with
// the gated output norm fused into its staging and the residual add into its
// epilogue. Per '*' block: the bf16 q|k|v projection with the RMSNorm fused,
// the cached attention with the KV-cache append, the bf16 output projection
// with the residual add. Every kernel is launched with programmatic dependent
// launch and waits for its predecessor before reading what it wrote.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/mamba2.h"
#include "m2_launch.h"

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t b) { return (b + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
    long HP, GN, W, CH;          // mixer widths; W = in_proj output row
    long QKV, AO;                // attention row widths
    size_t proj, y, mix, qkv, ao, attn, xn;  // workspace parts (bytes, aligned)
    size_t total;
};

m2_status plan(const m2_lm* m, int S, int T, int chunk, bool cached, Plan* p) {
    if (!m || !m->kinds || !m->layers || m->n_layers < 0 || S < 0 || T < 0) return M2_EINVAL;
    const m2_dims& d = m->mixer;
    if (d.act != M2_BF16) return M2_EUNSUPPORTED;
    if (m->hidden <= 0 || m->hidden % 64 != 0 || m->hidden > 16384) return M2_ESHAPE;
    if (d.nheads <= 0 || d.headdim <= 0 || d.dstate <= 0 || d.ngroups <= 0) return M2_EINVAL;
    p->HP = (long)d.nheads * d.headdim;
    p->GN = (long)d.ngroups * d.dstate;
    p->W = 2 * p->HP + 2 * p->GN + d.nheads;
    p->CH = p->HP + 2 * p->GN;
    if (p->W % 8 != 0 || p->HP % 64 != 0 || p->HP > 16384 || d.ngroups > 64 || (p->HP / d.ngroups) % 32 != 0)
        return M2_ESHAPE;
    bool any_attn = false;
    for (int l = 0; l < m->n_layers; ++l) {
        if (m->kinds[l] == '*') any_attn = true;
        else if (m->kinds[l] != 'M') return M2_EINVAL;
    }
    p->QKV = p->AO = 0;
    if (any_attn) {
        if (m->head_dim != 128 || m->n_heads <= 0 || m->n_kv_heads <= 0 || m->n_heads % m->n_kv_heads != 0 ||
            m->n_heads / m->n_kv_heads > m2::kAttnMaxR || m->max_len <= 0 || !isfinite(m->attn_scale))
            return M2_ESHAPE;
        p->QKV = (long)(m->n_heads + 2 * m->n_kv_heads) * m->head_dim;
        p->AO = (long)m->n_heads * m->head_dim;
        if (p->AO > 16384) return M2_ESHAPE;
    }
    if (!(m->norm_eps >= 0.f) || !(m->norm_eps < INFINITY)) return M2_EINVAL;
    const size_t rows = (size_t)S * T;
    m2_dims dd = d;
    dd.batch = S;
    dd.T = T;
    p->proj = up(rows * p->W * 2);
    p->y = up(rows * p->HP * 2);
    p->mix = up(cached ? mamba2_step_workspace_bytes(&dd, S) : mamba2_scan_workspace_bytes(&dd, chunk));
    p->qkv = up(rows * p->QKV * 2);
    p->ao = up(rows * p->AO * 2);
    p->attn = any_attn ? up(mamba2_attn_decode_workspace_bytes(S, m->n_heads, m->n_kv_heads, m->head_dim,
                                                                m->max_len, M2_BF16))
                       : 0;
    // a recompute of many rows normalises the projections' input rows into
    // their own buffer, so that the 4-bit projections run as GEMMs
    p->xn = (!cached && rows >= (size_t)m2::kQgemmMinRows)
                ? up(rows * (size_t)(m->hidden > p->HP ? m->hidden : p->HP) * 2)
                : 0;
    p->total = p->proj + p->y + p->mix + p->qkv + p->ao + p->attn + p->xn;
    return M2_OK;
}

// Pointer checks of every block before anything is launched.
m2_status check_layers(const m2_lm* m) {
    for (int l = 0; l < m->n_layers; ++l) {
        const m2_lm_layer& L = m->layers[l];
        if (!L.norm_w) return M2_EINVAL;
        if (m->kinds[l] == 'M') {
            const void* ptrs[] = {L.in_wq, L.in_scales, L.in_biases, L.A_log, L.D, L.dt_bias, L.conv_w, L.conv_b,
                                  L.gnorm_w, L.out_wq, L.out_scales, L.out_biases, L.ssm_state, L.conv_state};
            for (const void* q : ptrs)
                if (!q) return M2_EINVAL;
            const void* a16[] = {L.norm_w, L.in_wq, L.A_log, L.D, L.dt_bias, L.conv_w, L.conv_b, L.gnorm_w,
                                 L.out_wq, L.ssm_state, L.conv_state};
            for (const void* q : a16)
                if (!aligned16(q)) return M2_EALIGN;
        } else {
            const void* ptrs[] = {L.wqkv, L.wo, L.k_cache, L.v_cache};
            for (const void* q : ptrs)
                if (!q) return M2_EINVAL;
            const void* a16[] = {L.norm_w, L.wqkv, L.wo, L.k_cache, L.v_cache};
            for (const void* q : a16)
                if (!aligned16(q)) return M2_EALIGN;
        }
    }
    return M2_OK;
}

m2_status run(const m2_lm* m, int S, int T, void* hidden, const int32_t* lengths, int chunk, void* workspace,
              size_t workspace_bytes, void* stream, bool cached) {
    Plan p;
    m2_status st = plan(m, S, T, chunk, cached, &p);
    if (st != M2_OK) return st;
    if (!hidden || (!lengths && p.QKV > 0)) return M2_EINVAL;
    if (!aligned16(hidden) || (lengths && (reinterpret_cast<uintptr_t>(lengths) & 3u))) return M2_EALIGN;
    st = check_layers(m);
    if (st != M2_OK) return st;
    if (p.total && (!workspace || workspace_bytes < p.total)) return M2_EWORKSPACE;
    if (workspace && !aligned16(workspace)) return M2_EALIGN;
    st = m2::check_device();
    if (st != M2_OK) return st;
    if (S == 0 || T == 0 || m->n_layers == 0) return M2_OK;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* proj = reinterpret_cast<uint16_t*>(ws);
    uint16_t* y = reinterpret_cast<uint16_t*>(ws + p.proj);
    void* mix = ws + p.proj + p.y;
    uint16_t* qkv = reinterpret_cast<uint16_t*>(ws + p.proj + p.y + p.mix);
    uint16_t* ao = reinterpret_cast<uint16_t*>(ws + p.proj + p.y + p.mix + p.qkv);
    float* attn_ws = reinterpret_cast<float*>(ws + p.proj + p.y + p.mix + p.qkv + p.ao);
    uint16_t* xn = p.xn ? reinterpret_cast<uint16_t*>(ws + p.proj + p.y + p.mix + p.qkv + p.ao + p.attn) : nullptr;
    const int rows = S * T;
    auto row_norm = [&](const m2::RowNorm& nm, const void* x, long x_stride, int in) -> m2_status {
        cudaError_t e = m2::launch_row_norm(nm, x, x_stride, rows, in, xn, static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) return M2_OK;
        m2::record_cuda_error(e);
        return M2_ECUDA;
    };
    const m2_dims& md = m->mixer;
    const long HP = p.HP, GN = p.GN, W = p.W;

    for (int l = 0; l < m->n_layers; ++l) {
        const m2_lm_layer& L = m->layers[l];
        m2_row_norm pre{M2_NORM_RMS, L.norm_w, m->norm_eps, 1, nullptr, 0};
        if (m->kinds[l] == 'M') {
            // proj = in_proj(RMSNorm(h)): rows of z | x | B | C | dt (for many
            // rows: the norm into xn, then the projection as a GEMM)
            if (xn) {
                st = row_norm(m2::RowNorm{1, L.norm_w, m->norm_eps, 1, nullptr, 0}, hidden, m->hidden, m->hidden);
                if (st == M2_OK)
                    st = mamba2_qlinear_fused(rows, m->hidden, (int)W, 64, 4, xn, m->hidden, nullptr, L.in_wq,
                                              L.in_scales, L.in_biases, nullptr, proj, stream);
            } else {
                st = mamba2_qlinear_fused(rows, m->hidden, (int)W, 64, 4, hidden, m->hidden, &pre, L.in_wq,
                                          L.in_scales, L.in_biases, nullptr, proj, stream);
            }
            if (st != M2_OK) return st;
            const uint16_t* x = proj + HP;
            const uint16_t* B = x + HP;
            const uint16_t* C = B + GN;
            const uint16_t* dt = C + GN;
            m2_dims d = md;
            d.batch = S;
            d.T = T;
            if (cached)
                st = mamba2_step_strided(&d, S, x, B, C, dt, W, L.A_log, L.D, L.dt_bias, L.conv_w, L.conv_b,
                                         L.ssm_state, L.conv_state, y, mix, p.mix, stream);
            else
                st = mamba2_conv_scan_strided(&d, x, B, C, dt, W, L.A_log, L.D, L.dt_bias, L.conv_w, L.conv_b, chunk,
                                              L.ssm_state, L.conv_state, y, L.ssm_state, L.conv_state, mix, p.mix,
                                              stream);
            if (st != M2_OK) return st;
            // h = h + out_proj(gated_norm(y, z))
            if (xn) {
                st = row_norm(m2::RowNorm{2, L.gnorm_w, m->norm_eps, md.ngroups, proj, W}, y, HP, (int)HP);
                if (st == M2_OK)
                    st = mamba2_qlinear_fused(rows, (int)HP, m->hidden, 64, 4, xn, HP, nullptr, L.out_wq,
                                              L.out_scales, L.out_biases, hidden, hidden, stream);
            } else {
                m2_row_norm gated{M2_NORM_GATED, L.gnorm_w, m->norm_eps, md.ngroups, proj, W};
                st = mamba2_qlinear_fused(rows, (int)HP, m->hidden, 64, 4, y, HP, &gated, L.out_wq, L.out_scales,
                                          L.out_biases, hidden, hidden, stream);
            }
            if (st != M2_OK) return st;
        } else {
            // q | k | v = Wqkv RMSNorm(h)
            st = mamba2_linear_bf16(rows, m->hidden, (int)p.QKV, hidden, m->hidden, &pre, L.wqkv, nullptr, qkv,
                                    p.QKV, stream);
            if (st != M2_OK) return st;
            // the T positions in order: position t of session s reads row s*T + t
            for (int t = 0; t < T; ++t) {
                m2::AttnArgs a;
                a.S = S;
                a.Hq = m->n_heads;
                a.Hkv = m->n_kv_heads;
                a.Tmax = m->max_len;
                a.bf16 = true;
                a.lens = lengths;
                a.q = qkv + (size_t)t * p.QKV;
                a.k_new = qkv + (size_t)t * p.QKV + p.AO;
                a.v_new = qkv + (size_t)t * p.QKV + p.AO + (long)m->n_kv_heads * m->head_dim;
                a.k_cache = L.k_cache;
                a.v_cache = L.v_cache;
                a.scale = m->attn_scale;
                a.out = ao + (size_t)t * p.AO;
                a.ws = attn_ws;
                a.err = m2::device_error_word();
                a.q_ss = (long)T * p.QKV;
                a.kv_ss = (long)T * p.QKV;
                a.out_ss = (long)T * p.AO;
                a.len_add = t;
                cudaError_t e = m2::launch_attn_decode(a, static_cast<cudaStream_t>(stream));
                if (e != cudaSuccess) {
                    m2::record_cuda_error(e);
                    return M2_ECUDA;
                }
            }
            // h = h + Wo o
            st = mamba2_linear_bf16(rows, (int)p.AO, m->hidden, ao, p.AO, nullptr, L.wo, hidden, hidden, m->hidden,
                                    stream);
            if (st != M2_OK) return st;
        }
    }
    return M2_OK;
}

}  // namespace

extern "C" {

size_t mamba2_lm_workspace_bytes(const m2_lm* m, int n_sessions, int T, int chunk) {
    Plan p;
    if (plan(m, n_sessions, T, chunk, false, &p) != M2_OK) return 0;
    Plan q;
    if (plan(m, n_sessions, 1, 1, true, &q) != M2_OK) return 0;
    return T == 1 && p.total < q.total ? q.total : p.total;
}

m2_status mamba2_lm_step(const m2_lm* m, int n_sessions, void* hidden, const int32_t* lengths, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return run(m, n_sessions, 1, hidden, lengths, 1, workspace, workspace_bytes, stream, true);
}

m2_status mamba2_lm_prefill(const m2_lm* m, int n_sessions, int T, void* hidden, const int32_t* lengths, int chunk,
                            void* workspace, size_t workspace_bytes, void* stream) {
    if (chunk < 1 || chunk > 128) return M2_EINVAL;
    return run(m, n_sessions, T, hidden, lengths, chunk, workspace, workspace_bytes, stream, false);
}

}  // extern "C"
