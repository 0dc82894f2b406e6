// The C ABI of libmamba2.so (declared in include/mamba2.h): argument,
// shape and alignment validation on the host, then dispatch to the kernel
// launchers. Nothing here allocates device memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mamba2.h"
#include "m2_launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

// Device error word: bounded waits inside the kernels record why they gave up.
__device__ unsigned int g_dev_error = 0;

constexpr int kMaxDevices = 64;
// Per-device facts resolved once: 0 = unknown, 1 = sm_103, 2 = other.
int g_dev_kind[kMaxDevices] = {0};
unsigned int* g_dev_error_ptr[kMaxDevices] = {nullptr};
// Guards the per-device set-up above: two host threads making their first
// call on one device must not see the kind set before the pointer.
std::mutex g_dev_mutex;

m2_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return M2_ECUDA;
}

m2_status current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (*dev < 0 || *dev >= kMaxDevices) return M2_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_kind[*dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
        if (e != cudaSuccess) return cuda_fail(e);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dev_error);
        if (e != cudaSuccess) return cuda_fail(e);
        g_dev_error_ptr[*dev] = static_cast<unsigned int*>(p);
        g_dev_kind[*dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return g_dev_kind[*dev] == 1 ? M2_OK : M2_EUNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

m2_status check_dims(const m2_dims* d, bool need_seq) {
    if (!d) return M2_EINVAL;
    if (d->nheads <= 0 || d->headdim <= 0 || d->dstate <= 0 || d->ngroups <= 0 || d->dconv <= 0)
        return M2_EINVAL;
    if (need_seq && (d->batch < 0 || d->T < 0)) return M2_EINVAL;
    if (d->act != M2_BF16 && d->act != M2_F32) return M2_EINVAL;
    if (d->dconv != 4) return M2_ESHAPE;
    const int N = d->dstate;
    if (N != 16 && N != 32 && N != 64 && N != 128) return M2_ESHAPE;
    if (d->headdim % 16 != 0 || d->headdim > 80) return M2_ESHAPE;
    if (d->nheads % d->ngroups != 0) return M2_ESHAPE;
    if (((long)d->nheads * d->headdim) % 8 != 0 || ((long)d->ngroups * N) % 8 != 0) return M2_ESHAPE;
    return M2_OK;
}

m2::Shape shape_of(const m2_dims* d) {
    m2::Shape s;
    s.H = d->nheads;
    s.P = d->headdim;
    s.N = d->dstate;
    s.G = d->ngroups;
    s.K = d->dconv;
    s.bf16 = d->act == M2_BF16;
    return s;
}

}  // namespace

namespace m2 {
void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

m2_status check_step_args(const m2_dims* d, int n_sessions, const void* x, const void* B, const void* C,
                          const void* dt_raw, const float* A_log, const float* D, const float* dt_bias,
                          const float* conv_w, const float* conv_b, const float* ssm_state,
                          const void* conv_state, const void* y) {
    m2_status st = check_dims(d, false);
    if (st != M2_OK) return st;
    if (n_sessions < 0) return M2_EINVAL;
    const void* ptrs[] = {x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, ssm_state, conv_state, y};
    for (const void* p : ptrs)
        if (!p) return M2_EINVAL;
    for (const void* p : ptrs)
        if (!aligned16(p)) return M2_EALIGN;
    return M2_OK;
}

m2_status check_device() {
    int dev = 0;
    return current_device(&dev);
}

unsigned int* device_error_word() {
    int dev = 0;
    return current_device(&dev) == M2_OK ? g_dev_error_ptr[dev] : nullptr;
}
}  // namespace m2

extern "C" {

const char* mamba2_status_string(m2_status s) {
    switch (s) {
        case M2_OK: return "ok";
        case M2_EINVAL: return "invalid argument (null pointer or non-positive size)";
        case M2_ESHAPE: return "unsupported dimensions";
        case M2_EALIGN: return "pointer not 16-byte aligned";
        case M2_EUNSUPPORTED: return "current device is not an sm_103 GPU";
        case M2_ECUDA: return "CUDA error (see mamba2_last_cuda_error)";
        case M2_EWORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int mamba2_last_cuda_error(void) { return g_last_cuda_error; }

m2_status mamba2_device_error(void* stream, unsigned int* code) {
    if (!code) return M2_EINVAL;
    int dev = 0;
    m2_status st = current_device(&dev);
    if (st != M2_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyAsync(code, g_dev_error_ptr[dev], sizeof(unsigned int),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(g_dev_error_ptr[dev], &zero, sizeof(unsigned int), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

// Checks a row norm for rows of `in` inputs and fills `n` (kind 0 for NULL).
m2_status row_norm_setup(const m2_row_norm* norm, int in, m2::RowNorm* n) {
    n->kind = 0;
    n->weight = nullptr;
    n->eps = 0.f;
    n->groups = 1;
    n->gate = nullptr;
    n->gate_stride = 0;
    if (!norm || norm->kind == M2_NORM_NONE) return M2_OK;
    if (norm->kind != M2_NORM_RMS && norm->kind != M2_NORM_GATED) return M2_EINVAL;
    if (!norm->weight || !(norm->eps >= 0.f) || !(norm->eps < INFINITY)) return M2_EINVAL;
    if (!aligned16(norm->weight)) return M2_EALIGN;
    n->kind = norm->kind == M2_NORM_RMS ? 1 : 2;
    n->weight = norm->weight;
    n->eps = norm->eps;
    if (in % 32 != 0) return M2_ESHAPE;
    if (n->kind == 2) {
        if (!norm->gate || norm->groups <= 0 || norm->gate_stride < in) return M2_EINVAL;
        if (norm->groups > m2::kMaxNormGroups || in % norm->groups != 0 || (in / norm->groups) % 32 != 0)
            return M2_ESHAPE;
        if (!aligned16(norm->gate) || (norm->gate_stride * 2) % 16 != 0) return M2_EALIGN;
        n->groups = norm->groups;
        n->gate = norm->gate;
        n->gate_stride = norm->gate_stride;
    }
    return M2_OK;
}

}  // namespace

extern "C" {

m2_status mamba2_qlinear_fused(int rows, int in_features, int out_features, int group_size, int bits,
                               const void* x, long x_stride, const m2_row_norm* norm, const uint32_t* wq,
                               const void* scales, const void* biases, const void* residual, void* y,
                               void* stream) {
    if (rows < 0 || in_features <= 0 || out_features <= 0 || group_size <= 0 || bits <= 0) return M2_EINVAL;
    if (group_size != 64 || bits != 4) return M2_EUNSUPPORTED;
    if (in_features % 64 != 0 || in_features > m2::kQlMaxIn) return M2_ESHAPE;
    if (!x || !wq || !scales || !biases || !y || x_stride < in_features) return M2_EINVAL;
    if (!aligned16(x) || (x_stride * 2) % 16 != 0 || !aligned16(wq) || !aligned2(scales) || !aligned2(biases) ||
        !aligned2(y) || !aligned2(residual))
        return M2_EALIGN;
    m2::QLinearArgs a;
    m2_status st = row_norm_setup(norm, in_features, &a.norm);
    if (st != M2_OK) return st;
    int dev = 0;
    st = current_device(&dev);
    if (st != M2_OK) return st;
    if (rows == 0) return M2_OK;
    a.rows = rows;
    a.in = in_features;
    a.out = out_features;
    a.x = x;
    a.x_stride = x_stride;
    a.wq = wq;
    a.scales = static_cast<const uint16_t*>(scales);
    a.biases = static_cast<const uint16_t*>(biases);
    a.residual = residual;
    a.y = y;
    a.err = m2::device_error_word();
    cudaError_t e = m2::launch_qlinear(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_qlinear(int rows, int in_features, int out_features, int group_size, int bits, const void* x,
                         const uint32_t* wq, const void* scales, const void* biases, void* y, void* stream) {
    return mamba2_qlinear_fused(rows, in_features, out_features, group_size, bits, x, in_features, nullptr, wq,
                                scales, biases, nullptr, y, stream);
}

m2_status mamba2_linear_bf16(int rows, int in_features, int out_features, const void* x, long x_stride,
                             const m2_row_norm* norm, const void* w, const void* residual, void* y, long y_stride,
                             void* stream) {
    if (rows < 0 || in_features <= 0 || out_features <= 0) return M2_EINVAL;
    if (in_features % 32 != 0 || in_features > m2::kLinMaxIn) return M2_ESHAPE;
    if (!x || !w || !y || x_stride < in_features || y_stride < out_features) return M2_EINVAL;
    if (!aligned16(x) || (x_stride * 2) % 16 != 0 || !aligned16(w) || !aligned2(y) || !aligned2(residual))
        return M2_EALIGN;
    m2::LinearArgs a;
    m2_status st = row_norm_setup(norm, in_features, &a.norm);
    if (st != M2_OK) return st;
    int dev = 0;
    st = current_device(&dev);
    if (st != M2_OK) return st;
    if (rows == 0) return M2_OK;
    a.rows = rows;
    a.in = in_features;
    a.out = out_features;
    a.x = x;
    a.x_stride = x_stride;
    a.w = w;
    a.residual = residual;
    a.y = y;
    a.y_stride = y_stride;
    cudaError_t e = m2::launch_linear_bf16(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

size_t mamba2_step_workspace_bytes(const m2_dims* d, int n_sessions) {
    if (check_dims(d, false) != M2_OK || n_sessions < 0) return 0;
    return m2::step_workspace_bytes(shape_of(d), n_sessions);
}

namespace {
m2_status attn_sizes(int n_sessions, int n_heads, int n_kv_heads, int head_dim, int max_len, m2_dtype act) {
    if (n_sessions < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_len <= 0) return M2_EINVAL;
    if (act != M2_BF16 && act != M2_F32) return M2_EINVAL;
    if (head_dim != m2::kAttnD || n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > m2::kAttnMaxR)
        return M2_ESHAPE;
    if (n_kv_heads > 65535 || n_sessions > 65535) return M2_ESHAPE;
    return M2_OK;
}
}  // namespace

size_t mamba2_attn_decode_workspace_bytes(int n_sessions, int n_heads, int n_kv_heads, int head_dim, int max_len,
                                          m2_dtype act) {
    if (attn_sizes(n_sessions, n_heads, n_kv_heads, head_dim, max_len, act) != M2_OK) return 0;
    return m2::attn_workspace_bytes(n_sessions, n_heads, n_kv_heads, max_len, act == M2_BF16);
}

m2_status mamba2_attn_decode(int n_sessions, int n_heads, int n_kv_heads, int head_dim, int max_len, m2_dtype act,
                             const int32_t* lengths, const void* q, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, float scale, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    m2_status st = attn_sizes(n_sessions, n_heads, n_kv_heads, head_dim, max_len, act);
    if (st != M2_OK) return st;
    if (!isfinite(scale)) return M2_EINVAL;
    const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, out};
    if (!lengths) return M2_EINVAL;
    for (const void* p : ptrs)
        if (!p) return M2_EINVAL;
    if (reinterpret_cast<uintptr_t>(lengths) & 3u) return M2_EALIGN;
    for (const void* p : ptrs)
        if (!aligned16(p)) return M2_EALIGN;
    const size_t need = m2::attn_workspace_bytes(n_sessions, n_heads, n_kv_heads, max_len, act == M2_BF16);
    if (need && (!workspace || workspace_bytes < need)) return M2_EWORKSPACE;
    if (workspace && !aligned16(workspace)) return M2_EALIGN;
    int dev = 0;
    st = current_device(&dev);
    if (st != M2_OK) return st;
    if (n_sessions == 0) return M2_OK;
    m2::AttnArgs a;
    a.S = n_sessions;
    a.Hq = n_heads;
    a.Hkv = n_kv_heads;
    a.Tmax = max_len;
    a.bf16 = act == M2_BF16;
    a.lens = lengths;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.scale = scale;
    a.out = out;
    a.ws = static_cast<float*>(workspace);
    a.err = g_dev_error_ptr[dev];
    a.q_ss = (long)n_heads * head_dim;
    a.kv_ss = (long)n_kv_heads * head_dim;
    a.out_ss = (long)n_heads * head_dim;
    a.len_add = 0;
    cudaError_t e = m2::launch_attn_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_gated_norm(const m2_dims* d, int rows, const void* y, const void* z, const float* weight,
                            float eps, void* out, void* stream) {
    m2_status st = check_dims(d, false);
    if (st != M2_OK) return st;
    if (rows < 0 || !(eps >= 0.f) || !(eps < INFINITY)) return M2_EINVAL;
    if ((long)d->nheads / d->ngroups * d->headdim > 32768) return M2_EUNSUPPORTED;
    const void* ptrs[] = {y, z, weight, out};
    for (const void* p : ptrs)
        if (!p) return M2_EINVAL;
    for (const void* p : ptrs)
        if (!aligned16(p)) return M2_EALIGN;
    int dev = 0;
    st = current_device(&dev);
    if (st != M2_OK) return st;
    m2::NormArgs a;
    a.s = shape_of(d);
    a.rows = rows;
    a.y = y;
    a.z = z;
    a.weight = weight;
    a.eps = eps;
    a.out = out;
    cudaError_t e = m2::launch_gated_norm(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// mamba2_step and mamba2_step_strided: `sx`, `sbc`, `sdt` are the elements
// from one session's row of x, of B and C, and of dt_raw to the next.
m2_status step_impl(const m2_dims* d, int n_sessions, const void* x, const void* B, const void* C,
                    const void* dt_raw, long sx, long sbc, long sdt, const float* A_log, const float* D,
                    const float* dt_bias, const float* conv_w, const float* conv_b, float* ssm_state,
                    void* conv_state, void* y, void* workspace, size_t workspace_bytes, void* stream) {
    m2_status st = m2::check_step_args(d, n_sessions, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b,
                                       ssm_state, conv_state, y);
    if (st != M2_OK) return st;
    const m2::Shape s = shape_of(d);
    const size_t need = m2::step_workspace_bytes(s, n_sessions);
    if (!workspace || workspace_bytes < need) return M2_EWORKSPACE;
    if (!aligned16(workspace)) return M2_EALIGN;
    st = m2::check_device();
    if (st != M2_OK) return st;
    if (n_sessions == 0) return M2_OK;

    m2::StepArgs a;
    a.s = s;
    a.S = n_sessions;
    a.x = x;
    a.B = B;
    a.C = C;
    a.dt_raw = dt_raw;
    a.sx = sx;
    a.sbc = sbc;
    a.sdt = sdt;
    a.A_log = A_log;
    a.D = D;
    a.dt_bias = dt_bias;
    a.conv_w = conv_w;
    a.conv_b = conv_b;
    a.ssm = ssm_state;
    a.conv = conv_state;
    a.y = y;
    a.ws_u = static_cast<float*>(workspace);
    a.ws_dt = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       ((size_t)n_sessions * s.CH() * 4 + 255) / 256 * 256);
    cudaError_t e = m2::launch_step(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

m2_status mamba2_step(const m2_dims* d, int n_sessions, const void* x, const void* B,
                      const void* C, const void* dt_raw, const float* A_log, const float* D,
                      const float* dt_bias, const float* conv_w, const float* conv_b,
                      float* ssm_state, void* conv_state, void* y, void* workspace,
                      size_t workspace_bytes, void* stream) {
    const long HP = d ? (long)d->nheads * d->headdim : 0, GN = d ? (long)d->ngroups * d->dstate : 0;
    return step_impl(d, n_sessions, x, B, C, dt_raw, HP, GN, d ? d->nheads : 0, A_log, D, dt_bias, conv_w,
                     conv_b, ssm_state, conv_state, y, workspace, workspace_bytes, stream);
}

m2_status mamba2_step_strided(const m2_dims* d, int n_sessions, const void* x, const void* B, const void* C,
                              const void* dt_raw, long in_row_stride, const float* A_log, const float* D,
                              const float* dt_bias, const float* conv_w, const float* conv_b, float* ssm_state,
                              void* conv_state, void* y, void* workspace, size_t workspace_bytes, void* stream) {
    if (d && (in_row_stride <= 0 ||
              (in_row_stride * (d->act == M2_BF16 ? 2 : 4)) % 16 != 0))
        return in_row_stride <= 0 ? M2_EINVAL : M2_EALIGN;
    return step_impl(d, n_sessions, x, B, C, dt_raw, in_row_stride, in_row_stride, in_row_stride, A_log, D,
                     dt_bias, conv_w, conv_b, ssm_state, conv_state, y, workspace, workspace_bytes, stream);
}

size_t mamba2_scan_workspace_bytes(const m2_dims* d, int chunk) {
    if (check_dims(d, true) != M2_OK || chunk < 1 || chunk > 128) return 0;
    return m2::scan_workspace_bytes(shape_of(d), d->batch, d->T, chunk);
}

}  // extern "C"

namespace {

// Validates a scan call and fills `a`. Returns M2_OK when there is work to
// enqueue, or a status (M2_OK with a.batch == 0 means nothing to do).
m2_status scan_setup(const m2_dims* d, const void* x, const void* B, const void* C, const void* dt_raw,
                     const float* A_log, const float* D, const float* dt_bias, const float* conv_w,
                     const float* conv_b, int chunk, const float* init_ssm, const void* init_conv, void* y,
                     float* final_ssm, void* final_conv, void* workspace, size_t workspace_bytes,
                     m2::ScanArgs* a) {
    m2_status st = check_dims(d, true);
    if (st != M2_OK) return st;
    if (chunk < 1 || chunk > 128) return M2_EINVAL;
    const void* ptrs[] = {x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, y, final_ssm, final_conv};
    const bool empty = d->batch == 0 || d->T == 0;
    for (int i = 0; i < 12; ++i) {
        // sequence inputs and y may be NULL when there are no frames
        const bool seq = (i < 4) || i == 9;
        if (!ptrs[i] && !(empty && seq)) return M2_EINVAL;
    }
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return M2_EALIGN;
    if ((init_ssm && !aligned16(init_ssm)) || (init_conv && !aligned16(init_conv))) return M2_EALIGN;
    const m2::Shape s = shape_of(d);
    const size_t need = m2::scan_workspace_bytes(s, d->batch, d->T, chunk);
    if (need && (!workspace || workspace_bytes < need)) return M2_EWORKSPACE;
    if (workspace && !aligned16(workspace)) return M2_EALIGN;
    int dev = 0;
    st = current_device(&dev);
    if (st != M2_OK) return st;
    a->s = s;
    a->batch = d->batch;
    a->T = d->T;
    a->chunk = chunk;
    a->x = x;
    a->B = B;
    a->C = C;
    a->dt_raw = dt_raw;
    a->A_log = A_log;
    a->D = D;
    a->dt_bias = dt_bias;
    a->conv_w = conv_w;
    a->conv_b = conv_b;
    a->init_ssm = init_ssm;
    a->init_conv = init_conv;
    a->y = y;
    a->final_ssm = final_ssm;
    a->final_conv = final_conv;
    a->ws = workspace;
    a->ws_bytes = workspace_bytes;
    a->err = g_dev_error_ptr[dev];
    a->lens = nullptr;
    a->fx = s.HP();
    a->fbc = s.GN();
    a->fdt = s.H;
    return M2_OK;
}

}  // namespace

#define M2_SCAN_PARAMS                                                                              \
    const m2_dims *d, const void *x, const void *B, const void *C, const void *dt_raw,              \
        const float *A_log, const float *D, const float *dt_bias, const float *conv_w,              \
        const float *conv_b, int chunk, const float *init_ssm, const void *init_conv, void *y,      \
        float *final_ssm, void *final_conv, void *workspace, size_t workspace_bytes, void *stream
#define M2_SCAN_ARGS                                                                                 \
    d, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, chunk, init_ssm, init_conv, y, final_ssm, \
        final_conv, workspace, workspace_bytes

extern "C" {

m2_status mamba2_scan_prepare_bc(M2_SCAN_PARAMS) {
    m2::ScanArgs a;
    m2_status st = scan_setup(M2_SCAN_ARGS, &a);
    if (st != M2_OK || d->batch == 0) return st;
    cudaError_t e = m2::launch_scan_prepare(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_scan_chunks(M2_SCAN_PARAMS) {
    m2::ScanArgs a;
    m2_status st = scan_setup(M2_SCAN_ARGS, &a);
    if (st != M2_OK || d->batch == 0) return st;
    cudaError_t e = m2::launch_scan_chunks(a, false, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_conv_scan_varlen(const m2_dims* d, const int* lengths, const void* x, const void* B,
                                  const void* C, const void* dt_raw, const float* A_log, const float* D,
                                  const float* dt_bias, const float* conv_w, const float* conv_b, int chunk,
                                  const float* init_ssm, const void* init_conv, void* y, float* final_ssm,
                                  void* final_conv, void* workspace, size_t workspace_bytes, void* stream) {
    if (d && d->batch > 0) {
        if (!lengths) return M2_EINVAL;
        if ((reinterpret_cast<uintptr_t>(lengths) & 3u) != 0) return M2_EALIGN;
    }
    m2::ScanArgs a;
    m2_status st = scan_setup(M2_SCAN_ARGS, &a);
    if (st != M2_OK || d->batch == 0) return st;
    a.lens = lengths;
    cudaError_t e = m2::launch_scan_prepare(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = m2::launch_scan_chunks(a, true, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_conv_scan_strided(const m2_dims* d, const void* x, const void* B, const void* C, const void* dt_raw,
                                   long in_row_stride, const float* A_log, const float* D, const float* dt_bias,
                                   const float* conv_w, const float* conv_b, int chunk, const float* init_ssm,
                                   const void* init_conv, void* y, float* final_ssm, void* final_conv,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    if (d && in_row_stride <= 0) return M2_EINVAL;
    if (d && (in_row_stride * (d->act == M2_BF16 ? 2 : 4)) % 16 != 0) return M2_EALIGN;
    m2::ScanArgs a;
    m2_status st = scan_setup(M2_SCAN_ARGS, &a);
    if (st != M2_OK || d->batch == 0) return st;
    a.fx = a.fbc = a.fdt = in_row_stride;
    cudaError_t e = m2::launch_scan_prepare(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = m2::launch_scan_chunks(a, true, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

m2_status mamba2_conv_scan(M2_SCAN_PARAMS) {
    m2::ScanArgs a;
    m2_status st = scan_setup(M2_SCAN_ARGS, &a);
    if (st != M2_OK || d->batch == 0) return st;
    cudaError_t e = m2::launch_scan_prepare(a, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = m2::launch_scan_chunks(a, true, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M2_OK : cuda_fail(e);
}

}  // extern "C"
