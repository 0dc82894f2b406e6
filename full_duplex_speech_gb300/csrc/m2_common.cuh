// Shared device helpers of the Mamba2 mixer-core kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

namespace m2 {

// Activation element types: bf16 travels as its 16-bit pattern.
struct bf16_t { uint16_t bits; };

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// 8 consecutive activations -> fp32 (16 B of bf16 or 32 B of fp32).
// Read-only loads issued exactly where they stand. A volatile asm statement
// with a memory clobber is not moved by the compiler, so a load placed ahead
// of a barrier or a long wait is in flight during it instead of being sunk
// to its first use.
__device__ __forceinline__ uint4 ldg_pinned_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}
__device__ __forceinline__ float4 ldg_pinned_f4(const void* p) {
    float4 r;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}
__device__ __forceinline__ float ldg_pinned_f32(const void* p) {
    float r;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p) : "memory");
    return r;
}
__device__ __forceinline__ uint16_t ldg_pinned_u16(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p) : "memory");
    return r;
}

template <typename TA> struct Act8;

template <> struct Act8<bf16_t> {
    uint4 raw;
    __device__ __forceinline__ void load(const void* base, size_t elem) {
        raw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + elem));
    }
    __device__ __forceinline__ void load_pinned(const void* base, size_t elem) {
        raw = ldg_pinned_u4(reinterpret_cast<const uint16_t*>(base) + elem);
    }
    // plain (coherent) load, for data that this kernel also writes
    __device__ __forceinline__ void load_rw(const void* base, size_t elem) {
        raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + elem);
    }
    __device__ __forceinline__ void store(void* base, size_t elem) const {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + elem) = raw;
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t w = (&raw.x)[j >> 1];
        return bf16_bits_to_float((j & 1) ? (w >> 16) : (w & 0xFFFFu));
    }
};

template <> struct Act8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const void* base, size_t elem) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem);
        a = __ldg(p);
        b = __ldg(p + 1);
    }
    __device__ __forceinline__ void load_pinned(const void* base, size_t elem) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem);
        a = ldg_pinned_f4(p);
        b = ldg_pinned_f4(p + 1);
    }
    __device__ __forceinline__ void load_rw(const void* base, size_t elem) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem);
        a = p[0];
        b = p[1];
    }
    __device__ __forceinline__ void store(void* base, size_t elem) const {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem);
        p[0] = a;
        p[1] = b;
    }
    __device__ __forceinline__ float get(int j) const { return j < 4 ? (&a.x)[j] : (&b.x)[j - 4]; }
};

template <typename TA> __device__ __forceinline__ void store_act(void* base, size_t elem, float v);
template <> __device__ __forceinline__ void store_act<bf16_t>(void* base, size_t elem, float v) {
    reinterpret_cast<uint16_t*>(base)[elem] = float_to_bf16_bits(v);
}
template <> __device__ __forceinline__ void store_act<float>(void* base, size_t elem, float v) {
    reinterpret_cast<float*>(base)[elem] = v;
}

template <typename TA> __device__ __forceinline__ float load_act(const void* base, size_t elem);
template <> __device__ __forceinline__ float load_act<bf16_t>(const void* base, size_t elem) {
    return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + elem));
}
template <> __device__ __forceinline__ float load_act<float>(const void* base, size_t elem) {
    return __ldg(reinterpret_cast<const float*>(base) + elem);
}

// One activation element as stored (bf16 bits or fp32), loaded where it
// stands and not converted yet, so that nothing waits on it until raw_to_f32.
template <typename TA> using ActRaw = typename std::conditional<sizeof(TA) == 2, uint16_t, float>::type;
template <typename TA> __device__ __forceinline__ ActRaw<TA> load_raw_pinned(const void* base, size_t elem) {
    if constexpr (sizeof(TA) == 2)
        return ldg_pinned_u16(reinterpret_cast<const uint16_t*>(base) + elem);
    else
        return ldg_pinned_f32(reinterpret_cast<const float*>(base) + elem);
}
template <typename TA> __device__ __forceinline__ float raw_to_f32(ActRaw<TA> r) {
    if constexpr (sizeof(TA) == 2)
        return bf16_bits_to_float(r);
    else
        return r;
}

// softplus(z) = log(1 + e^z), evaluated without overflow on either side.
__device__ __forceinline__ float softplus_f32(float z) {
    return z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
}

// SiLU(u) = u * sigmoid(u) = u / (1 + e^-u), with the fast exponential and
// division intrinsics (relative error ~1e-7 here). Where the divisor is huge (u below about -87) the fast
// division returns 0 (its reciprocal of a value above 2^126, or of +inf, is
// 0), where the exact result is below 1e-36 in magnitude.
__device__ __forceinline__ float silu_fast(float u) { return __fdividef(u, 1.f + __expf(-u)); }

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start before its predecessor in the stream finishes;
// pdl_wait() blocks until the predecessor has completed and its writes are
// visible (a no-op without the launch attribute). pdl_trigger() lets the
// next such kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Codes written to the device error word: a bounded wait that ran out, or an
// input that only the device sees and that the kernel refused.
enum : unsigned int {
    ERR_NONE = 0,
    ERR_MBAR_TIMEOUT_LOAD = 0x101,
    ERR_MBAR_TIMEOUT_MMA = 0x102,
    ERR_TMEM_ALLOC = 0x103,
    ERR_ATTN_LENGTH = 0x104,  // a cached length outside [0, max_len)
};

}  // namespace m2
