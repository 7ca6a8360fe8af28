// Shared device helpers of libattn (CUDA side only; the CPU oracle shares nothing with this).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "libattn.h"

namespace attn {

// Device error word values (written with atomicMax so the worst one stays).
enum : unsigned {
    kDevOk = 0,
    kDevCheck = 1,     // device-side consistency check failed
    kDevTimeout = 2,   // a bounded wait ran out
};

// One second: the limit of every spin-wait in these kernels.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_device_error(unsigned *err, unsigned code) {
    if (err) atomicMax(err, code);
}

// bf16 <-> f32 (bit-level; RNE for the narrowing).
__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low 16 bits), .y = hi
    return *reinterpret_cast<uint32_t *>(&h);
}

// f16 <-> f32 (RNE for the narrowing).
__device__ __forceinline__ float f16_lo(uint32_t packed) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(packed & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t packed) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(packed >> 16)));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);               // .x = lo (low 16 bits), .y = hi
    return *reinterpret_cast<uint32_t *>(&h);
}

// The two 16-bit storage types behind one interface: H16<true> is f16,
// H16<false> bf16.
template <bool F16> struct H16;
template <> struct H16<false> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float lo(uint32_t w) { return bf16_lo(w); }
    static __device__ __forceinline__ float hi(uint32_t w) { return bf16_hi(w); }
    static __device__ __forceinline__ uint32_t pack(float a, float b) { return pack_bf16x2(a, b); }
    static __device__ __forceinline__ T from(float x) { return __float2bfloat16_rn(x); }
    static constexpr uint16_t kOne = 0x3F80;             // 1.0
};
template <> struct H16<true> {
    using T = __half;
    static __device__ __forceinline__ float lo(uint32_t w) { return f16_lo(w); }
    static __device__ __forceinline__ float hi(uint32_t w) { return f16_hi(w); }
    static __device__ __forceinline__ uint32_t pack(float a, float b) { return pack_f16x2(a, b); }
    static __device__ __forceinline__ T from(float x) { return __float2half_rn(x); }
    static constexpr uint16_t kOne = 0x3C00;             // 1.0
};

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float load(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void store(__half *p, float x) { *p = __float2half_rn(x); }
};

// NATTEN boundary window along one axis (candle PR #11, "kernel exceeds grid
// extent"): k_eff = min(k, n); window [start, start + k_eff) with
// start = clamp(i - k/2, 0, n - k_eff).  Every neighborhood kernel and the
// window-start export call this one function.
__host__ __device__ __forceinline__ int na_window_start(int i, int n, int k) {
    const int keff = k < n ? k : n;
    int st = i - k / 2;
    st = st < 0 ? 0 : st;
    return st > n - keff ? n - keff : st;
}

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace attn
