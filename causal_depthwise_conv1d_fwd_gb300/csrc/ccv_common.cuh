// Shared device and host helpers of the ccv CUDA library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ccv.h"

namespace ccv {

constexpr int kMinWidth = 2;
constexpr int kMaxWidth = 5;
constexpr unsigned kFullMask = 0xffffffffu;

// ------------------------------------------------------------ bf16 data ----

// A bf16 is the upper half of a binary32, so widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round two floats to bf16 (round-to-nearest-even) and pack them, lo first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint16_t round_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// VEC consecutive bf16 values as raw bits: one 16-byte vector or one element.
template <int VEC> struct Raw;
template <> struct Raw<8> {
    uint4 v;
    __device__ __forceinline__ void zero() { v = make_uint4(0u, 0u, 0u, 0u); }
    __device__ __forceinline__ void to_float(float (&f)[8]) const {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ __forceinline__ void from_float(const float (&f)[8]) {
        v.x = pack_bf16x2(f[0], f[1]);
        v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]);
        v.w = pack_bf16x2(f[6], f[7]);
    }
    __device__ __forceinline__ uint16_t elem(int i) const {
        const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
        return uint16_t((i & 1) ? (w >> 16) : (w & 0xffffu));
    }
    __device__ __forceinline__ void set_elem(int i, uint16_t b) {
        uint32_t &w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
        w = (i & 1) ? ((w & 0x0000ffffu) | (uint32_t(b) << 16)) : ((w & 0xffff0000u) | b);
    }
};
template <> struct Raw<1> {
    uint16_t v;
    __device__ __forceinline__ void zero() { v = 0; }
    __device__ __forceinline__ void to_float(float (&f)[1]) const { f[0] = bf16_bits(v); }
    __device__ __forceinline__ void from_float(const float (&f)[1]) { v = round_bf16(f[0]); }
    __device__ __forceinline__ uint16_t elem(int) const { return v; }
    __device__ __forceinline__ void set_elem(int, uint16_t b) { v = b; }
};

// Loads of data read once (x): read-only path.  Stores of data written once
// (out): streaming hint so they do not displace reusable lines in L2.
template <int VEC>
__device__ __forceinline__ Raw<VEC> load_stream(const uint16_t *p) {
    Raw<VEC> r;
    if constexpr (VEC == 8) r.v = __ldg(reinterpret_cast<const uint4 *>(p));
    else r.v = __ldg(reinterpret_cast<const unsigned short *>(p));
    return r;
}
// Loads that another thread block may also read (halo rows): default caching.
template <int VEC>
__device__ __forceinline__ Raw<VEC> load_plain(const uint16_t *p) {
    Raw<VEC> r;
    if constexpr (VEC == 8) r.v = *reinterpret_cast<const uint4 *>(p);
    else r.v = *p;
    return r;
}
template <int VEC>
__device__ __forceinline__ void store_stream(uint16_t *p, const Raw<VEC> &r) {
    if constexpr (VEC == 8) __stcs(reinterpret_cast<uint4 *>(p), r.v);
    else *p = r.v;
}
template <int VEC>
__device__ __forceinline__ void store_plain(uint16_t *p, const Raw<VEC> &r) {
    if constexpr (VEC == 8) *reinterpret_cast<uint4 *>(p) = r.v;
    else *p = r.v;
}

// ------------------------------------------------------------- numerics ----

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// SiLU v / (1 + exp(-v)); for v < -88 exp overflows to inf and the result is -0.
__device__ __forceinline__ float silu(float v) { return v * rcp_approx(1.0f + __expf(-v)); }

__device__ __forceinline__ void count_error(int *err_count) {
    if (err_count) atomicAdd(err_count, 1);
}

// Floor division for a possibly negative numerator and a positive divisor.
__device__ __forceinline__ int floor_div(int a, int b) {
    int q = a / b;
    return (a % b != 0 && a < 0) ? q - 1 : q;
}

// ------------------------------------------------------------ host side ----

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CCV_OK : static_cast<int>(e);
}

// Byte range [lo, hi] covered by a strided 2-D or 3-D bf16 view (strides >= 0).
struct Extent {
    uintptr_t lo, hi;
};
inline Extent extent_of(const void *p, int64_t n0, int64_t s0, int64_t n1, int64_t s1,
                        int64_t n2 = 1, int64_t s2 = 0) {
    uintptr_t base = reinterpret_cast<uintptr_t>(p);
    int64_t last = (n0 - 1) * s0 + (n1 - 1) * s1 + (n2 - 1) * s2;
    return Extent{base, base + static_cast<uintptr_t>(last) * 2u + 1u};
}
inline bool overlaps(const Extent &a, const Extent &b) { return a.lo <= b.hi && b.lo <= a.hi; }

constexpr int kMaxDevices = 64;

// Streaming multiprocessors of the current device (cached per device).
inline int current_device_sms(int *device_out = nullptr) {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    if (device_out) *device_out = dev;
    if (dev < 0 || dev >= kMaxDevices) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

// Prepare `fn` to run with `threads` threads and `bytes` of dynamic shared
// memory on the current device and return how many of its blocks fit on one
// SM (0 on error, with *err set).  The attribute and the occupancy are
// computed once per (kernel, device) and cached, so later calls -- including
// ones made while a CUDA graph is being captured -- only read the cache.
template <auto kKernel>
inline int resident_blocks(int threads, size_t bytes, int dev, cudaError_t *err) {
    static int cache[kMaxDevices] = {0};  // one cache per kernel instantiation
    const auto fn = kKernel;
    *err = cudaSuccess;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable && cache[dev] > 0) return cache[dev];
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    int blocks = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, threads, bytes);
    if (e != cudaSuccess || blocks <= 0) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        return 0;
    }
    if (cacheable) cache[dev] = blocks;
    return blocks;
}

}  // namespace ccv
