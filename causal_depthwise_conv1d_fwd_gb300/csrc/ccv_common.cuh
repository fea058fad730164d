// Shared device and host helpers of the ccv CUDA library (sm_103a).
#pragma once

#include <atomic>
#include <utility>

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

// ------------------------------------------ programmatic dependent launch ----
//
// Every kernel of the library is launched with programmatic stream
// serialization (launch_pdl below): it may be scheduled while the previous
// kernel of the stream is still finishing, so its launch and block set-up
// overlap that kernel's tail.  Such a kernel must not touch global memory --
// no read and no write, since the previous kernel may still read what this
// one overwrites -- before wait_prior_grid(), which returns once the previous
// kernel has completed and its writes are visible.  release_next_grid() lets
// the next kernel of the stream be scheduled; it only ever starts early, and
// it waits in its own wait_prior_grid() for this kernel to complete.  Without
// a programmatic predecessor the wait returns at once.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void release_next_grid() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// The weights of 8 consecutive channels c0..c0+7 as tap-major bf16x2 words:
// wpk[k] word q holds (w[c0+2q][k], w[c0+2q+1][k]).  When the weight matrix
// is contiguous (dim, W) and 16-byte aligned, the thread's 8W values are W
// 16-byte loads regrouped with one byte permute per word; otherwise they are
// gathered one by one.  Channels at or beyond `dim` read as 0.
template <int W>
__device__ __forceinline__ void load_weights8(const uint16_t *w, int64_t ws_d, int64_t ws_k, int c0,
                                              int dim, bool contiguous, uint4 (&wpk)[W]) {
    uint32_t words[W][4];
    if (contiguous && c0 + 8 <= dim) {
        uint32_t raw[4 * W];  // elements c0*W .. c0*W + 8W - 1, two per word
        const uint4 *src = reinterpret_cast<const uint4 *>(w + static_cast<int64_t>(c0) * W);
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const uint4 v = __ldg(src + i);
            raw[4 * i] = v.x;
            raw[4 * i + 1] = v.y;
            raw[4 * i + 2] = v.z;
            raw[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int k = 0; k < W; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e1 = (2 * q) * W + k, e2 = (2 * q + 1) * W + k;
                const uint32_t sel = ((e1 & 1) ? 0x32u : 0x10u) | ((e2 & 1) ? 0x7600u : 0x5400u);
                words[k][q] = __byte_perm(raw[e1 >> 1], raw[e2 >> 1], sel);
            }
    } else {
#pragma unroll
        for (int k = 0; k < W; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ca = c0 + 2 * q, cb = ca + 1;
                const uint32_t lo = ca < dim ? __ldg(w + ca * ws_d + k * ws_k) : 0u;
                const uint32_t hi = cb < dim ? __ldg(w + cb * ws_d + k * ws_k) : 0u;
                words[k][q] = lo | (hi << 16);
            }
    }
#pragma unroll
    for (int k = 0; k < W; ++k) wpk[k] = make_uint4(words[k][0], words[k][1], words[k][2], words[k][3]);
}

// Bias of channels c0..c0+7 as fp32 (0 when absent or beyond dim).
__device__ __forceinline__ void load_bias8(const uint16_t *bias, int c0, int dim, bool aligned,
                                           float (&bs)[8]) {
    if (bias == nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) bs[i] = 0.0f;
        return;
    }
    if (aligned && c0 + 8 <= dim) {
        Raw<8> r;
        r.v = __ldg(reinterpret_cast<const uint4 *>(bias + c0));
        r.to_float(bs);
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) bs[i] = c0 + i < dim ? bf16_bits(__ldg(bias + c0 + i)) : 0.0f;
}

// ------------------------------------------------------------ host side ----

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CCV_OK : static_cast<int>(e);
}

// Launch `kernel` on `stream` with programmatic stream serialization (see
// wait_prior_grid).  Returns CCV_OK or the cudaError_t of the launch.
template <typename... Params, typename... Args>
inline int launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) {
        cudaGetLastError();  // the error is returned; do not leave it for the next call
        return static_cast<int>(e);
    }
    return launch_status();
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
// The caches below may be filled by several host threads at once; every
// writer stores the same value, and relaxed atomics make that well defined.
inline int current_device_sms(int *device_out = nullptr) {
    static std::atomic<int> cache[kMaxDevices];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    if (device_out) *device_out = dev;
    if (dev < 0 || dev >= kMaxDevices) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    int cached = cache[dev].load(std::memory_order_relaxed);
    if (cached == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached = n > 0 ? n : 1;
        cache[dev].store(cached, std::memory_order_relaxed);
    }
    return cached;
}

// Prepare `fn` to run with `threads` threads and `bytes` of dynamic shared
// memory on the current device and return how many of its blocks fit on one
// SM (0 on error, with *err set).  The attribute and the occupancy are
// computed once per (kernel, device) and cached, so later calls -- including
// ones made while a CUDA graph is being captured -- only read the cache.
template <auto kKernel>
inline int resident_blocks(int threads, size_t bytes, int dev, cudaError_t *err) {
    static std::atomic<int> cache[kMaxDevices];  // one cache per kernel instantiation
    const auto fn = kKernel;
    *err = cudaSuccess;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable) {
        const int cached = cache[dev].load(std::memory_order_relaxed);
        if (cached > 0) return cached;
    }
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    int blocks = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, threads, bytes);
    if (e != cudaSuccess || blocks <= 0) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        return 0;
    }
    if (cacheable) cache[dev].store(blocks, std::memory_order_relaxed);
    return blocks;
}

}  // namespace ccv
