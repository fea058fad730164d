// paged_sconv_fwd / paged_sconv_seq_metadata: depthwise causal short conv
// over a paged sliding-window cache, with the cache insert fused in.
//
// Semantics: vLLM Inkling sconv.py -- module docstring (cache layout
// [num_blocks, H, N, D], a stream in the D-range [off_s, off_s + ws), the
// cache holds the conv input at every absolute position), `_fused_sconv_kernel`
// part 1 (insert each real token at its slot) and part 2 (W taps ending at the
// token's absolute position: in-forward taps from x, pre-forward taps from the
// cache through block_table, no bias, SiLU, residual), and
// `_seq_metadata_kernel` (token -> request by binary search over
// query_start_loc, padded rows zero).
//
// Layout of the work: a lane owns 8 consecutive channels (one 16-byte vector,
// all in one head because ws is a multiple of 8) and walks a run of tokens;
// the in-forward taps of a token are the x rows just before it, which the
// thread already holds in registers, so x is read from memory once (plus a
// W-1 row halo per run).  Only pre-forward taps touch the cache.  The grid
// depends on T and C only, so CUDA graphs replay it unchanged.  Writes go to
// this forward's slots and reads to earlier positions, which the caller keeps
// disjoint, so one launch is race-free.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kRun = 16;  // tokens per warp
constexpr int kBlockTokens = kWarps * kRun;

struct PagedArgs {
    const uint16_t *x;
    int64_t xs_t;
    uint16_t *cache;
    int64_t cs_blk, cs_h, cs_n;
    int num_blocks, N;
    const uint16_t *w;
    int64_t ws_c, ws_k;
    uint16_t *out;
    int64_t os_t;
    const int64_t *pos;
    const int32_t *seq_idx;
    const int64_t *slot;
    const int32_t *bt;
    int64_t bt_r;
    int bt_rows, max_blocks;
    const int32_t *qstart;
    int T, off_s, ws, C;
    int *err;
};

template <int W, bool SILU, bool RESID, int VEC>
__global__ void __launch_bounds__(kThreads) paged_kernel(const PagedArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c0 = (blockIdx.y * 32 + lane) * VEC;
    if (c0 >= a.C) return;
    const int t0 = blockIdx.x * kBlockTokens + warp * kRun;
    const int t1 = min(t0 + kRun, a.T);
    if (t0 >= t1) return;

    const int head = c0 / a.ws;
    const int cd = a.off_s + c0 % a.ws;
    const int64_t head_off = static_cast<int64_t>(head) * a.cs_h + cd;

    float wt[W][VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v)
#pragma unroll
        for (int k = 0; k < W; ++k) wt[k][v] = bf16_bits(__ldg(a.w + (c0 + v) * a.ws_c + k * a.ws_k));

    // ring[m] holds x row (t - (W-1) + m) for the token t being processed.
    float ring[W - 1][VEC];
#pragma unroll
    for (int m = 0; m < W - 1; ++m) {
        const int row = t0 - (W - 1) + m;
        if (row >= 0) load_plain<VEC>(a.x + row * a.xs_t + c0).to_float(ring[m]);
        else
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[m][v] = 0.0f;
    }

    for (int t = t0; t < t1; ++t) {
        const int64_t slot = __ldg(a.slot + t);
        const int64_t pos = __ldg(a.pos + t);
        const int req = __ldg(a.seq_idx + t);
        const int qs = __ldg(a.qstart + t);
        const Raw<VEC> xr = load_stream<VEC>(a.x + t * a.xs_t + c0);
        float xf[VEC];
        xr.to_float(xf);
        const bool real = slot >= 0;

        // Part 1: insert this token's input at its slot.
        if (real) {
            const int64_t blk = slot / a.N;
            if (blk < a.num_blocks) {
                uint16_t *dst = a.cache + blk * a.cs_blk + (slot % a.N) * a.cs_n + head_off;
                store_plain<VEC>(dst, xr);
            } else if (c0 == 0) {
                count_error(a.err);
            }
        }

        // Part 2: the W taps ending at this token's absolute position.
        float acc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = 0.0f;
#pragma unroll
        for (int iw = 0; iw < W; ++iw) {
            const int64_t src = pos - (W - 1) + iw;
            const int row = t - (W - 1) + iw;
            if (!real || src < 0) continue;
            float tap[VEC];
            if (row >= qs) {
                if (row < 0) {
                    if (c0 == 0) count_error(a.err);
                    continue;
                }
#pragma unroll
                for (int v = 0; v < VEC; ++v) tap[v] = iw == W - 1 ? xf[v] : ring[iw][v];
            } else {
                int64_t lblk = src / a.N;
                if (lblk > a.max_blocks - 1) lblk = a.max_blocks - 1;
                if (req < 0 || req >= a.bt_rows) {
                    if (c0 == 0) count_error(a.err);
                    continue;
                }
                const int64_t blk = __ldg(a.bt + req * a.bt_r + lblk);
                if (blk < 0 || blk >= a.num_blocks) {
                    if (c0 == 0) count_error(a.err);
                    continue;
                }
                load_plain<VEC>(a.cache + blk * a.cs_blk + (src % a.N) * a.cs_n + head_off)
                    .to_float(tap);
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = fmaf(tap[v], wt[iw][v], acc[v]);
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            if (SILU) acc[v] = silu(acc[v]);
            if (RESID) acc[v] = acc[v] + xf[v];
        }
        Raw<VEC> o;
        o.from_float(acc);
        store_stream<VEC>(a.out + t * a.os_t + c0, o);

#pragma unroll
        for (int m = 0; m < W - 2; ++m)
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[m][v] = ring[m + 1][v];
#pragma unroll
        for (int v = 0; v < VEC; ++v) ring[W - 2][v] = xf[v];
    }
}

using PagedFn = void (*)(PagedArgs);

template <int VEC, int W>
PagedFn pick_w(bool silu, bool resid) {
    if (silu) return resid ? paged_kernel<W, true, true, VEC> : paged_kernel<W, true, false, VEC>;
    return resid ? paged_kernel<W, false, true, VEC> : paged_kernel<W, false, false, VEC>;
}

template <int VEC>
PagedFn pick_kernel(int width, bool silu, bool resid) {
    switch (width) {
        case 2: return pick_w<VEC, 2>(silu, resid);
        case 3: return pick_w<VEC, 3>(silu, resid);
        case 4: return pick_w<VEC, 4>(silu, resid);
        case 5: return pick_w<VEC, 5>(silu, resid);
    }
    return nullptr;
}

constexpr int kMetaThreads = 256;

__global__ void __launch_bounds__(kMetaThreads)
seq_metadata_kernel(const int32_t *qsl, int num_reqs, int num_actual, int num_padded,
                    int32_t *seq_idx, int32_t *query_start) {
    const int t = blockIdx.x * kMetaThreads + threadIdx.x;
    if (t >= num_padded) return;
    if (t >= num_actual) {
        seq_idx[t] = 0;
        query_start[t] = 0;
        return;
    }
    // Largest j in [0, num_reqs) with qsl[j] <= t.
    int lo = 0, hi = num_reqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(qsl + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    seq_idx[t] = lo;
    query_start[t] = __ldg(qsl + lo);
}

}  // namespace
}  // namespace ccv

extern "C" int paged_sconv_seq_metadata(const int32_t *query_start_loc, int num_reqs,
                                        int num_actual_tokens, int num_padded_tokens,
                                        int32_t *seq_idx_out, int32_t *query_start_out,
                                        int out_capacity, ccv_stream_t stream) {
    using namespace ccv;
    if (num_reqs < 0 || num_actual_tokens < 0 || out_capacity < 0) return CCV_ERR_SIZE;
    if (num_padded_tokens < num_actual_tokens) return CCV_ERR_SIZE;
    if (num_reqs == 0 && num_actual_tokens > 0) return CCV_ERR_SIZE;
    if (out_capacity < num_padded_tokens) return CCV_ERR_CAPACITY;
    if (num_padded_tokens == 0) return CCV_OK;
    if (seq_idx_out == nullptr || query_start_out == nullptr ||
        (num_actual_tokens > 0 && query_start_loc == nullptr))
        return CCV_ERR_NULL_POINTER;
    const int blocks = (num_padded_tokens + kMetaThreads - 1) / kMetaThreads;
    seq_metadata_kernel<<<blocks, kMetaThreads, 0, stream>>>(
        query_start_loc, num_reqs, num_actual_tokens, num_padded_tokens, seq_idx_out,
        query_start_out);
    return launch_status();
}

extern "C" int paged_sconv_fwd(const void *x, int64_t x_stride_t, void *cache,
                               int64_t c_stride_blk, int64_t c_stride_h, int64_t c_stride_n,
                               int num_blocks, int H, int N, int D, const void *weight,
                               int64_t w_stride_c, int64_t w_stride_w, void *out,
                               int64_t out_stride_t, const int64_t *positions,
                               const int32_t *seq_idx, const int64_t *slot_mapping,
                               const int32_t *block_table, int64_t bt_stride_r, int bt_rows,
                               int max_blocks, const int32_t *query_start, int T, int off_s,
                               int ws, int width, int silu, int residual, int *err_count,
                               ccv_stream_t stream) {
    using namespace ccv;
    if (width < kMinWidth || width > kMaxWidth) return CCV_ERR_WIDTH;
    if (T < 0 || num_blocks < 0 || H <= 0 || N <= 0 || D <= 0 || ws <= 0 || bt_rows < 0 ||
        max_blocks <= 0)
        return CCV_ERR_SIZE;
    if (off_s < 0 || off_s + ws > D) return CCV_ERR_RANGE;
    if (x_stride_t < 0 || c_stride_blk < 0 || c_stride_h < 0 || c_stride_n < 0 ||
        w_stride_c < 0 || w_stride_w < 0 || out_stride_t < 0 || bt_stride_r < 0)
        return CCV_ERR_STRIDE;
    const int64_t C64 = static_cast<int64_t>(H) * ws;
    if (C64 > 0x7fffffffLL) return CCV_ERR_SIZE;
    const int C = static_cast<int>(C64);
    if (T == 0) return CCV_OK;
    if (x == nullptr || cache == nullptr || weight == nullptr || out == nullptr ||
        positions == nullptr || seq_idx == nullptr || slot_mapping == nullptr ||
        block_table == nullptr || query_start == nullptr)
        return CCV_ERR_NULL_POINTER;
    const Extent ex = extent_of(x, T, x_stride_t, C, 1);
    const Extent eo = extent_of(out, T, out_stride_t, C, 1);
    const Extent ec = extent_of(cache, num_blocks > 0 ? num_blocks : 1, c_stride_blk, H,
                                c_stride_h, N, c_stride_n);
    const Extent ec_full{ec.lo, ec.hi + static_cast<uintptr_t>(D - 1) * 2u};
    if (overlaps(ex, eo) || overlaps(eo, ec_full)) return CCV_ERR_ALIAS;

    PagedArgs a;
    a.x = static_cast<const uint16_t *>(x);
    a.xs_t = x_stride_t;
    a.cache = static_cast<uint16_t *>(cache);
    a.cs_blk = c_stride_blk;
    a.cs_h = c_stride_h;
    a.cs_n = c_stride_n;
    a.num_blocks = num_blocks;
    a.N = N;
    a.w = static_cast<const uint16_t *>(weight);
    a.ws_c = w_stride_c;
    a.ws_k = w_stride_w;
    a.out = static_cast<uint16_t *>(out);
    a.os_t = out_stride_t;
    a.pos = positions;
    a.seq_idx = seq_idx;
    a.slot = slot_mapping;
    a.bt = block_table;
    a.bt_r = bt_stride_r;
    a.bt_rows = bt_rows;
    a.max_blocks = max_blocks;
    a.qstart = query_start;
    a.T = T;
    a.off_s = off_s;
    a.ws = ws;
    a.C = C;
    a.err = err_count;

    const bool vec = ws % 8 == 0 && off_s % 8 == 0 && aligned16(x) && aligned16(out) &&
                     aligned16(cache) && x_stride_t % 8 == 0 && out_stride_t % 8 == 0 &&
                     c_stride_blk % 8 == 0 && c_stride_h % 8 == 0 && c_stride_n % 8 == 0;
    const int vw = vec ? 8 : 1;
    PagedFn fn = vec ? pick_kernel<8>(width, silu != 0, residual != 0)
                     : pick_kernel<1>(width, silu != 0, residual != 0);
    const dim3 grid(static_cast<unsigned>((T + kBlockTokens - 1) / kBlockTokens),
                    static_cast<unsigned>((C + 32 * vw - 1) / (32 * vw)));
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    fn<<<grid, kThreads, 0, stream>>>(a);
    return launch_status();
}
