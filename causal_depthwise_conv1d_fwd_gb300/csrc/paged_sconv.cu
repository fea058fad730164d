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
constexpr int kRun = 16;  // tokens per warp (at most 32: one lane plans each)
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

// Tap source kinds, two bits per tap in TokenPlan::kinds.
constexpr int kTapZero = 0;    // PAD row or a position before 0: contributes nothing
constexpr int kTapX = 1;       // in this forward: x row (t - (W-1) + iw)
constexpr int kTapCache = 2;   // before this forward: cache entry at TokenPlan::off[iw]

// What every channel of a token needs: where each tap comes from, and where
// the token's input goes (ins < 0: nowhere).  Offsets exclude the channel's
// head and D offset, which each thread adds.
template <int W>
struct TokenPlan {
    int kinds;
    int64_t off[W];
    int64_t ins;
};

// Lane l of a warp resolves the plan of token t (one lane per token), so the
// per-token index loads and block-table lookups are issued once per warp and
// overlap across the warp's tokens.
template <int W>
__device__ __forceinline__ TokenPlan<W> plan_token(const PagedArgs &a, int t) {
    TokenPlan<W> p;
    p.kinds = 0;
    p.ins = -1;
#pragma unroll
    for (int iw = 0; iw < W; ++iw) p.off[iw] = 0;
    const int64_t slot = __ldg(a.slot + t);
    if (slot < 0) return p;  // PAD row: every tap is zero, nothing is inserted
    const int64_t pos = __ldg(a.pos + t);
    const int req = __ldg(a.seq_idx + t);
    const int qs = __ldg(a.qstart + t);
    const int64_t blk = slot / a.N;
    if (blk < a.num_blocks) p.ins = blk * a.cs_blk + (slot % a.N) * a.cs_n;
    else count_error(a.err);
#pragma unroll
    for (int iw = 0; iw < W; ++iw) {
        const int64_t src = pos - (W - 1) + iw;
        const int row = t - (W - 1) + iw;
        if (src < 0) continue;
        if (row >= qs) {
            if (row < 0) {
                count_error(a.err);
                continue;
            }
            p.kinds |= kTapX << (2 * iw);
            continue;
        }
        int64_t lblk = src / a.N;
        if (lblk > a.max_blocks - 1) lblk = a.max_blocks - 1;
        if (req < 0 || req >= a.bt_rows) {
            count_error(a.err);
            continue;
        }
        const int64_t pb = __ldg(a.bt + req * a.bt_r + lblk);
        if (pb < 0 || pb >= a.num_blocks) {
            count_error(a.err);
            continue;
        }
        p.kinds |= kTapCache << (2 * iw);
        p.off[iw] = pb * a.cs_blk + (src % a.N) * a.cs_n;
    }
    return p;
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
    const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
    const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
    return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

template <int W, bool SILU, bool RESID, int VEC>
__global__ void __launch_bounds__(kThreads) paged_kernel(const PagedArgs a) {
    constexpr int TILE_C = 32 * VEC;
    constexpr int G = 8;  // x rows loaded together
    __shared__ __align__(16) uint16_t s_w[W * TILE_C];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cbase = blockIdx.y * TILE_C;
    for (int i = threadIdx.x; i < W * TILE_C; i += kThreads) {
        const int cl = i / W;
        const int k = i - cl * W;
        const int c = cbase + cl;
        s_w[k * TILE_C + cl] = c < a.C ? __ldg(a.w + c * a.ws_c + k * a.ws_k) : uint16_t(0);
    }
    __syncthreads();

    const int t0 = blockIdx.x * kBlockTokens + warp * kRun;
    const int t1 = min(t0 + kRun, a.T);
    if (t0 >= t1) return;  // warp-uniform
    const int c0 = cbase + lane * VEC;
    const bool active = c0 < a.C;  // inactive lanes still take part in the shuffles

    float wt[W][VEC];
#pragma unroll
    for (int k = 0; k < W; ++k)
        reinterpret_cast<const Raw<VEC> *>(s_w + k * TILE_C)[lane].to_float(wt[k]);

    TokenPlan<W> mine;
    mine.kinds = 0;
    mine.ins = -1;
#pragma unroll
    for (int iw = 0; iw < W; ++iw) mine.off[iw] = 0;
    if (t0 + lane < t1) mine = plan_token<W>(a, t0 + lane);

    const int head = active ? c0 / a.ws : 0;
    const int64_t chan_off = static_cast<int64_t>(head) * a.cs_h + a.off_s + (active ? c0 % a.ws : 0);

    // ring[m] holds x row (t - (W-1) + m) for the token t being processed.
    float ring[W - 1][VEC];
#pragma unroll
    for (int m = 0; m < W - 1; ++m) {
        const int row = t0 - (W - 1) + m;
        if (active && row >= 0) load_plain<VEC>(a.x + row * a.xs_t + c0).to_float(ring[m]);
        else
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[m][v] = 0.0f;
    }

    for (int g = t0; g < t1; g += G) {
        Raw<VEC> xg[G];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            if (active && g + u < t1) xg[u] = load_stream<VEC>(a.x + (g + u) * a.xs_t + c0);
            else xg[u].zero();
        }
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int t = g + u;
            if (t >= t1) break;  // warp-uniform
            const int src_lane = t - t0;
            const int kinds = __shfl_sync(kFullMask, mine.kinds, src_lane);
            int64_t off[W];
#pragma unroll
            for (int iw = 0; iw < W; ++iw) off[iw] = shfl64(mine.off[iw], src_lane);
            const int64_t ins = shfl64(mine.ins, src_lane);

            float xf[VEC];
            xg[u].to_float(xf);
            if (active && ins >= 0) store_plain<VEC>(a.cache + ins + chan_off, xg[u]);

            Raw<VEC> cached[W];
#pragma unroll
            for (int iw = 0; iw < W; ++iw) {
                if (active && ((kinds >> (2 * iw)) & 3) == kTapCache)
                    cached[iw] = load_plain<VEC>(a.cache + off[iw] + chan_off);
                else
                    cached[iw].zero();
            }
            float acc[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = 0.0f;
#pragma unroll
            for (int iw = 0; iw < W; ++iw) {
                const int kind = (kinds >> (2 * iw)) & 3;
                if (kind == kTapZero) continue;
                float tap[VEC];
                if (kind == kTapX) {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) tap[v] = iw == W - 1 ? xf[v] : ring[iw][v];
                } else {
                    cached[iw].to_float(tap);
                }
#pragma unroll
                for (int v = 0; v < VEC; ++v) acc[v] = fmaf(tap[v], wt[iw][v], acc[v]);
            }
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                if (SILU) acc[v] = silu(acc[v]);
                if (RESID) acc[v] = acc[v] + xf[v];
            }
            if (active) {
                Raw<VEC> o;
                o.from_float(acc);
                store_stream<VEC>(a.out + t * a.os_t + c0, o);
            }
#pragma unroll
            for (int m = 0; m < W - 2; ++m)
#pragma unroll
                for (int v = 0; v < VEC; ++v) ring[m][v] = ring[m + 1][v];
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[W - 2][v] = xf[v];
        }
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
