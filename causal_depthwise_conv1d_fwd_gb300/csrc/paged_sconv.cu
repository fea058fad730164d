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
// Layout of the work: in the vector kernel a lane owns 8 consecutive
// channels (one 16-byte vector, all in one head because ws is a multiple of
// 8) and a warp a run of 8 tokens; the scalar fallback has one channel per
// lane and runs of 8.  One lane per token resolves the token's tap sources
// once (shift/mask block arithmetic for power-of-two block sizes) and shares
// them by shuffle.  In-forward taps are x rows; only pre-forward taps touch
// the cache.  The grid depends on T and C only, so CUDA graphs replay it
// unchanged.  Writes go to this forward's slots and reads to earlier
// positions, which the caller keeps disjoint, so one launch is race-free.
#include "ccv_common.cuh"
#include "ccv_math2.cuh"
#include "ccv_pipeline.cuh"

namespace ccv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kRun = 8;  // tokens per warp (at most 32: one lane plans each)
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
    int n_shift;  // log2(N) when N is a power of two, else -1
    int w_vec;    // weights contiguous [C, W] and 16-byte aligned
    int *err;
    // With own_meta the kernel finds each token's request and first x-row
    // from qsl itself, exactly as paged_sconv_seq_metadata does, instead of
    // reading seq_idx and qstart, and writes them to seq_out / qs_out when
    // set.  qsl is read only when num_reqs > 0.
    int own_meta;
    const int32_t *qsl;
    int num_reqs, num_actual;
    int32_t *seq_out, *qs_out;
};

// The fields that differ between the conv streams of one layer (each stream
// owns its own x, weights, output and D-range of the shared cache).
constexpr int kMaxStreams = 8;
struct StreamFields {
    const uint16_t *x;
    int64_t xs_t;
    const uint16_t *w;
    int64_t ws_c, ws_k;
    uint16_t *out;
    int64_t os_t;
    int off_s, ws, C, w_vec;
};

// One launch of the vector kernel: the shared arguments, and for a fused
// multi-stream launch (gridDim.z > 1) the streams blockIdx.z selects.
struct PagedLaunch {
    PagedArgs a;
    StreamFields s[kMaxStreams];
};

__host__ __device__ __forceinline__ void apply_stream(PagedArgs &a, const StreamFields &f) {
    a.x = f.x;
    a.xs_t = f.xs_t;
    a.w = f.w;
    a.ws_c = f.ws_c;
    a.ws_k = f.ws_k;
    a.out = f.out;
    a.os_t = f.os_t;
    a.off_s = f.off_s;
    a.ws = f.ws;
    a.C = f.C;
    a.w_vec = f.w_vec;
}

// (block, offset) of a non-negative flat position in blocks of N.
__device__ __forceinline__ void split_pos(const PagedArgs &a, int64_t p, int64_t &blk, int64_t &off) {
    if (a.n_shift >= 0) {
        blk = p >> a.n_shift;
        off = p & ((int64_t(1) << a.n_shift) - 1);
    } else {
        blk = p / a.N;
        off = p - blk * a.N;
    }
}

// Tap source kinds, two bits per tap in TokenPlan::kinds.
constexpr int kTapZero = 0;    // PAD row or a position before 0: contributes nothing
constexpr int kTapX = 1;       // in this forward: x row (t - (W-1) + iw)
constexpr int kTapCache = 2;   // before this forward: cache entry at TokenPlan::off[iw]
// A PAD row's kinds: every tap field zero, plus a flag bit above them.
constexpr int kPadRow = 1 << 30;

// What every channel of a token needs: where each tap comes from, and where
// the token's input goes (ins < 0: nowhere).  Offsets exclude the channel's
// head and D offset, which each thread adds.
template <int W>
struct TokenPlan {
    int kinds;
    int64_t off[W];
    int64_t ins;
};

// The four per-token index values.
struct TokenMeta {
    int64_t slot, pos;
    int req, qs;
};

// Request and first x-row of token t from query_start_loc, with the steps
// of the metadata kernel: the largest j in [0, num_reqs) with qsl[j] <= t
// (0 if none) by the same binary search, and qsl[j]; rows from num_actual
// on get 0 and 0.  Warp-cooperative: every lane of the warp calls it for its
// own token.  Up to 32 requests lane i holds qsl[i] and the search reads it
// by shuffle (one round trip for the warp); beyond, each lane searches
// global memory on its own.
__device__ __forceinline__ void resolve_request(const PagedArgs &a, int t, bool valid, TokenMeta &m) {
    const int lane = threadIdx.x & 31;
    int lo = 0;
    if (a.num_reqs > 0 && a.num_reqs <= 32) {  // warp-uniform
        const int q = lane < a.num_reqs ? __ldg(a.qsl + lane) : 0;
        int hi = a.num_reqs - 1;
        // A fixed count of steps keeps every lane in the shuffles; five
        // halvings settle any window of up to 32 entries.
#pragma unroll
        for (int step = 0; step < 6; ++step) {
            const int mid = (lo + hi + 1) >> 1;
            const int qm = __shfl_sync(kFullMask, q, mid);
            if (lo < hi) {
                if (qm <= t) lo = mid;
                else hi = mid - 1;
            }
        }
        m.qs = __shfl_sync(kFullMask, q, lo);
    } else if (a.num_reqs > 32) {
        int hi = a.num_reqs - 1;
        if (valid && t < a.num_actual) {
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(a.qsl + mid) <= t) lo = mid;
                else hi = mid - 1;
            }
            m.qs = __ldg(a.qsl + lo);
        }
    }
    m.req = lo;
    if (!valid || t >= a.num_actual) {
        m.req = 0;
        m.qs = 0;
    }
}

// The four per-token index values; a token past T reads as a PAD row.
// Every lane of the warp calls this (the request search may be shared).
__device__ __forceinline__ TokenMeta load_meta(const PagedArgs &a, int t, bool valid) {
    TokenMeta m{-1, 0, 0, 0};
    if (valid) {
        m.slot = __ldg(a.slot + t);
        m.pos = __ldg(a.pos + t);
        if (!a.own_meta) {
            m.req = __ldg(a.seq_idx + t);
            m.qs = __ldg(a.qstart + t);
        }
    }
    if (a.own_meta) resolve_request(a, t, valid, m);
    return m;
}

// Write the token's request and first x-row where the caller asked for them
// (one channel block per token writes).
__device__ __forceinline__ void store_meta(const PagedArgs &a, int t, bool valid, const TokenMeta &m) {
    if (!valid) return;
    if (a.seq_out != nullptr) a.seq_out[t] = m.req;
    if (a.qs_out != nullptr) a.qs_out[t] = m.qs;
}

// Lane l of a warp resolves the plan of token t (one lane per token), so the
// per-token index loads and block-table lookups are issued once per warp and
// overlap across the warp's tokens.
template <int W>
__device__ __forceinline__ TokenPlan<W> plan_token(const PagedArgs &a, int t, const TokenMeta &m) {
    TokenPlan<W> p;
    p.kinds = 0;
    p.ins = -1;
#pragma unroll
    for (int iw = 0; iw < W; ++iw) p.off[iw] = 0;
    const int64_t slot = m.slot, pos = m.pos;
    const int req = m.req, qs = m.qs;
    if (slot < 0) {  // PAD row: every tap is zero, nothing is inserted
        p.kinds = kPadRow;
        return p;
    }
    int64_t blk, boff;
    split_pos(a, slot, blk, boff);
    if (blk < a.num_blocks) p.ins = blk * a.cs_blk + boff * a.cs_n;
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
        int64_t lblk, soff;
        split_pos(a, src, lblk, soff);
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
        p.off[iw] = pb * a.cs_blk + soff * a.cs_n;
    }
    return p;
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
    const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
    const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
    return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// Fallback for unaligned or odd-width layouts: one channel per lane.
template <int W, bool SILU, bool RESID>
__global__ void __launch_bounds__(kThreads) paged_scalar_kernel(const PagedArgs a) {
    release_next_grid();
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kBlockTokens + warp * kRun;
    const int t1 = min(t0 + kRun, a.T);
    if (t0 >= t1) return;  // warp-uniform
    const int c0 = blockIdx.y * 32 + lane;
    const bool active = c0 < a.C;  // inactive lanes still take part in the shuffles

    float ring[W - 1];
#pragma unroll
    for (int m = 0; m < W - 1; ++m) {
        const int row = t0 - (W - 1) + m;
        ring[m] = active && row >= 0 ? bf16_bits(a.x[row * a.xs_t + c0]) : 0.0f;
    }
    uint16_t xg[kRun];
#pragma unroll
    for (int u = 0; u < kRun; ++u) xg[u] = active && t0 + u < t1 ? __ldg(a.x + (t0 + u) * a.xs_t + c0) : 0;

    const TokenMeta meta = load_meta(a, t0 + lane, t0 + lane < t1);
    if (blockIdx.y == 0) store_meta(a, t0 + lane, t0 + lane < t1, meta);
    const TokenPlan<W> mine = plan_token<W>(a, t0 + lane, meta);

    const int head = active ? c0 / a.ws : 0;
    const int64_t chan_off = static_cast<int64_t>(head) * a.cs_h + a.off_s + (active ? c0 % a.ws : 0);
    float wt[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wt[k] = active ? bf16_bits(__ldg(a.w + c0 * a.ws_c + k * a.ws_k)) : 0.0f;

#pragma unroll
    for (int u = 0; u < kRun; ++u) {
        const int t = t0 + u;
        if (t >= t1) break;  // warp-uniform
        const int kinds = __shfl_sync(kFullMask, mine.kinds, u);
        int64_t off[W];
#pragma unroll
        for (int iw = 0; iw < W; ++iw) off[iw] = shfl64(mine.off[iw], u);
        const int64_t ins = shfl64(mine.ins, u);
        const float xf = bf16_bits(xg[u]);
        if (active && ins >= 0) a.cache[ins + chan_off] = xg[u];
        float acc = 0.0f;
#pragma unroll
        for (int iw = 0; iw < W; ++iw) {
            const int kind = (kinds >> (2 * iw)) & 3;
            if (kind == kTapZero) continue;
            const float tap = kind == kTapX ? (iw == W - 1 ? xf : ring[iw < W - 1 ? iw : 0])
                                            : bf16_bits(a.cache[off[iw] + chan_off]);
            acc = fmaf(tap, wt[iw], acc);
        }
        if (SILU) acc = silu(acc);
        if (RESID) acc = acc + xf;
        if (active) a.out[t * a.os_t + c0] = round_bf16(acc);
#pragma unroll
        for (int m = 0; m < W - 2; ++m) ring[m] = ring[m + 1];
        ring[W - 2] = xf;
    }
}

// Row kernel: a block covers a run of kRowRun tokens across up to
// kRowMaxThreads * 8 channels, a thread per 8 consecutive channels (one
// 16-byte vector, all in one head because ws is a multiple of 8).  The first
// warp's token metadata and every thread's weights are requested first;
// then each thread streams its x vectors of the run and of the W-1 rows
// before it into a private ring of shared-memory slots with asynchronous
// copies (it reads back only its own slots, so its own wait is the only
// synchronisation for them).  The first warp resolves every token's plan
// once -- tap sources through the block table, insert slot -- into shared
// memory, and one barrier publishes it to the block.  When every token of
// the run takes all W taps from x and has an insert slot, or is a PAD row
// (an interior stretch of a prefill, the usual case), a straight loop keeps
// the taps in a register ring of raw bf16 rows; otherwise each token
// follows its plan (x rows from the ring, cache taps from global memory).
// Taps are native bf16 x bf16 + fp32 FMAs on packed weights; the residual
// enters the same way (x * 1 + act, one rounding).  Blocks of 128 threads
// (two per 2048-channel run) spread the runs more evenly over the SMs than
// one 256-thread block per run (measured faster).
constexpr int kRowRun = 8;           // tokens per block (at most 32: one planning lane each)
constexpr int kRowMaxThreads = 128;  // 1024 channels per block
constexpr int kStageGroup = 4;       // staged rows per asynchronous-copy group

// One run's plans, written by the first warp and read by every thread.
template <int W>
struct RunPlan {
    int64_t ins[kRowRun];
    int64_t off[kRowRun][W];
    int kinds[kRowRun];
    int all_x;
};

template <int W>
constexpr int row_slots() {
    return kRowRun + W - 1;
}

template <int W>
constexpr int all_x_kinds() {
    int k = 0;
    for (int iw = 0; iw < W; ++iw) k |= kTapX << (2 * iw);
    return k;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

constexpr uint32_t kBf16OnePair = 0x3f803f80u;  // (1.0, 1.0) as bf16x2

// SiLU, then the residual (x of the token times 1 plus the activation: one
// rounding, the same value as the fp32 sum), then bf16 rounding of one
// thread's 8 outputs.
template <bool SILU, bool RESID>
__device__ __forceinline__ uint4 finish_row(float (&acc)[8], const uint4 &xr) {
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float lo = acc[2 * q], hi = acc[2 * q + 1];
        if (SILU) unpack2(silu2(pack2(lo, hi)), lo, hi);
        if (RESID) fma_bf16x2(lo, hi, word_of(xr, q), kBf16OnePair);
        o[q] = f32x2_to_bf16x2(pack2(lo, hi));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// One token whose W taps all come from x: ring[0..W-2] (oldest first) and
// xr, native bf16 x bf16 + fp32 FMAs from zero (no bias), taps in order.
template <int W, bool SILU, bool RESID>
__device__ __forceinline__ uint4 paged_row(const uint4 (&wpk)[W], const uint4 (&ring)[W - 1],
                                           const uint4 &xr) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        fma_bf16x2_init(acc[2 * q], acc[2 * q + 1], word_of(ring[0], q), word_of(wpk[0], q), 0.0f, 0.0f);
#pragma unroll
    for (int k = 1; k < W; ++k) {
        const uint4 &u = k < W - 1 ? ring[k < W - 1 ? k : 0] : xr;
#pragma unroll
        for (int q = 0; q < 4; ++q) fma_bf16x2(acc[2 * q], acc[2 * q + 1], word_of(u, q), word_of(wpk[k], q));
    }
    return finish_row<SILU, RESID>(acc, xr);
}

template <int W, bool SILU, bool RESID>
__global__ void __launch_bounds__(kRowMaxThreads, 8) paged_row_kernel(const PagedLaunch pl) {
    extern __shared__ uint4 stage[];  // [row_slots<W>()][blockDim.x]
    __shared__ RunPlan<W> plan;
    constexpr int R = row_slots<W>();
    release_next_grid();
    wait_prior_grid();
    PagedArgs a = pl.a;
    if (gridDim.z > 1) {
        // constant indices only: no dynamic indexing into the parameters
        switch (blockIdx.z) {
            case 0: apply_stream(a, pl.s[0]); break;
            case 1: apply_stream(a, pl.s[1]); break;
            case 2: apply_stream(a, pl.s[2]); break;
            case 3: apply_stream(a, pl.s[3]); break;
            case 4: apply_stream(a, pl.s[4]); break;
            case 5: apply_stream(a, pl.s[5]); break;
            case 6: apply_stream(a, pl.s[6]); break;
            default: apply_stream(a, pl.s[7]); break;
        }
    }
    const int nthreads = blockDim.x;
    const int tile_c = nthreads * 8;
    if (static_cast<int>(blockIdx.y) * tile_c >= a.C) return;  // block-uniform: this stream is narrower
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * kRowRun;
    const int n = min(kRowRun, a.T - t0);  // >= 1: the grid covers T exactly
    const int c0 = blockIdx.y * tile_c + tid * 8;
    const bool active = c0 < a.C;
    uint4 *xs = stage + tid;  // row m of the run's window at xs[m * nthreads]

    // The first warp's token metadata and every thread's weights go out
    // first: the plan waits on the one and the block's barrier on the other
    // (the weights are regrouped as they arrive), and queued behind the x
    // streams of all blocks, which go out at once, they would wait for all
    // of them.  Then the x stream: rows t0-(W-1) .. t0+n-1, in commit groups
    // of kStageGroup rows so the straight loop can start on the first ones.
    TokenMeta meta{-1, 0, 0, 0};
    if (tid < 32) meta = load_meta(a, t0 + tid, tid < n);  // lane u: token t0 + u
    uint4 wpk[W];
    load_weights8<W>(a.w, a.ws_c, a.ws_k, active ? c0 : 0, a.C, a.w_vec, wpk);
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int row = t0 - (W - 1) + m;
        if (active && row >= 0 && row < t0 + n) cp_async16(xs + m * nthreads, a.x + row * a.xs_t + c0);
        else xs[m * nthreads] = make_uint4(0u, 0u, 0u, 0u);
        if (m % kStageGroup == kStageGroup - 1 || m == R - 1) cp_async_commit();
    }
    if (tid < 32) {
        if (blockIdx.y == 0 && blockIdx.z == 0) store_meta(a, t0 + tid, tid < n, meta);
        // Lane u plans token t0 + u; lanes past the run carry an empty plan.
        const TokenPlan<W> p = plan_token<W>(a, t0 + tid, meta);
        if (tid < kRowRun) {
            plan.kinds[tid] = p.kinds;
            plan.ins[tid] = p.ins;
#pragma unroll
            for (int iw = 0; iw < W; ++iw) plan.off[tid][iw] = p.off[iw];
        }
        // The straight loop serves tokens whose taps all come from x and
        // that have an insert slot, and PAD rows.
        const bool ax = __all_sync(kFullMask, tid >= n || p.kinds == kPadRow ||
                                                  (p.kinds == all_x_kinds<W>() && p.ins >= 0));
        if (tid == 0) plan.all_x = ax;
    }
    __syncthreads();
    if (!active) return;  // no copies were issued for an inactive thread

    const int head = c0 / a.ws;
    const int64_t chan_off = static_cast<int64_t>(head) * a.cs_h + a.off_s + c0 % a.ws;
    uint16_t *op = a.out + static_cast<int64_t>(t0) * a.os_t + c0;

    if (plan.all_x) {
        // Token u needs staged rows up to u + W - 1: wait only for the copy
        // groups up to that row, so stores start while later rows arrive.
        constexpr int kGroups = (R + kStageGroup - 1) / kStageGroup;
        uint4 ring[W - 1];
        cp_async_wait<kGroups - 1 - (W - 1) / kStageGroup>();  // rows 0 .. W-1
#pragma unroll
        for (int m = 0; m < W - 1; ++m) ring[m] = xs[m * nthreads];
#pragma unroll
        for (int u = 0; u < kRowRun; ++u) {
            if (u >= n) break;  // block-uniform
            // Wait only where the needed group changes: a wait orders all
            // memory accesses around it, so tokens between two waits can
            // still be interleaved by the compiler.
            const int need = (u + W - 1) / kStageGroup;
            if (u > 0 && need != (u + W - 2) / kStageGroup) cp_async_wait_upto(kGroups - 1 - need);
            const uint4 xr = xs[(u + W - 1) * nthreads];
            const int64_t ins = plan.ins[u];
            if (ins >= 0) {  // block-uniform
                *reinterpret_cast<uint4 *>(a.cache + ins + chan_off) = xr;
                __stcs(reinterpret_cast<uint4 *>(op), paged_row<W, SILU, RESID>(wpk, ring, xr));
            } else {
                // A PAD row: every tap is zero, so the output is act(0) plus
                // the residual, and nothing is inserted.
                float zero[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
                __stcs(reinterpret_cast<uint4 *>(op), finish_row<SILU, RESID>(zero, xr));
            }
            op += a.os_t;
#pragma unroll
            for (int m = 0; m < W - 2; ++m) ring[m] = ring[m + 1];
            ring[W - 2] = xr;
        }
        return;
    }

    // General path.  First pull every cache tap of the run into L1:
    // prefetches hold no registers, so the whole run's round trip overlaps,
    // and the grouped loads below hit L1.  Pre-forward positions are never
    // written in this launch, so their lines in L1 stay valid.
#pragma unroll 1
    for (int u = 0; u < n; ++u) {
        const int kinds = plan.kinds[u];
#pragma unroll
        for (int iw = 0; iw < W; ++iw)
            if (((kinds >> (2 * iw)) & 3) == kTapCache) prefetch_l1(a.cache + plan.off[u][iw] + chan_off);
    }
    cp_async_wait<0>();
#pragma unroll 1
    for (int u = 0; u < n; ++u) {
        const int kinds = plan.kinds[u];
        const int64_t ins = plan.ins[u];
        const uint4 xr = xs[(u + W - 1) * nthreads];
        // The taps are read before the insert is written: the compiler cannot
        // prove them disjoint, and a read after the store would wait for it.
        uint4 tap[W];
#pragma unroll
        for (int iw = 0; iw < W; ++iw) {
            const int kind = (kinds >> (2 * iw)) & 3;
            // The token's own position (iw = W-1) comes from the cache only
            // when its query start lies after it (inconsistent metadata); it
            // is read like any other cached tap.
            tap[iw] = kind == kTapX      ? xs[(u + iw) * nthreads]
                      : kind == kTapCache ? *reinterpret_cast<const uint4 *>(a.cache + plan.off[u][iw] + chan_off)
                                          : make_uint4(0u, 0u, 0u, 0u);
        }
        if (ins >= 0) *reinterpret_cast<uint4 *>(a.cache + ins + chan_off) = xr;
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int iw = 0; iw < W; ++iw)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                fma_bf16x2(acc[2 * q], acc[2 * q + 1], word_of(tap[iw], q), word_of(wpk[iw], q));
        __stcs(reinterpret_cast<uint4 *>(op), finish_row<SILU, RESID>(acc, xr));
        op += a.os_t;
    }
}

using ScalarFn = void (*)(PagedArgs);

template <int W>
ScalarFn pick_scalar_w(bool silu, bool resid) {
    if (silu) return resid ? paged_scalar_kernel<W, true, true> : paged_scalar_kernel<W, true, false>;
    return resid ? paged_scalar_kernel<W, false, true> : paged_scalar_kernel<W, false, false>;
}

ScalarFn pick_scalar(int width, bool silu, bool resid) {
    switch (width) {
        case 2: return pick_scalar_w<2>(silu, resid);
        case 3: return pick_scalar_w<3>(silu, resid);
        case 4: return pick_scalar_w<4>(silu, resid);
        case 5: return pick_scalar_w<5>(silu, resid);
    }
    return nullptr;
}

constexpr int kMetaThreads = 256;

__global__ void __launch_bounds__(kMetaThreads)
seq_metadata_kernel(const int32_t *qsl, int num_reqs, int num_actual, int num_padded,
                    int32_t *seq_idx, int32_t *query_start) {
    release_next_grid();
    wait_prior_grid();
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
    return launch_pdl(seq_metadata_kernel, dim3(blocks), dim3(kMetaThreads), 0, stream,
                      query_start_loc, num_reqs, num_actual_tokens, num_padded_tokens, seq_idx_out,
                      query_start_out);
}

namespace ccv {
namespace {

// Shared arguments of every paged conv call (cache, token metadata, sizes).
struct PagedShared {
    void *cache;
    int64_t cs_blk, cs_h, cs_n;
    int num_blocks, H, N, D;
    const int64_t *pos;
    const int32_t *seq_idx;
    const int64_t *slot;
    const int32_t *bt;
    int64_t bt_r;
    int bt_rows, max_blocks;
    const int32_t *qstart;
    int T, width, silu, residual;
    int *err;
    // set for the single-launch call that resolves the metadata itself
    int own_meta = 0;
    const int32_t *qsl = nullptr;
    int num_reqs = 0, num_actual = 0;
    int32_t *seq_out = nullptr, *qs_out = nullptr;
};

int check_shared(const PagedShared &p) {
    if (p.width < kMinWidth || p.width > kMaxWidth) return CCV_ERR_WIDTH;
    if (p.T < 0 || p.num_blocks < 0 || p.H <= 0 || p.N <= 0 || p.D <= 0 || p.bt_rows < 0 ||
        p.max_blocks <= 0)
        return CCV_ERR_SIZE;
    if (p.cs_blk < 0 || p.cs_h < 0 || p.cs_n < 0 || p.bt_r < 0) return CCV_ERR_STRIDE;
    return CCV_OK;
}

int check_stream(const PagedShared &p, const ccv_paged_stream &st) {
    if (st.ws <= 0) return CCV_ERR_SIZE;
    if (st.off_s < 0 || st.off_s + st.ws > p.D) return CCV_ERR_RANGE;
    if (st.x_stride_t < 0 || st.w_stride_c < 0 || st.w_stride_w < 0 || st.out_stride_t < 0)
        return CCV_ERR_STRIDE;
    if (static_cast<int64_t>(p.H) * st.ws > 0x7fffffffLL) return CCV_ERR_SIZE;
    return CCV_OK;
}

Extent cache_extent(const PagedShared &p) {
    const Extent ec = extent_of(p.cache, p.num_blocks > 0 ? p.num_blocks : 1, p.cs_blk, p.H,
                                p.cs_h, p.N, p.cs_n);
    return Extent{ec.lo, ec.hi + static_cast<uintptr_t>(p.D - 1) * 2u};
}

PagedArgs shared_args(const PagedShared &p) {
    PagedArgs a{};
    a.cache = static_cast<uint16_t *>(p.cache);
    a.cs_blk = p.cs_blk;
    a.cs_h = p.cs_h;
    a.cs_n = p.cs_n;
    a.num_blocks = p.num_blocks;
    a.N = p.N;
    a.pos = p.pos;
    a.seq_idx = p.seq_idx;
    a.slot = p.slot;
    a.bt = p.bt;
    a.bt_r = p.bt_r;
    a.bt_rows = p.bt_rows;
    a.max_blocks = p.max_blocks;
    a.qstart = p.qstart;
    a.T = p.T;
    a.n_shift = (p.N & (p.N - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(p.N)) : -1;
    a.err = p.err;
    a.own_meta = p.own_meta;
    a.qsl = p.qsl;
    a.num_reqs = p.num_reqs;
    a.num_actual = p.num_actual;
    a.seq_out = p.seq_out;
    a.qs_out = p.qs_out;
    return a;
}

StreamFields stream_fields(const PagedShared &p, const ccv_paged_stream &st) {
    StreamFields f;
    f.x = static_cast<const uint16_t *>(st.x);
    f.xs_t = st.x_stride_t;
    f.w = static_cast<const uint16_t *>(st.weight);
    f.ws_c = st.w_stride_c;
    f.ws_k = st.w_stride_w;
    f.out = static_cast<uint16_t *>(st.out);
    f.os_t = st.out_stride_t;
    f.off_s = st.off_s;
    f.ws = st.ws;
    f.C = p.H * st.ws;
    f.w_vec = st.w_stride_w == 1 && st.w_stride_c == p.width && aligned16(st.weight);
    return f;
}

// The 16-byte vector kernel applies: whole 8-channel vectors everywhere.
bool vec_ok(const PagedShared &p, const ccv_paged_stream &st) {
    return st.ws % 8 == 0 && st.off_s % 8 == 0 && aligned16(st.x) && aligned16(st.out) &&
           aligned16(p.cache) && st.x_stride_t % 8 == 0 && st.out_stride_t % 8 == 0 &&
           p.cs_blk % 8 == 0 && p.cs_h % 8 == 0 && p.cs_n % 8 == 0;
}

// Launch the given streams (all vector-capable) as one grid, blockIdx.z = stream.
// The row kernel for width W with its shared-memory limit raised, once per
// device, to what its largest block needs.
template <int W, bool SILU, bool RESID>
int launch_row_w(const PagedLaunch &pl, dim3 grid, int threads, ccv_stream_t stream) {
    constexpr size_t kMaxBytes = sizeof(uint4) * kRowMaxThreads * row_slots<W>();
    int dev = 0;
    current_device_sms(&dev);
    cudaError_t e;
    if (resident_blocks<paged_row_kernel<W, SILU, RESID>>(kRowMaxThreads, kMaxBytes, dev, &e) == 0)
        return static_cast<int>(e);
    const size_t bytes = sizeof(uint4) * static_cast<size_t>(threads) * row_slots<W>();
    return launch_pdl(paged_row_kernel<W, SILU, RESID>, grid, dim3(threads), bytes, stream, pl);
}

template <int W>
int launch_row(const PagedLaunch &pl, dim3 grid, int threads, bool silu, bool resid,
               ccv_stream_t stream) {
    if (silu) return resid ? launch_row_w<W, true, true>(pl, grid, threads, stream)
                           : launch_row_w<W, true, false>(pl, grid, threads, stream);
    return resid ? launch_row_w<W, false, true>(pl, grid, threads, stream)
                 : launch_row_w<W, false, false>(pl, grid, threads, stream);
}

// Launch the given streams (all vector-capable) as one grid, blockIdx.z =
// stream: blocks of kRowRun tokens by up to kRowMaxThreads * 8 channels
// (fewer threads when the widest stream is narrower).
int launch_vec(const PagedShared &p, const ccv_paged_stream *streams, int n, ccv_stream_t stream) {
    PagedLaunch pl;
    pl.a = shared_args(p);
    int max_c = 0;
    for (int i = 0; i < kMaxStreams; ++i) pl.s[i] = stream_fields(p, streams[i < n ? i : 0]);
    for (int i = 0; i < n; ++i) max_c = pl.s[i].C > max_c ? pl.s[i].C : max_c;
    apply_stream(pl.a, pl.s[0]);
    const int vecs = (max_c + 7) / 8;
    const int threads = vecs >= kRowMaxThreads ? kRowMaxThreads : (vecs + 31) / 32 * 32;
    const dim3 grid(static_cast<unsigned>((p.T + kRowRun - 1) / kRowRun),
                    static_cast<unsigned>((max_c + threads * 8 - 1) / (threads * 8)),
                    static_cast<unsigned>(n));
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    const bool silu = p.silu != 0, resid = p.residual != 0;
    switch (p.width) {
        case 2: return launch_row<2>(pl, grid, threads, silu, resid, stream);
        case 3: return launch_row<3>(pl, grid, threads, silu, resid, stream);
        case 4: return launch_row<4>(pl, grid, threads, silu, resid, stream);
        case 5: return launch_row<5>(pl, grid, threads, silu, resid, stream);
    }
    return CCV_ERR_WIDTH;
}

int launch_scalar(const PagedShared &p, const ccv_paged_stream &st, ccv_stream_t stream) {
    PagedArgs a = shared_args(p);
    apply_stream(a, stream_fields(p, st));
    const dim3 grid(static_cast<unsigned>((p.T + kBlockTokens - 1) / kBlockTokens),
                    static_cast<unsigned>((a.C + 31) / 32));
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    return launch_pdl(pick_scalar(p.width, p.silu != 0, p.residual != 0), grid, dim3(kThreads), 0,
                      stream, a);
}

int paged_run(const PagedShared &p, const ccv_paged_stream *streams, int n, ccv_stream_t stream) {
    int rc = check_shared(p);
    if (rc != CCV_OK) return rc;
    if (n < 1 || n > kMaxStreams) return CCV_ERR_SIZE;
    if (streams == nullptr) return CCV_ERR_NULL_POINTER;
    for (int i = 0; i < n; ++i) {
        rc = check_stream(p, streams[i]);
        if (rc != CCV_OK) return rc;
        for (int j = 0; j < i; ++j) {
            // streams own disjoint D-ranges of the shared cache
            const int lo = streams[i].off_s > streams[j].off_s ? streams[i].off_s : streams[j].off_s;
            const int hi_i = streams[i].off_s + streams[i].ws, hi_j = streams[j].off_s + streams[j].ws;
            if (lo < (hi_i < hi_j ? hi_i : hi_j)) return CCV_ERR_RANGE;
        }
    }
    if (p.T == 0) return CCV_OK;
    if (p.cache == nullptr || p.pos == nullptr || p.slot == nullptr || p.bt == nullptr)
        return CCV_ERR_NULL_POINTER;
    if (!p.own_meta && (p.seq_idx == nullptr || p.qstart == nullptr)) return CCV_ERR_NULL_POINTER;
    const Extent ec = cache_extent(p);
    for (int i = 0; i < n; ++i) {
        const ccv_paged_stream &st = streams[i];
        if (st.x == nullptr || st.weight == nullptr || st.out == nullptr) return CCV_ERR_NULL_POINTER;
        const int C = p.H * st.ws;
        const Extent eo = extent_of(st.out, p.T, st.out_stride_t, C, 1);
        if (overlaps(eo, ec)) return CCV_ERR_ALIAS;
        for (int j = 0; j < n; ++j) {
            const Extent ex = extent_of(streams[j].x, p.T, streams[j].x_stride_t, p.H * streams[j].ws, 1);
            if (overlaps(eo, ex)) return CCV_ERR_ALIAS;
            if (j < i && overlaps(eo, extent_of(streams[j].out, p.T, streams[j].out_stride_t,
                                                p.H * streams[j].ws, 1)))
                return CCV_ERR_ALIAS;
        }
    }
    bool all_vec = true;
    for (int i = 0; i < n; ++i) all_vec = all_vec && vec_ok(p, streams[i]);
    if (all_vec) return launch_vec(p, streams, n, stream);
    // Mixed layouts: each stream on its own, in order.
    for (int i = 0; i < n; ++i) {
        rc = vec_ok(p, streams[i]) ? launch_vec(p, streams + i, 1, stream)
                                   : launch_scalar(p, streams[i], stream);
        if (rc != CCV_OK) return rc;
    }
    return CCV_OK;
}

}  // namespace
}  // namespace ccv

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
    const ccv::PagedShared p{cache, c_stride_blk, c_stride_h, c_stride_n, num_blocks, H, N, D,
                             positions, seq_idx, slot_mapping, block_table, bt_stride_r, bt_rows,
                             max_blocks, query_start, T, width, silu, residual, err_count};
    const ccv_paged_stream st{x, x_stride_t, weight, w_stride_c, w_stride_w, out, out_stride_t,
                              off_s, ws};
    return ccv::paged_run(p, &st, 1, stream);
}

extern "C" int paged_sconv_fwd_streams(const ccv_paged_stream *streams, int num_streams,
                                       void *cache, int64_t c_stride_blk, int64_t c_stride_h,
                                       int64_t c_stride_n, int num_blocks, int H, int N, int D,
                                       const int64_t *positions, const int32_t *seq_idx,
                                       const int64_t *slot_mapping, const int32_t *block_table,
                                       int64_t bt_stride_r, int bt_rows, int max_blocks,
                                       const int32_t *query_start, int T, int width, int silu,
                                       int residual, int *err_count, ccv_stream_t stream) {
    const ccv::PagedShared p{cache, c_stride_blk, c_stride_h, c_stride_n, num_blocks, H, N, D,
                             positions, seq_idx, slot_mapping, block_table, bt_stride_r, bt_rows,
                             max_blocks, query_start, T, width, silu, residual, err_count};
    return ccv::paged_run(p, streams, num_streams, stream);
}

extern "C" int paged_sconv_fwd_with_metadata(
    const void *x, int64_t x_stride_t, void *cache, int64_t c_stride_blk, int64_t c_stride_h,
    int64_t c_stride_n, int num_blocks, int H, int N, int D, const void *weight,
    int64_t w_stride_c, int64_t w_stride_w, void *out, int64_t out_stride_t,
    const int64_t *positions, const int32_t *query_start_loc, int num_reqs,
    int num_actual_tokens, int32_t *seq_idx_out, int32_t *query_start_out,
    const int64_t *slot_mapping, const int32_t *block_table, int64_t bt_stride_r, int bt_rows,
    int max_blocks, int T, int off_s, int ws, int width, int silu, int residual, int *err_count,
    ccv_stream_t stream) {
    using namespace ccv;
    if (num_reqs < 0 || num_actual_tokens < 0 || T < 0) return CCV_ERR_SIZE;
    if (num_actual_tokens > T) return CCV_ERR_SIZE;
    if (num_reqs == 0 && num_actual_tokens > 0) return CCV_ERR_SIZE;
    if (T > 0 && num_reqs > 0 && query_start_loc == nullptr) return CCV_ERR_NULL_POINTER;
    PagedShared p{cache, c_stride_blk, c_stride_h, c_stride_n, num_blocks, H, N, D,
                  positions, nullptr, slot_mapping, block_table, bt_stride_r, bt_rows,
                  max_blocks, nullptr, T, width, silu, residual, err_count};
    p.own_meta = 1;
    p.qsl = query_start_loc;
    p.num_reqs = num_reqs;
    p.num_actual = num_actual_tokens;
    p.seq_out = seq_idx_out;
    p.qs_out = query_start_out;
    const ccv_paged_stream st{x, x_stride_t, weight, w_stride_c, w_stride_w, out, out_stride_t,
                              off_s, ws};
    return paged_run(p, &st, 1, stream);
}
