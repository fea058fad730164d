// ccv_fwd: varlen causal depthwise conv1d prefill with conv_state.
//
// Semantics: tokenspeed causal_conv1d.py, `causal_conv1d_fn` and its kernel
// `_causal_conv1d_fwd_kernel` (chunk-0 state read, state update, halo of
// later chunks, token loop); the reference formulation is atrex-bench #003
// `causal_conv1d` (concatenate the state, grouped conv1d, SiLU).
//
// Work decomposition.  One thread block owns one (sequence chunk, channel
// tile), so state handling never mixes sequences.  The grid is fixed by the
// host-known sizes only: chunk slot j of a sequence i that starts at token
// q_i is j = floor(q_i / CHUNK) + i + chunk, which is unique per (i, chunk)
// and bounded by floor(total_tokens / CHUNK) + batch, so blockIdx.x finds its
// sequence by a binary search over query_start_loc and surplus blocks exit.
// No host-side chunk list, no device-to-host copy, CUDA-graph capturable.
//
// The conv_state write-back is done by the block that reads the old state
// (chunk 0 of the sequence): it is the only reader of that line, so reading
// before writing needs no inter-block ordering.  It takes the sequence's last
// width-1 inputs straight from x.
//
// Two layouts get their own kernel:
//   * channel-last  (x stride over channels == 1): a lane owns 8 consecutive
//     channels (one 16-byte vector per token row) and walks a run of tokens,
//     keeping the width-1 previous inputs in registers;
//   * channel-first (x stride over tokens == 1): a warp owns one channel row,
//     a lane owns 8 consecutive tokens (one 16-byte vector), and the halo of
//     width-1 earlier tokens arrives from the neighbouring lane by shuffle.
// A VEC = 1 instantiation of each handles unaligned or arbitrary strides.
// Accumulation is fp32 in the pages' order (bias first, taps 0..W-1), SiLU
// in fp32, one round-to-nearest-even store to bf16.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

// channel-last tiling: 4 warps take consecutive runs of kClRun tokens.
constexpr int kClRun = 32;
constexpr int kClChunk = kWarps * kClRun;
constexpr int kClUnroll = 8;

// channel-first tiling: a chunk is kCfSegs warp-wide segments of 32*VEC tokens.
constexpr int kCfSegs = 8;
constexpr int kCfUnroll = 4;

struct FwdArgs {
    const uint16_t *x;
    int64_t xs_d, xs_t;
    uint16_t *out;
    int64_t os_d, os_t;
    const uint16_t *w;
    int64_t ws_d, ws_k;
    const uint16_t *bias;
    uint16_t *st;
    int64_t ss_l, ss_d, ss_t;
    int num_lines;
    const int32_t *qsl;
    int batch;
    const int32_t *cidx;
    const uint8_t *has_init;
    int dim, total, pad;
    int *err;
    int st_vec;  // channel-last: state columns are 16-byte vectors over channels
};

struct ChunkInfo {
    int seq, chunk, start, len;
};

// Map chunk slot `slot` to its (sequence, chunk); false for a surplus slot.
// Warp-cooperative, every lane gets the same answer.  f(i) = floor(qsl[i] /
// chunk_tokens) + i increases strictly with i for a valid query_start_loc, so
// {i : f(i) <= slot} is a prefix of [0, batch); each round samples 32 evenly
// spaced candidates of the current window and keeps the 1/32 slice after the
// last one that satisfies it: one round trip for up to 32 sequences, two for
// up to 1024.  Garbage offsets only lead to a wrong (validated, skipped) pick.
__device__ __forceinline__ bool locate_chunk(const FwdArgs &a, int chunk_tokens, int slot,
                                             ChunkInfo &ci) {
    const int lane = threadIdx.x & 31;
    int lo = 0, n = a.batch;
    while (n > 1) {
        const int stride = (n + 31) >> 5;
        const int off = lane * stride;
        bool le = false;
        if (off < n) {
            const int i = lo + off;
            le = floor_div(__ldg(a.qsl + i), chunk_tokens) + i <= slot;
        }
        const unsigned m = __ballot_sync(kFullMask, le);
        if (m == 0u) break;
        const int top = 31 - __clz(m);
        lo += top * stride;
        n = min(stride, n - top * stride);
    }
    const int start = __ldg(a.qsl + lo);
    const int end = __ldg(a.qsl + lo + 1);
    if (start < 0 || end < start || end > a.total) return false;
    const int k = slot - (start / chunk_tokens + lo);
    if (k < 0 || static_cast<int64_t>(k) * chunk_tokens >= end - start) return false;
    ci.seq = lo;
    ci.chunk = k;
    ci.start = start;
    ci.len = end - start;
    return true;
}

// Stage the block's weight tile (tile_c channels from cbase, W taps) and bias
// in shared memory as [tap][channel] bf16, with coalesced global loads; every
// thread of the block must call this (it ends with a barrier).
template <int W>
__device__ __forceinline__ void stage_weights(const uint16_t *w, int64_t ws_d, int64_t ws_k,
                                              const uint16_t *bias, int dim, int cbase,
                                              int tile_c, uint16_t *s_w, uint16_t *s_b) {
    for (int i = threadIdx.x; i < W * tile_c; i += blockDim.x) {
        const int cl = i / W;
        const int k = i - cl * W;
        const int c = cbase + cl;
        s_w[k * tile_c + cl] = c < dim ? __ldg(w + c * ws_d + k * ws_k) : uint16_t(0);
    }
    for (int i = threadIdx.x; i < tile_c; i += blockDim.x) {
        const int c = cbase + i;
        s_b[i] = (bias != nullptr && c < dim) ? __ldg(bias + c) : uint16_t(0);
    }
    __syncthreads();
}

// Blocks (x < batch, y == 0) each check one sequence's indices and count
// invalid ones; the chunk blocks skip such sequences silently.
__device__ __forceinline__ void validate_sequence(const FwdArgs &a) {
    if (a.err == nullptr || blockIdx.y != 0 || threadIdx.x != 0) return;
    const int i = blockIdx.x;
    if (i >= a.batch) return;
    const int line = a.cidx ? __ldg(a.cidx + i) : i;
    if (line == a.pad) return;
    const int s = __ldg(a.qsl + i), e = __ldg(a.qsl + i + 1);
    bool bad = s < 0 || e < s || e > a.total;
    if (!bad && a.st != nullptr && e > s && (line < 0 || line >= a.num_lines)) bad = true;
    if (bad) atomicAdd(a.err, 1);
}

// Resolve the state line of the chunk's sequence; false = skip the sequence.
__device__ __forceinline__ bool sequence_line(const FwdArgs &a, const ChunkInfo &ci, int &line) {
    line = a.cidx ? __ldg(a.cidx + ci.seq) : ci.seq;
    if (line == a.pad) return false;
    if (a.st != nullptr && (line < 0 || line >= a.num_lines)) return false;
    return true;
}

template <int VEC>
__device__ __forceinline__ Raw<VEC> load_state(const FwdArgs &a, int line, int c0, int col) {
    const uint16_t *p = a.st + line * a.ss_l + c0 * a.ss_d + col * a.ss_t;
    Raw<VEC> r;
    if (VEC == 8 && a.st_vec) {
        r = load_plain<VEC>(p);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r.set_elem(v, p[v * a.ss_d]);
    }
    return r;
}

template <int VEC>
__device__ __forceinline__ void store_state(const FwdArgs &a, int line, int c0, int col,
                                            const Raw<VEC> &r) {
    uint16_t *p = a.st + line * a.ss_l + c0 * a.ss_d + col * a.ss_t;
    if (VEC == 8 && a.st_vec) {
        store_plain<VEC>(p, r);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) p[v * a.ss_d] = r.elem(v);
    }
}

// ------------------------------------------------------ channel-last ----

template <int W, bool SILU, int VEC>
__device__ __forceinline__ void cl_token(const float (&wt)[W][VEC], const float (&bs)[VEC],
                                         float (&ring)[W - 1][VEC], const Raw<VEC> &xv,
                                         uint16_t *dst) {
    float xf[VEC];
    xv.to_float(xf);
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        float s = bs[v];
#pragma unroll
        for (int k = 0; k < W - 1; ++k) s = fmaf(wt[k][v], ring[k][v], s);
        s = fmaf(wt[W - 1][v], xf[v], s);
        acc[v] = SILU ? silu(s) : s;
    }
    Raw<VEC> o;
    o.from_float(acc);
    store_stream<VEC>(dst, o);
#pragma unroll
    for (int k = 0; k < W - 2; ++k)
#pragma unroll
        for (int v = 0; v < VEC; ++v) ring[k][v] = ring[k + 1][v];
#pragma unroll
    for (int v = 0; v < VEC; ++v) ring[W - 2][v] = xf[v];
}

template <int W, bool SILU, int VEC>
__global__ void __launch_bounds__(kThreads) fwd_cl_kernel(const FwdArgs a) {
    constexpr int TILE_C = 32 * VEC;
    __shared__ __align__(16) uint16_t s_w[W * TILE_C];
    __shared__ __align__(16) uint16_t s_b[TILE_C];
    validate_sequence(a);
    ChunkInfo ci;
    if (!locate_chunk(a, kClChunk, blockIdx.x, ci)) return;
    int line;
    if (!sequence_line(a, ci, line)) return;
    stage_weights<W>(a.w, a.ws_d, a.ws_k, a.bias, a.dim, blockIdx.y * TILE_C, TILE_C, s_w, s_b);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int c0 = (blockIdx.y * 32 + lane) * VEC;
    if (c0 >= a.dim) return;

    const int cbeg = ci.start + ci.chunk * kClChunk;
    const int cend = ci.start + min(ci.len, (ci.chunk + 1) * kClChunk);
    const int r0 = cbeg + warp * kClRun;
    const int r1 = min(r0 + kClRun, cend);
    if (r0 >= r1) return;  // the first run of a sequence is never empty

    const uint16_t *xc = a.x + c0 * a.xs_d;
    uint16_t *oc = a.out + c0 * a.os_d;

    float wt[W][VEC], bs[VEC];
#pragma unroll
    for (int k = 0; k < W; ++k)
        reinterpret_cast<const Raw<VEC> *>(s_w + k * TILE_C)[lane].to_float(wt[k]);
    reinterpret_cast<const Raw<VEC> *>(s_b)[lane].to_float(bs);

    float ring[W - 1][VEC];
    if (ci.chunk == 0 && warp == 0) {
        // First run of the sequence: the prior comes from the state line.
        Raw<VEC> prior[W - 1];
        const bool init = a.st != nullptr && a.has_init != nullptr && a.has_init[ci.seq] != 0;
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            if (init) prior[j] = load_state<VEC>(a, line, c0, j);
            else prior[j].zero();
            prior[j].to_float(ring[j]);
        }
        if (a.st != nullptr) {
            // New state = last W-1 entries of prior ++ x[sequence].
            Raw<VEC> nw[W - 1];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) {
                const int idx = ci.len + j;
                if (idx < W - 1) {
#pragma unroll
                    for (int q = 0; q < W - 1; ++q)
                        if (q == idx) nw[j] = prior[q];
                } else {
                    nw[j] = load_plain<VEC>(xc + (ci.start + idx - (W - 1)) * a.xs_t);
                }
            }
#pragma unroll
            for (int j = 0; j < W - 1; ++j) store_state<VEC>(a, line, c0, j, nw[j]);
        }
    } else {
        // Later runs: the halo is the previous W-1 tokens of the same sequence.
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            load_plain<VEC>(xc + (r0 - (W - 1) + j) * a.xs_t).to_float(ring[j]);
    }

    int t = r0;
    for (; t + kClUnroll <= r1; t += kClUnroll) {
        Raw<VEC> xv[kClUnroll];
#pragma unroll
        for (int u = 0; u < kClUnroll; ++u) xv[u] = load_stream<VEC>(xc + (t + u) * a.xs_t);
#pragma unroll
        for (int u = 0; u < kClUnroll; ++u)
            cl_token<W, SILU, VEC>(wt, bs, ring, xv[u], oc + (t + u) * a.os_t);
    }
    for (; t < r1; ++t) {
        const Raw<VEC> xv = load_stream<VEC>(xc + t * a.xs_t);
        cl_token<W, SILU, VEC>(wt, bs, ring, xv, oc + t * a.os_t);
    }
}

// ----------------------------------------------------- channel-first ----

template <int W>
__device__ __forceinline__ uint16_t pick(const uint16_t (&arr)[W - 1], int idx) {
    uint16_t r = 0;
#pragma unroll
    for (int q = 0; q < W - 1; ++q)
        if (q == idx) r = arr[q];
    return r;
}

template <int W, bool SILU, int VEC>
__global__ void __launch_bounds__(kThreads) fwd_cf_kernel(const FwdArgs a) {
    constexpr int SEG = 32 * VEC;
    constexpr int CHUNK = kCfSegs * SEG;
    validate_sequence(a);
    ChunkInfo ci;
    if (!locate_chunk(a, CHUNK, blockIdx.x, ci)) return;
    int line;
    if (!sequence_line(a, ci, line)) return;

    const int lane = threadIdx.x & 31;
    const int c = blockIdx.y * kWarps + (threadIdx.x >> 5);
    if (c >= a.dim) return;  // warp-uniform

    const int cbeg = ci.start + ci.chunk * CHUNK;
    const int cend = ci.start + min(ci.len, (ci.chunk + 1) * CHUNK);
    const bool chunk0 = ci.chunk == 0;
    const uint16_t *xc = a.x + c * a.xs_d;
    uint16_t *oc = a.out + c * a.os_d;

    float wt[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wt[k] = bf16_bits(__ldg(a.w + c * a.ws_d + k * a.ws_k));
    const float bs = a.bias ? bf16_bits(__ldg(a.bias + c)) : 0.0f;

    uint16_t prior[W - 1];
    const bool init = chunk0 && a.st != nullptr && a.has_init != nullptr && a.has_init[ci.seq] != 0;
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
        prior[j] = init ? a.st[line * a.ss_l + c * a.ss_d + j * a.ss_t] : uint16_t(0);

    // Segments start at a 16-byte boundary of this row (VEC = 8, stride 1).
    int a0 = cbeg;
    if (VEC == 8) {
        const int phase = static_cast<int>((reinterpret_cast<uintptr_t>(xc) >> 1) & 7u);
        a0 = cbeg - ((phase + cbeg) & 7);
    }
    const int lo_x = chunk0 ? cbeg : cbeg - (W - 1);  // first token read from x
    // Logical input u at token t (x inside the chunk, prior or x in the halo).
    auto value = [&](int t) -> uint16_t {
        if (t >= lo_x && t < cend) return xc[t * a.xs_t];
        if (chunk0 && t >= cbeg - (W - 1) && t < cbeg) return pick<W>(prior, t - cbeg + (W - 1));
        return uint16_t(0);
    };

    // The segment before the first one, as far as the halo needs it.
    float prev[VEC];
    {
        Raw<VEC> r;
#pragma unroll
        for (int i = 0; i < VEC; ++i) r.set_elem(i, value(a0 - SEG + lane * VEC + i));
        r.to_float(prev);
    }

    const int nseg = (cend - a0 + SEG - 1) / SEG;
    for (int s0 = 0; s0 < nseg; s0 += kCfUnroll) {
        Raw<VEC> cur[kCfUnroll];
#pragma unroll
        for (int u = 0; u < kCfUnroll; ++u) {
            const int tok0 = a0 + (s0 + u) * SEG + lane * VEC;
            if (s0 + u < nseg) {
                if (tok0 >= lo_x && tok0 + VEC <= cend) {
                    cur[u] = load_stream<VEC>(xc + tok0 * a.xs_t);
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) cur[u].set_elem(i, value(tok0 + i));
                }
            } else {
                cur[u].zero();
            }
        }
#pragma unroll
        for (int u = 0; u < kCfUnroll; ++u) {
            if (s0 + u >= nseg) break;  // warp-uniform
            const int tok0 = a0 + (s0 + u) * SEG + lane * VEC;
            float cf[VEC];
            cur[u].to_float(cf);
            // halo[m-1] = u[tok0 - m], m = 1..W-1, from the lanes before.
            float halo[W - 1];
#pragma unroll
            for (int m = 1; m <= W - 1; ++m) {
                const int d = VEC == 1 ? m : 1;
                const int e = VEC == 1 ? 0 : VEC - m;
                const float from_cur = __shfl_up_sync(kFullMask, cf[e], d);
                const float from_prev = __shfl_sync(kFullMask, prev[e], (lane - d) & 31);
                halo[m - 1] = lane >= d ? from_cur : from_prev;
            }
            float o[VEC];
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                float s = bs;
#pragma unroll
                for (int k = 0; k < W; ++k) {
                    // tap k reads token tok0 + i - (W-1) + k: own vector or halo
                    const int idx = i - (W - 1) + k;
                    const float u = idx >= 0 ? cf[max(idx, 0)] : halo[max(-idx - 1, 0)];
                    s = fmaf(wt[k], u, s);
                }
                o[i] = SILU ? silu(s) : s;
            }
            if (tok0 >= cbeg && tok0 + VEC <= cend) {
                Raw<VEC> r;
                r.from_float(o);
                store_stream<VEC>(oc + tok0 * a.os_t, r);
            } else {
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const int t = tok0 + i;
                    if (t >= cbeg && t < cend) oc[t * a.os_t] = round_bf16(o[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < VEC; ++i) prev[i] = cf[i];
        }
    }

    if (chunk0 && a.st != nullptr) {
        // New state = last W-1 entries of prior ++ x[sequence]; every lane has
        // finished reading the old state before any lane writes it.
        uint16_t nb = 0;
        if (lane < W - 1) {
            const int idx = ci.len + lane;
            nb = idx < W - 1 ? pick<W>(prior, idx) : xc[(ci.start + idx - (W - 1)) * a.xs_t];
        }
        __syncwarp();
        if (lane < W - 1) a.st[line * a.ss_l + c * a.ss_d + lane * a.ss_t] = nb;
    }
}

// ----------------------------------------------------------- dispatch ----

using KernelFn = void (*)(FwdArgs);

template <int VEC, bool CL>
KernelFn pick_kernel(int width, bool silu) {
#define CCV_FWD_CASE(W)                                                              \
    case W:                                                                          \
        if (CL) return silu ? fwd_cl_kernel<W, true, VEC> : fwd_cl_kernel<W, false, VEC>; \
        return silu ? fwd_cf_kernel<W, true, VEC> : fwd_cf_kernel<W, false, VEC>;
    switch (width) {
        CCV_FWD_CASE(2)
        CCV_FWD_CASE(3)
        CCV_FWD_CASE(4)
        CCV_FWD_CASE(5)
    }
#undef CCV_FWD_CASE
    return nullptr;
}

}  // namespace
}  // namespace ccv

extern "C" int ccv_fwd(const void *x, int64_t x_stride_dim, int64_t x_stride_tok,
                       void *out, int64_t out_stride_dim, int64_t out_stride_tok,
                       const void *weight, int64_t w_stride_dim, int64_t w_stride_w,
                       const void *bias,
                       void *conv_states, int64_t s_stride_line, int64_t s_stride_dim,
                       int64_t s_stride_tok, int num_cache_lines, int state_len,
                       const int32_t *query_start_loc, int batch,
                       const int32_t *cache_indices, const uint8_t *has_initial_state,
                       int dim, int total_tokens, int width, int pad_slot_id, int silu,
                       int *err_count, ccv_stream_t stream) {
    using namespace ccv;
    if (width < kMinWidth || width > kMaxWidth) return CCV_ERR_WIDTH;
    if (dim < 0 || total_tokens < 0 || batch < 0 || num_cache_lines < 0) return CCV_ERR_SIZE;
    if (x_stride_dim < 0 || x_stride_tok < 0 || out_stride_dim < 0 || out_stride_tok < 0 ||
        w_stride_dim < 0 || w_stride_w < 0 || s_stride_line < 0 || s_stride_dim < 0 ||
        s_stride_tok < 0)
        return CCV_ERR_STRIDE;
    if (has_initial_state != nullptr && conv_states == nullptr) return CCV_ERR_ARGUMENT;
    if (conv_states != nullptr && state_len < width - 1) return CCV_ERR_STATE_LEN;
    if (batch == 0 || total_tokens == 0 || dim == 0) return CCV_OK;
    if (x == nullptr || out == nullptr || weight == nullptr || query_start_loc == nullptr)
        return CCV_ERR_NULL_POINTER;
    if (overlaps(extent_of(x, dim, x_stride_dim, total_tokens, x_stride_tok),
                 extent_of(out, dim, out_stride_dim, total_tokens, out_stride_tok)))
        return CCV_ERR_ALIAS;

    FwdArgs a;
    a.x = static_cast<const uint16_t *>(x);
    a.xs_d = x_stride_dim;
    a.xs_t = x_stride_tok;
    a.out = static_cast<uint16_t *>(out);
    a.os_d = out_stride_dim;
    a.os_t = out_stride_tok;
    a.w = static_cast<const uint16_t *>(weight);
    a.ws_d = w_stride_dim;
    a.ws_k = w_stride_w;
    a.bias = static_cast<const uint16_t *>(bias);
    a.st = static_cast<uint16_t *>(conv_states);
    a.ss_l = s_stride_line;
    a.ss_d = s_stride_dim;
    a.ss_t = s_stride_tok;
    a.num_lines = num_cache_lines;
    a.qsl = query_start_loc;
    a.batch = batch;
    a.cidx = cache_indices;
    a.has_init = has_initial_state;
    a.dim = dim;
    a.total = total_tokens;
    a.pad = pad_slot_id;
    a.err = err_count;
    a.st_vec = 0;

    const bool is_silu = silu != 0;
    KernelFn fn = nullptr;
    dim3 grid;
    if (x_stride_dim == 1 && out_stride_dim == 1) {
        const bool vec = dim % 8 == 0 && aligned16(x) && aligned16(out) &&
                         x_stride_tok % 8 == 0 && out_stride_tok % 8 == 0;
        const int vec_w = vec ? 8 : 1;
        fn = vec ? pick_kernel<8, true>(width, is_silu) : pick_kernel<1, true>(width, is_silu);
        a.st_vec = vec && conv_states != nullptr && s_stride_dim == 1 && aligned16(conv_states) &&
                   s_stride_line % 8 == 0 && s_stride_tok % 8 == 0;
        grid = dim3(static_cast<unsigned>(total_tokens / kClChunk + batch),
                    static_cast<unsigned>((dim + 32 * vec_w - 1) / (32 * vec_w)));
    } else if (x_stride_tok == 1 && out_stride_tok == 1) {
        const uintptr_t xo = (reinterpret_cast<uintptr_t>(x) >> 1) & 7u;
        const uintptr_t oo = (reinterpret_cast<uintptr_t>(out) >> 1) & 7u;
        const bool vec = (reinterpret_cast<uintptr_t>(x) & 1u) == 0 &&
                         (reinterpret_cast<uintptr_t>(out) & 1u) == 0 && xo == oo &&
                         (x_stride_dim - out_stride_dim) % 8 == 0;
        const int seg = 32 * (vec ? 8 : 1);
        fn = vec ? pick_kernel<8, false>(width, is_silu) : pick_kernel<1, false>(width, is_silu);
        grid = dim3(static_cast<unsigned>(total_tokens / (kCfSegs * seg) + batch),
                    static_cast<unsigned>((dim + kWarps - 1) / kWarps));
    } else {
        fn = pick_kernel<1, true>(width, is_silu);
        grid = dim3(static_cast<unsigned>(total_tokens / kClChunk + batch),
                    static_cast<unsigned>((dim + 31) / 32));
    }
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    fn<<<grid, kThreads, 0, stream>>>(a);
    return launch_status();
}
