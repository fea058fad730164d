// ccv_update: decode step of the causal depthwise conv1d with an in-place
// conv_state shift.
//
// Semantics: tokenspeed causal_conv1d.py, `causal_conv1d_update` and
// `_causal_conv1d_update_kernel` (STEP 1 read the state window, STEP 2 shift
// the state left and append the new inputs, STEPS 3-5 bias, weights and the
// token loop), with its speculative-decoding extras: the window read at
// column num_accepted_tokens-1, the window after every token saved to the
// intermediate buffer and/or scattered to an output state line, and no
// in-place shift when either of those is requested.
//
// Three kernels, picked on the host from the sizes alone (so a CUDA graph
// replays the same launch):
//   * update_kernel<.., 8>: single-token rows without the spec extras; a
//     thread owns 8 consecutive channels (16-byte vectors) of kRows rows;
//   * spec_kernel: several tokens per row or any spec extra, 8 channels and
//     one row per thread;
//   * update_kernel<.., 1>: everything else (dims that are not a multiple of
//     8), one channel per thread.
// Every element of a state line and of out is read and written by the same
// thread, which makes the in-place state shift and out == x (the page's
// wrapper writes the output over x) hazard-free.
#include "ccv_common.cuh"
#include "ccv_math2.cuh"

namespace ccv {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 2;  // batch rows per thread

struct UpdArgs {
    const uint16_t *x;
    int64_t xs_b, xs_d, xs_t;
    uint16_t *out;
    int64_t os_b, os_d, os_t;
    const uint16_t *w;
    int64_t ws_d, ws_k;
    const uint16_t *bias;
    uint16_t *st;
    int64_t ss_l, ss_d, ss_t;
    int num_lines;
    const int32_t *idx;
    int batch, dim, seqlen, pad;
    int *err;
    int ctiles;
    int x_vec, o_vec, st_vec;  // operand is addressable as 16-byte channel vectors
    int w_vec, b_vec;          // weights contiguous (dim, W) / bias, 16-byte aligned
    // speculative decoding
    int state_len;
    const int32_t *nacc;       // num_accepted_tokens [batch] or null
    uint16_t *inter;           // window after each token: (b, step, c, j) or null
    int64_t is_b, is_t, is_d, is_w;
    int inter_vec;
    const int32_t *oidx;       // output state line per (b, step) or null
    int64_t ois_b, ois_t;
    int shift;                 // shift the state in place (neither buffer given)
    int plain;                 // no speculative extras at all
};

template <int VEC>
__device__ __forceinline__ Raw<VEC> gather(const uint16_t *p, int64_t stride, bool vec) {
    Raw<VEC> r;
    if (VEC == 8 && vec) {
        r = load_plain<VEC>(p);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r.set_elem(v, p[v * stride]);
    }
    return r;
}

// Stores of outputs, state lines and windows: plain stores.  The streaming
// (evict-first) hint was measured both ways: with decode right after the
// channel-first prefill (whose stores then carried the hint too) it made the
// whole step 1% faster, and in the step as the bench now runs it (prefill in
// both layouts, paged conv, decode) 0.35% slower; neither changes this
// kernel's own time.
template <int VEC>
__device__ __forceinline__ void scatter(uint16_t *p, int64_t stride, bool vec, const Raw<VEC> &r) {
    if (VEC == 8 && vec) {
        store_plain<VEC>(p, r);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) p[v * stride] = r.elem(v);
    }
}

// Stage the block's weights and bias as [tap][channel] bf16 in shared memory
// with coalesced loads; every thread of the block calls this.
template <int W>
__device__ __forceinline__ void stage_weights(const UpdArgs &a, int cbase, int tile_c,
                                              uint16_t *s_w, uint16_t *s_b) {
    for (int i = threadIdx.x; i < W * tile_c; i += blockDim.x) {
        const int cl = i / W;
        const int k = i - cl * W;
        const int c = cbase + cl;
        s_w[k * tile_c + cl] = c < a.dim ? __ldg(a.w + c * a.ws_d + k * a.ws_k) : uint16_t(0);
    }
    for (int i = threadIdx.x; i < tile_c; i += blockDim.x) {
        const int c = cbase + i;
        s_b[i] = (a.bias != nullptr && c < a.dim) ? __ldg(a.bias + c) : uint16_t(0);
    }
    __syncthreads();
}

template <int W, bool SILU, int VEC>
__device__ __forceinline__ void conv_token(const float (&wt)[W][VEC], const float (&bs)[VEC],
                                           const float (&ring)[W - 1][VEC], const float (&xf)[VEC],
                                           Raw<VEC> &o) {
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        float s = bs[v];
#pragma unroll
        for (int k = 0; k < W - 1; ++k) s = fmaf(wt[k][v], ring[k][v], s);
        s = fmaf(wt[W - 1][v], xf[v], s);
        acc[v] = SILU ? silu(s) : s;
    }
    o.from_float(acc);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// Single-token decode for 8 channels of one row: taps over the raw state
// window win[0..W-2] (oldest first) and x, native mixed-precision FMAs with
// the bias entering through the first tap.
template <int W, bool SILU>
__device__ __forceinline__ uint4 decode_row(const uint4 (&wpk)[W], const float (&bs)[8],
                                            const uint4 (&win)[W - 1], const uint4 &xv) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        fma_bf16x2_init(acc[2 * q], acc[2 * q + 1], word_of(win[0], q), word_of(wpk[0], q),
                        bs[2 * q], bs[2 * q + 1]);
#pragma unroll
    for (int k = 1; k < W; ++k) {
        const uint4 &u = k < W - 1 ? win[k < W - 1 ? k : 0] : xv;
#pragma unroll
        for (int q = 0; q < 4; ++q) fma_bf16x2(acc[2 * q], acc[2 * q + 1], word_of(u, q), word_of(wpk[k], q));
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f32x2 r = pack2(acc[2 * q], acc[2 * q + 1]);
        if (SILU) r = silu2(r);
        o[q] = f32x2_to_bf16x2(r);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Resolve the rows' state lines (skipped rows get line -1).
__device__ __forceinline__ void resolve_lines(const UpdArgs &a, int rg, bool active, int c0,
                                              int (&lines)[kRows]) {
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const int b = rg * kRows + r;
        int line = -1;
        if (active && b < a.batch) {
            line = a.idx ? __ldg(a.idx + b) : b;
            if (line == a.pad) {
                line = -1;
            } else if (line < 0 || line >= a.num_lines) {
                if (c0 == 0) count_error(a.err);
                line = -1;
            }
        }
        lines[r] = line;
    }
}

// General rows: any seqlen and the spec extras, fp32 arithmetic; the block's
// weights and bias are staged as [tap][channel] (this thread's at s_w + k *
// tile_c and s_b).
template <int W, bool SILU, int VEC>
__device__ __forceinline__ void general_rows(const UpdArgs &a, int rg, int c0, const int (&lines)[kRows],
                                             const uint16_t *s_w, const uint16_t *s_b, int tile_c) {
    float wt[W][VEC], bs[VEC];
#pragma unroll
    for (int k = 0; k < W; ++k) reinterpret_cast<const Raw<VEC> *>(s_w + k * tile_c)->to_float(wt[k]);
    reinterpret_cast<const Raw<VEC> *>(s_b)->to_float(bs);
    for (int r = 0; r < kRows; ++r) {
        if (lines[r] < 0) continue;
        const int b = rg * kRows + r;
        // A verify step that accepted k drafts reads its window k-1 columns in.
        int off = 0;
        if (a.nacc != nullptr) {
            off = __ldg(a.nacc + b) - 1;
            if (off < 0 || off + W - 1 > a.state_len) {
                count_error(a.err);
                continue;
            }
        }
        uint16_t *sp = a.st + lines[r] * a.ss_l + c0 * a.ss_d;
        Raw<VEC> win[W - 1];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) win[j] = gather<VEC>(sp + (off + j) * a.ss_t, a.ss_d, a.st_vec);
        float ring[W - 1][VEC];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) win[j].to_float(ring[j]);
        // Columns 0..W-3 take the window's columns 1..W-2; the new inputs go
        // to columns W-2 onwards.
        if (a.shift) {
#pragma unroll
            for (int j = 0; j + 1 < W - 1; ++j) scatter<VEC>(sp + j * a.ss_t, a.ss_d, a.st_vec, win[j + 1]);
        }
        const uint16_t *xp = a.x + b * a.xs_b + c0 * a.xs_d;
        uint16_t *op = a.out + b * a.os_b + c0 * a.os_d;
        for (int t = 0; t < a.seqlen; ++t) {
            const Raw<VEC> xr = gather<VEC>(xp + t * a.xs_t, a.xs_d, a.x_vec);
            float xf[VEC];
            xr.to_float(xf);
            Raw<VEC> o;
            conv_token<W, SILU, VEC>(wt, bs, ring, xf, o);
            scatter<VEC>(op + t * a.os_t, a.os_d, a.o_vec, o);
            if (a.shift) scatter<VEC>(sp + (W - 2 + t) * a.ss_t, a.ss_d, a.st_vec, xr);
#pragma unroll
            for (int k = 0; k < W - 2; ++k) {
                win[k] = win[k + 1];
#pragma unroll
                for (int v = 0; v < VEC; ++v) ring[k][v] = ring[k + 1][v];
            }
            win[W - 2] = xr;
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[W - 2][v] = xf[v];
            // win is now the window after token t.
            if (a.inter != nullptr) {
                uint16_t *ip = a.inter + b * a.is_b + t * a.is_t + c0 * a.is_d;
#pragma unroll
                for (int j = 0; j < W - 1; ++j) scatter<VEC>(ip + j * a.is_w, a.is_d, a.inter_vec, win[j]);
            }
            if (a.oidx != nullptr) {
                const int line = __ldg(a.oidx + b * a.ois_b + t * a.ois_t);
                if (line >= a.num_lines) {
                    count_error(a.err);
                } else if (line >= 0) {
                    uint16_t *dp = a.st + line * a.ss_l + c0 * a.ss_d;
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) scatter<VEC>(dp + j * a.ss_t, a.ss_d, a.st_vec, win[j]);
                }
            }
        }
    }
}

// A block covers kThreads*VEC channels of kRows consecutive batch rows.
// With 8-channel vectors this kernel only ever runs single-token rows without
// the spec extras (the host sends everything else to spec_kernel): weights
// and bias are requested first, overlapping the round trip for the rows'
// state-line indices, then every row's state window and input, then the
// mixed-precision taps.  With one channel per thread it is the general
// path: any seqlen, the spec extras, fp32 arithmetic.
template <int W, bool SILU, int VEC>
__global__ void __launch_bounds__(kThreads, VEC == 8 ? 7 : 1) update_kernel(const UpdArgs a) {
    release_next_grid();
    wait_prior_grid();
    constexpr int TILE_C = kThreads * VEC;
    const int rg = blockIdx.x / a.ctiles;
    const int ct = blockIdx.x - rg * a.ctiles;
    const int c0 = ct * TILE_C + threadIdx.x * VEC;
    const bool active = c0 < a.dim;

    if constexpr (VEC == 8) {
        // The state-line indices gate the only dependent loads, so they go
        // out first; the rows' inputs, the weights and the bias do not depend
        // on them and follow, so only the state windows wait for the lines.
        int lines[kRows];
        resolve_lines(a, rg, active, c0, lines);
        uint4 xv[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int b = rg * kRows + r;
            xv[r] = make_uint4(0u, 0u, 0u, 0u);
            if (active && b < a.batch) xv[r] = gather<8>(a.x + b * a.xs_b + c0 * a.xs_d, a.xs_d, a.x_vec).v;
        }
        uint4 wpk[W];
        float bs[8];
        if (active) {
            load_weights8<W>(a.w, a.ws_d, a.ws_k, c0, a.dim, a.w_vec, wpk);
            load_bias8(a.bias, c0, a.dim, a.b_vec, bs);
        }
        uint4 win[kRows][W - 1];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (lines[r] < 0) continue;
            const uint16_t *sp = a.st + lines[r] * a.ss_l + c0 * a.ss_d;
#pragma unroll
            for (int j = 0; j < W - 1; ++j) win[r][j] = gather<8>(sp + j * a.ss_t, a.ss_d, a.st_vec).v;
        }
        if (!active) return;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (lines[r] < 0) continue;
            const int b = rg * kRows + r;
            uint16_t *sp = a.st + lines[r] * a.ss_l + c0 * a.ss_d;
            Raw<8> o;
            o.v = decode_row<W, SILU>(wpk, bs, win[r], xv[r]);
            scatter<8>(a.out + b * a.os_b + c0 * a.os_d, a.os_d, a.o_vec, o);
            // The state keeps all but its oldest column and appends the input.
#pragma unroll
            for (int j = 0; j + 1 < W - 1; ++j) {
                Raw<8> keep;
                keep.v = win[r][j + 1];
                scatter<8>(sp + j * a.ss_t, a.ss_d, a.st_vec, keep);
            }
            Raw<8> xin;
            xin.v = xv[r];
            scatter<8>(sp + (W - 2) * a.ss_t, a.ss_d, a.st_vec, xin);
        }
    } else {
        __shared__ __align__(16) uint16_t s_w[W * TILE_C];
        __shared__ __align__(16) uint16_t s_b[TILE_C];
        int lines[kRows];
        resolve_lines(a, rg, active, c0, lines);
        stage_weights<W>(a, ct * TILE_C, TILE_C, s_w, s_b);
        if (!active) return;
        general_rows<W, SILU, VEC>(a, rg, c0, lines, s_w + threadIdx.x * VEC, s_b + threadIdx.x * VEC,
                                   TILE_C);
    }
}

// Multi-token and speculative-verify rows, 8 channels per thread, one row
// per thread: a chain of one memory round trip for the row's line and
// accepted-token count (with the weights, bias, and the first chunk of
// kSpecChunk tokens of x and their output-line indices), one for the
// window, then compute and stores; longer rows load further chunks.  In
// place (out == x) is safe: a token's x is loaded before its output is
// stored, by the same thread, and later chunks touch other tokens.
constexpr int kSpecThreads = 128;
constexpr int kSpecChunk = 4;

template <int W, bool SILU>
__global__ void __launch_bounds__(kSpecThreads) spec_kernel(const UpdArgs a) {
    release_next_grid();
    wait_prior_grid();
    const int b = blockIdx.x / a.ctiles;
    const int ct = blockIdx.x - b * a.ctiles;
    const int c0 = ct * kSpecThreads * 8 + threadIdx.x * 8;
    if (c0 >= a.dim || b >= a.batch) return;

    int line = a.idx ? __ldg(a.idx + b) : b;
    const int acc_tokens = a.nacc ? __ldg(a.nacc + b) : 1;
    uint4 wpk[W];
    load_weights8<W>(a.w, a.ws_d, a.ws_k, c0, a.dim, a.w_vec, wpk);
    float bs[8];
    load_bias8(a.bias, c0, a.dim, a.b_vec, bs);
    const uint16_t *xp = a.x + b * a.xs_b + c0 * a.xs_d;
    uint4 xv[kSpecChunk];
    int oline[kSpecChunk];
    // A chunk of x and its output-line indices; the first goes out with the
    // row's index loads (neither depends on the row's state line).
    auto load_chunk = [&](int t0) {
#pragma unroll
        for (int u = 0; u < kSpecChunk; ++u) {
            const int t = t0 + u;
            xv[u] = make_uint4(0u, 0u, 0u, 0u);
            oline[u] = -1;
            if (t < a.seqlen) {
                xv[u] = gather<8>(xp + t * a.xs_t, a.xs_d, a.x_vec).v;
                if (a.oidx != nullptr) oline[u] = __ldg(a.oidx + b * a.ois_b + t * a.ois_t);
            }
        }
    };
    load_chunk(0);
    if (line == a.pad) return;
    if (line < 0 || line >= a.num_lines) {
        count_error(a.err);
        return;
    }
    const int off = acc_tokens - 1;
    if (off < 0 || off + W - 1 > a.state_len) {
        count_error(a.err);
        return;
    }
    uint16_t *sp = a.st + line * a.ss_l + c0 * a.ss_d;
    uint16_t *op = a.out + b * a.os_b + c0 * a.os_d;
    uint4 win[W - 1];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) win[j] = gather<8>(sp + (off + j) * a.ss_t, a.ss_d, a.st_vec).v;

    for (int t0 = 0; t0 < a.seqlen; t0 += kSpecChunk) {
        if (t0 > 0) load_chunk(t0);
        if (t0 == 0 && a.shift) {
            // Columns 0..W-3 take the window's columns 1..W-2.
#pragma unroll
            for (int j = 0; j + 1 < W - 1; ++j) {
                Raw<8> keep;
                keep.v = win[j + 1];
                scatter<8>(sp + j * a.ss_t, a.ss_d, a.st_vec, keep);
            }
        }
#pragma unroll
        for (int u = 0; u < kSpecChunk; ++u) {
            const int t = t0 + u;
            if (t >= a.seqlen) break;
            Raw<8> o, xr;
            o.v = decode_row<W, SILU>(wpk, bs, win, xv[u]);
            xr.v = xv[u];
            scatter<8>(op + t * a.os_t, a.os_d, a.o_vec, o);
            if (a.shift) scatter<8>(sp + (W - 2 + t) * a.ss_t, a.ss_d, a.st_vec, xr);
#pragma unroll
            for (int j = 0; j < W - 2; ++j) win[j] = win[j + 1];
            win[W - 2] = xv[u];
            // win is now the window after token t.
            if (a.inter != nullptr) {
                uint16_t *ip = a.inter + b * a.is_b + t * a.is_t + c0 * a.is_d;
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    Raw<8> wj;
                    wj.v = win[j];
                    scatter<8>(ip + j * a.is_w, a.is_d, a.inter_vec, wj);
                }
            }
            if (oline[u] >= a.num_lines) {
                count_error(a.err);
            } else if (oline[u] >= 0) {
                uint16_t *dp = a.st + oline[u] * a.ss_l + c0 * a.ss_d;
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    Raw<8> wj;
                    wj.v = win[j];
                    scatter<8>(dp + j * a.ss_t, a.ss_d, a.st_vec, wj);
                }
            }
        }
    }
}

using KernelFn = void (*)(UpdArgs);

template <int VEC>
KernelFn pick_kernel(int width, bool silu) {
    switch (width) {
        case 2: return silu ? update_kernel<2, true, VEC> : update_kernel<2, false, VEC>;
        case 3: return silu ? update_kernel<3, true, VEC> : update_kernel<3, false, VEC>;
        case 4: return silu ? update_kernel<4, true, VEC> : update_kernel<4, false, VEC>;
        case 5: return silu ? update_kernel<5, true, VEC> : update_kernel<5, false, VEC>;
    }
    return nullptr;
}

KernelFn pick_spec_kernel(int width, bool silu) {
    switch (width) {
        case 2: return silu ? spec_kernel<2, true> : spec_kernel<2, false>;
        case 3: return silu ? spec_kernel<3, true> : spec_kernel<3, false>;
        case 4: return silu ? spec_kernel<4, true> : spec_kernel<4, false>;
        case 5: return silu ? spec_kernel<5, true> : spec_kernel<5, false>;
    }
    return nullptr;
}

}  // namespace
}  // namespace ccv

namespace ccv {
namespace {

struct SpecArgs {
    const int32_t *nacc = nullptr;
    void *inter = nullptr;
    int64_t is_b = 0, is_t = 0, is_d = 0, is_w = 0;
    int inter_steps = 0;
    const int32_t *oidx = nullptr;
    int64_t ois_b = 0, ois_t = 0;
    int oidx_steps = 0;
};

int update_launch(const void *x, int64_t x_stride_b, int64_t x_stride_dim, int64_t x_stride_tok,
                  void *out, int64_t out_stride_b, int64_t out_stride_dim, int64_t out_stride_tok,
                  const void *weight, int64_t w_stride_dim, int64_t w_stride_w, const void *bias,
                  void *conv_state, int64_t s_stride_line, int64_t s_stride_dim,
                  int64_t s_stride_tok, int num_cache_lines, int state_len,
                  const int32_t *conv_state_indices, const SpecArgs &sp, int batch, int dim,
                  int seqlen, int width, int pad_slot_id, int silu, int *err_count,
                  ccv_stream_t stream) {
    if (width < kMinWidth || width > kMaxWidth) return CCV_ERR_WIDTH;
    if (batch < 0 || dim < 0 || seqlen < 0 || num_cache_lines < 0) return CCV_ERR_SIZE;
    if (x_stride_b < 0 || x_stride_dim < 0 || x_stride_tok < 0 || out_stride_b < 0 ||
        out_stride_dim < 0 || out_stride_tok < 0 || w_stride_dim < 0 || w_stride_w < 0 ||
        s_stride_line < 0 || s_stride_dim < 0 || s_stride_tok < 0 || sp.is_b < 0 || sp.is_t < 0 ||
        sp.is_d < 0 || sp.is_w < 0 || sp.ois_b < 0 || sp.ois_t < 0)
        return CCV_ERR_STRIDE;
    const bool shift = sp.inter == nullptr && sp.oidx == nullptr;
    // Shifting writes width-2+seqlen columns; otherwise only the window's
    // width-1 columns are read (the accepted-token offset is checked per row).
    const int need = shift ? width - 2 + (seqlen > 0 ? seqlen : 1) : width - 1;
    if (state_len < need) return CCV_ERR_STATE_LEN;
    if ((sp.inter != nullptr && sp.inter_steps < seqlen) ||
        (sp.oidx != nullptr && sp.oidx_steps < seqlen))
        return CCV_ERR_CAPACITY;
    if (batch == 0 || dim == 0 || seqlen == 0) return CCV_OK;
    if (x == nullptr || out == nullptr || weight == nullptr || conv_state == nullptr)
        return CCV_ERR_NULL_POINTER;
    const bool in_place = x == out && x_stride_b == out_stride_b &&
                          x_stride_dim == out_stride_dim && x_stride_tok == out_stride_tok;
    const Extent ex = extent_of(x, batch, x_stride_b, dim, x_stride_dim, seqlen, x_stride_tok);
    const Extent eo = extent_of(out, batch, out_stride_b, dim, out_stride_dim, seqlen, out_stride_tok);
    if (!in_place && overlaps(ex, eo)) return CCV_ERR_ALIAS;
    if (sp.inter != nullptr) {
        const uintptr_t base = reinterpret_cast<uintptr_t>(sp.inter);
        const int64_t last = (batch - 1) * sp.is_b + (seqlen - 1) * sp.is_t +
                             (dim - 1) * sp.is_d + (width - 2) * sp.is_w;
        const Extent ei_full{base, base + static_cast<uintptr_t>(last) * 2u + 1u};
        const Extent es = extent_of(conv_state, num_cache_lines > 0 ? num_cache_lines : 1,
                                    s_stride_line, dim, s_stride_dim, state_len, s_stride_tok);
        if (overlaps(ei_full, ex) || overlaps(ei_full, eo) || overlaps(ei_full, es))
            return CCV_ERR_ALIAS;
    }

    UpdArgs a;
    a.x = static_cast<const uint16_t *>(x);
    a.xs_b = x_stride_b;
    a.xs_d = x_stride_dim;
    a.xs_t = x_stride_tok;
    a.out = static_cast<uint16_t *>(out);
    a.os_b = out_stride_b;
    a.os_d = out_stride_dim;
    a.os_t = out_stride_tok;
    a.w = static_cast<const uint16_t *>(weight);
    a.ws_d = w_stride_dim;
    a.ws_k = w_stride_w;
    a.bias = static_cast<const uint16_t *>(bias);
    a.st = static_cast<uint16_t *>(conv_state);
    a.ss_l = s_stride_line;
    a.ss_d = s_stride_dim;
    a.ss_t = s_stride_tok;
    a.num_lines = num_cache_lines;
    a.idx = conv_state_indices;
    a.batch = batch;
    a.dim = dim;
    a.seqlen = seqlen;
    a.pad = pad_slot_id;
    a.err = err_count;
    a.state_len = state_len;
    a.nacc = sp.nacc;
    a.inter = static_cast<uint16_t *>(sp.inter);
    a.is_b = sp.is_b;
    a.is_t = sp.is_t;
    a.is_d = sp.is_d;
    a.is_w = sp.is_w;
    a.oidx = sp.oidx;
    a.ois_b = sp.ois_b;
    a.ois_t = sp.ois_t;
    a.shift = shift;
    a.plain = shift && sp.nacc == nullptr;

    const bool vec = dim % 8 == 0;
    const int vw = vec ? 8 : 1;
    a.x_vec = vec && x_stride_dim == 1 && aligned16(x) && x_stride_b % 8 == 0 &&
              (seqlen == 1 || x_stride_tok % 8 == 0);
    a.o_vec = vec && out_stride_dim == 1 && aligned16(out) && out_stride_b % 8 == 0 &&
              (seqlen == 1 || out_stride_tok % 8 == 0);
    a.st_vec = vec && s_stride_dim == 1 && aligned16(conv_state) && s_stride_line % 8 == 0 &&
               s_stride_tok % 8 == 0;
    a.inter_vec = vec && sp.inter != nullptr && sp.is_d == 1 && aligned16(sp.inter) &&
                  sp.is_b % 8 == 0 && sp.is_t % 8 == 0 && sp.is_w % 8 == 0;
    a.w_vec = w_stride_w == 1 && w_stride_dim == width && aligned16(weight);
    a.b_vec = bias != nullptr && aligned16(bias);
    if (vec && !(seqlen == 1 && a.plain)) {
        // several tokens per row, or the speculative-decoding extras
        a.ctiles = (dim + kSpecThreads * 8 - 1) / (kSpecThreads * 8);
        const int64_t blocks = static_cast<int64_t>(batch) * a.ctiles;
        if (blocks > 0x7fffffffLL) return CCV_ERR_SIZE;
        return launch_pdl(pick_spec_kernel(width, silu != 0), dim3(static_cast<unsigned>(blocks)),
                          dim3(kSpecThreads), 0, stream, a);
    }
    a.ctiles = (dim + kThreads * vw - 1) / (kThreads * vw);
    const int64_t blocks = static_cast<int64_t>((batch + kRows - 1) / kRows) * a.ctiles;
    if (blocks > 0x7fffffffLL) return CCV_ERR_SIZE;
    KernelFn fn = vec ? pick_kernel<8>(width, silu != 0) : pick_kernel<1>(width, silu != 0);
    return launch_pdl(fn, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream, a);
}

}  // namespace
}  // namespace ccv

extern "C" int ccv_update(const void *x, int64_t x_stride_b, int64_t x_stride_dim,
                          int64_t x_stride_tok, void *out, int64_t out_stride_b,
                          int64_t out_stride_dim, int64_t out_stride_tok, const void *weight,
                          int64_t w_stride_dim, int64_t w_stride_w, const void *bias,
                          void *conv_state, int64_t s_stride_line, int64_t s_stride_dim,
                          int64_t s_stride_tok, int num_cache_lines, int state_len,
                          const int32_t *conv_state_indices, int batch, int dim, int seqlen,
                          int width, int pad_slot_id, int silu, int *err_count,
                          ccv_stream_t stream) {
    return ccv::update_launch(x, x_stride_b, x_stride_dim, x_stride_tok, out, out_stride_b,
                              out_stride_dim, out_stride_tok, weight, w_stride_dim, w_stride_w,
                              bias, conv_state, s_stride_line, s_stride_dim, s_stride_tok,
                              num_cache_lines, state_len, conv_state_indices, ccv::SpecArgs{},
                              batch, dim, seqlen, width, pad_slot_id, silu, err_count, stream);
}

extern "C" int ccv_update_spec(const void *x, int64_t x_stride_b, int64_t x_stride_dim,
                               int64_t x_stride_tok, void *out, int64_t out_stride_b,
                               int64_t out_stride_dim, int64_t out_stride_tok, const void *weight,
                               int64_t w_stride_dim, int64_t w_stride_w, const void *bias,
                               void *conv_state, int64_t s_stride_line, int64_t s_stride_dim,
                               int64_t s_stride_tok, int num_cache_lines, int state_len,
                               const int32_t *conv_state_indices,
                               const int32_t *num_accepted_tokens,
                               void *intermediate_conv_window, int64_t i_stride_b,
                               int64_t i_stride_step, int64_t i_stride_dim, int64_t i_stride_win,
                               int inter_steps, const int32_t *output_state_indices,
                               int64_t oi_stride_b, int64_t oi_stride_step, int oidx_steps,
                               int batch, int dim, int seqlen, int width, int pad_slot_id,
                               int silu, int *err_count, ccv_stream_t stream) {
    ccv::SpecArgs sp;
    sp.nacc = num_accepted_tokens;
    sp.inter = intermediate_conv_window;
    sp.is_b = i_stride_b;
    sp.is_t = i_stride_step;
    sp.is_d = i_stride_dim;
    sp.is_w = i_stride_win;
    sp.inter_steps = inter_steps;
    sp.oidx = output_state_indices;
    sp.ois_b = oi_stride_b;
    sp.ois_t = oi_stride_step;
    sp.oidx_steps = oidx_steps;
    return ccv::update_launch(x, x_stride_b, x_stride_dim, x_stride_tok, out, out_stride_b,
                              out_stride_dim, out_stride_tok, weight, w_stride_dim, w_stride_w,
                              bias, conv_state, s_stride_line, s_stride_dim, s_stride_tok,
                              num_cache_lines, state_len, conv_state_indices, sp, batch, dim,
                              seqlen, width, pad_slot_id, silu, err_count, stream);
}
