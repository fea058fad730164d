// ccv_update: decode step of the causal depthwise conv1d with an in-place
// conv_state shift.
//
// Semantics: tokenspeed causal_conv1d.py, `causal_conv1d_update` and
// `_causal_conv1d_update_kernel` (STEP 1 read the state window, STEP 2 shift
// the state left and append the new inputs, STEPS 3-5 bias, weights and the
// token loop), non-speculative path.
//
// One thread owns 8 consecutive channels (16-byte vectors) of one batch row;
// the grid is batch x ceil(dim / 1024) blocks, fixed by the sizes, so a CUDA
// graph replays it unchanged.  Every element of the state line and of out is
// read and written by the same thread, which makes the in-place state shift
// and out == x (the page's wrapper writes the output over x) hazard-free.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kThreads = 128;

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

template <int VEC>
__device__ __forceinline__ void scatter(uint16_t *p, int64_t stride, bool vec, const Raw<VEC> &r) {
    if (VEC == 8 && vec) {
        store_plain<VEC>(p, r);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) p[v * stride] = r.elem(v);
    }
}

template <int W, bool SILU, int VEC>
__global__ void __launch_bounds__(kThreads) update_kernel(const UpdArgs a) {
    const int b = blockIdx.x / a.ctiles;
    const int ct = blockIdx.x - b * a.ctiles;
    const int c0 = (ct * kThreads + threadIdx.x) * VEC;
    if (c0 >= a.dim) return;
    const int line = a.idx ? __ldg(a.idx + b) : b;
    if (line == a.pad) return;
    if (line < 0 || line >= a.num_lines) {
        if (c0 == 0) count_error(a.err);
        return;
    }

    float wt[W][VEC], bs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) wt[k][v] = bf16_bits(__ldg(a.w + (c0 + v) * a.ws_d + k * a.ws_k));
        bs[v] = a.bias ? bf16_bits(__ldg(a.bias + c0 + v)) : 0.0f;
    }

    uint16_t *sp = a.st + line * a.ss_l + c0 * a.ss_d;
    Raw<VEC> win[W - 1];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) win[j] = gather<VEC>(sp + j * a.ss_t, a.ss_d, a.st_vec);
    float ring[W - 1][VEC];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) win[j].to_float(ring[j]);
    // The state keeps everything but its oldest column: columns 0..W-3 take
    // the old columns 1..W-2; the new inputs go to columns W-2 onwards.
#pragma unroll
    for (int j = 0; j + 1 < W - 1; ++j) scatter<VEC>(sp + j * a.ss_t, a.ss_d, a.st_vec, win[j + 1]);

    const uint16_t *xp = a.x + b * a.xs_b + c0 * a.xs_d;
    uint16_t *op = a.out + b * a.os_b + c0 * a.os_d;
    for (int t = 0; t < a.seqlen; ++t) {
        const Raw<VEC> xv = gather<VEC>(xp + t * a.xs_t, a.xs_d, a.x_vec);
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
        scatter<VEC>(op + t * a.os_t, a.os_d, a.o_vec, o);
        scatter<VEC>(sp + (W - 2 + t) * a.ss_t, a.ss_d, a.st_vec, xv);
#pragma unroll
        for (int k = 0; k < W - 2; ++k)
#pragma unroll
            for (int v = 0; v < VEC; ++v) ring[k][v] = ring[k + 1][v];
#pragma unroll
        for (int v = 0; v < VEC; ++v) ring[W - 2][v] = xf[v];
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
    using namespace ccv;
    if (width < kMinWidth || width > kMaxWidth) return CCV_ERR_WIDTH;
    if (batch < 0 || dim < 0 || seqlen < 0 || num_cache_lines < 0) return CCV_ERR_SIZE;
    if (x_stride_b < 0 || x_stride_dim < 0 || x_stride_tok < 0 || out_stride_b < 0 ||
        out_stride_dim < 0 || out_stride_tok < 0 || w_stride_dim < 0 || w_stride_w < 0 ||
        s_stride_line < 0 || s_stride_dim < 0 || s_stride_tok < 0)
        return CCV_ERR_STRIDE;
    if (state_len < width - 2 + (seqlen > 0 ? seqlen : 1)) return CCV_ERR_STATE_LEN;
    if (batch == 0 || dim == 0 || seqlen == 0) return CCV_OK;
    if (x == nullptr || out == nullptr || weight == nullptr || conv_state == nullptr)
        return CCV_ERR_NULL_POINTER;
    const bool in_place = x == out && x_stride_b == out_stride_b &&
                          x_stride_dim == out_stride_dim && x_stride_tok == out_stride_tok;
    if (!in_place &&
        overlaps(extent_of(x, batch, x_stride_b, dim, x_stride_dim, seqlen, x_stride_tok),
                 extent_of(out, batch, out_stride_b, dim, out_stride_dim, seqlen, out_stride_tok)))
        return CCV_ERR_ALIAS;

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

    const bool vec = dim % 8 == 0;
    const int vw = vec ? 8 : 1;
    a.x_vec = vec && x_stride_dim == 1 && aligned16(x) && x_stride_b % 8 == 0 &&
              (seqlen == 1 || x_stride_tok % 8 == 0);
    a.o_vec = vec && out_stride_dim == 1 && aligned16(out) && out_stride_b % 8 == 0 &&
              (seqlen == 1 || out_stride_tok % 8 == 0);
    a.st_vec = vec && s_stride_dim == 1 && aligned16(conv_state) && s_stride_line % 8 == 0 &&
               s_stride_tok % 8 == 0;
    a.ctiles = (dim + kThreads * vw - 1) / (kThreads * vw);
    const int64_t blocks = static_cast<int64_t>(batch) * a.ctiles;
    if (blocks > 0x7fffffffLL) return CCV_ERR_SIZE;
    KernelFn fn = vec ? pick_kernel<8>(width, silu != 0) : pick_kernel<1>(width, silu != 0);
    fn<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
    return launch_status();
}
