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
// and bounded by floor(total_tokens / CHUNK) + batch, so a block finds its
// sequence from its slot by a binary search over query_start_loc and surplus
// blocks exit.
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
//
// Short problems (total_tokens * dim up to kShortMaxElems) take two more
// kernels, one per layout, built for latency instead of streaming.
//
// The note on the streaming kernels' launches.  Every kernel is launched
// with programmatic stream serialization and waits for its predecessor
// before touching memory.  The streaming kernels do not release their own
// successor early: they run many waves, and letting the next kernel take
// their SMs during their last wave made a bench step (channel-last prefill,
// channel-first prefill, decode, paged) 4% slower on GB300, while launches
// of the same kernel back to back gained nothing from it (measured).  The
// short kernels, one wave each, release at once.
#include <cstdlib>
#include <cstring>
#include <type_traits>
#include <utility>

#include "ccv_common.cuh"
#include "ccv_math2.cuh"
#include "ccv_pipeline.cuh"

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

// One thread of the work unit (block or warp) of chunk slot i < batch in
// the first channel tile checks sequence i's indices and counts invalid
// ones; the chunk units skip such sequences silently.  validate_sequence:
// slot blockIdx.x, tile blockIdx.y, thread 0.
__device__ __forceinline__ void validate_sequence_at(const FwdArgs &a, int i, bool lead) {
    if (a.err == nullptr || !lead) return;
    if (i >= a.batch) return;
    const int line = a.cidx ? __ldg(a.cidx + i) : i;
    if (line == a.pad) return;
    const int s = __ldg(a.qsl + i), e = __ldg(a.qsl + i + 1);
    bool bad = s < 0 || e < s || e > a.total;
    if (!bad && a.st != nullptr && e > s && (line < 0 || line >= a.num_lines)) bad = true;
    if (bad) atomicAdd(a.err, 1);
}
__device__ __forceinline__ void validate_sequence(const FwdArgs &a) {
    validate_sequence_at(a, blockIdx.x, blockIdx.y == 0 && threadIdx.x == 0);
}

// Resolve the state line of the chunk's sequence; false = skip the sequence.
__device__ __forceinline__ bool sequence_line(const FwdArgs &a, const ChunkInfo &ci, int &line) {
    line = a.cidx ? __ldg(a.cidx + ci.seq) : ci.seq;
    if (line == a.pad) return false;
    if (a.st != nullptr && (line < 0 || line >= a.num_lines)) return false;
    return true;
}

struct SeqChunk {
    int seq, chunk, start, len, line;
    bool init;
};

// Slot -> (sequence, chunk) as locate_chunk, plus the sequence's state line
// and has_initial_state flag, in one round trip for up to 32 * PER
// sequences: lane l of the final round loads candidates PER*l .. PER*l+PER-1
// of the window (their offsets, lines and flags together), and the winner's
// are shuffled to every lane.  false for a surplus slot, a pad or invalid
// line, or bad offsets.
template <int PER>
__device__ __forceinline__ bool locate_seq(const FwdArgs &a, int chunk_tokens, int slot, SeqChunk &sc) {
    const int lane = threadIdx.x & 31;
    int lo = 0, n = a.batch;
    while (n > 32 * PER) {  // narrow to at most 32 * PER candidates
        const int stride = (n + 31) >> 5;
        const int off = lane * stride;
        bool le = false;
        if (off < n) {
            const int i = lo + off;
            le = floor_div(__ldg(a.qsl + i), chunk_tokens) + i <= slot;
        }
        const unsigned m = __ballot_sync(kFullMask, le);
        if (m == 0u) return false;
        const int top = 31 - __clz(m);
        lo += top * stride;
        n = min(stride, n - top * stride);
    }
    const int base = PER * lane;  // this lane's first candidate, from lo
    int s[PER + 1], line[PER], init[PER];
#pragma unroll
    for (int k = 0; k <= PER; ++k) s[k] = base + k <= n ? __ldg(a.qsl + lo + base + k) : 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = lo + base + k;
        const bool in = base + k < n;
        line[k] = in ? (a.cidx ? __ldg(a.cidx + i) : i) : 0;
        init[k] = in && a.has_init != nullptr ? a.has_init[i] : 0;
    }
    int pick = -1;  // this lane's last candidate at or before the slot
#pragma unroll
    for (int k = 0; k < PER; ++k)
        if (base + k < n && floor_div(s[k], chunk_tokens) + lo + base + k <= slot) pick = k;
    const unsigned m = __ballot_sync(kFullMask, pick >= 0);
    if (m == 0u) return false;
    const int top = 31 - __clz(m);
    int ps = 0, pe = 0, pl = 0, pi = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        if (k == pick) {
            ps = s[k];
            pe = s[k + 1];
            pl = line[k];
            pi = init[k];
        }
    }
    sc.seq = lo + PER * top + __shfl_sync(kFullMask, pick, top);
    sc.start = __shfl_sync(kFullMask, ps, top);
    const int end = __shfl_sync(kFullMask, pe, top);
    sc.line = __shfl_sync(kFullMask, pl, top);
    sc.init = a.st != nullptr && __shfl_sync(kFullMask, pi, top) != 0;
    if (sc.start < 0 || end < sc.start || end > a.total) return false;
    const int k = slot - (sc.start / chunk_tokens + sc.seq);
    if (k < 0 || static_cast<int64_t>(k) * chunk_tokens >= end - sc.start) return false;
    if (sc.line == a.pad) return false;
    if (a.st != nullptr && (sc.line < 0 || sc.line >= a.num_lines)) return false;
    sc.chunk = k;
    sc.len = end - sc.start;
    return true;
}
__device__ __forceinline__ bool locate_short(const FwdArgs &a, int chunk_tokens, int slot, SeqChunk &sc) {
    return locate_seq<1>(a, chunk_tokens, slot, sc);
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
    wait_prior_grid();  // no early release: see the note on the streaming kernels' launches
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
    wait_prior_grid();  // no early release: see the note on the streaming kernels' launches
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

// ------------------------------------------ channel-last, cp.async ----
//
// One block owns one (sequence chunk of kCaChunk tokens, 256-channel tile);
// warp w takes the chunk's w-th run of kCaRun tokens, lane l channels
// 8l..8l+7 of the tile.  Each thread streams its rows through a private ring
// of kCaSlots 16-byte shared-memory slots with cp.async, keeping kCaSlots-1
// rows in flight at no register cost, and reads back only what it copied
// (so no barrier is needed).  The row loop is unrolled by the ring size so
// slot offsets are constants and the W-1 previous rows are renamed rather
// than moved.  Weights stay packed bf16x2 and feed native mixed-precision
// bf16 x bf16 + fp32 FMAs (one rounding, the same value as the fp32 fma of
// the widened operands); the bias enters through the first tap.  The first
// run of a sequence takes its prior from conv_state, the others from the W-1
// rows before the run.

constexpr int kCaThreads = 256;
constexpr int kCaWarps = kCaThreads / 32;
constexpr int kCaRun = 32;
constexpr int kCaChunk = kCaWarps * kCaRun;
constexpr int kCaSlots = 16;
constexpr int kCaTileC = 256;
constexpr size_t kCaSmem = sizeof(uint4) * kCaSlots * kCaThreads;  // dynamic: the slot rings

// A warp's W-1 halo rows are read twice: by this warp first, and by the warp
// that owns them (the previous warp of the block, or the last warp of the
// previous chunk's block) at the end of its run, about one block lifetime
// (~15 us) later.  Copying them with the evict-last L2 policy keeps them
// resident until that second read; with the default policy part of them had
// left L2 and came from DRAM twice (measured: the kernel 2.6 us faster).
__device__ __forceinline__ void cp_async16_keep(void *smem_dst, const void *gmem_src) {
    uint64_t policy;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
                 "l"(gmem_src), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint4 load8_state(const FwdArgs &a, int line, int c0, int col) {
    const uint16_t *p = a.st + line * a.ss_l + c0 * a.ss_d + col * a.ss_t;
    if (a.st_vec) return *reinterpret_cast<const uint4 *>(p);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = uint32_t(p[(2 * q) * a.ss_d]) | (uint32_t(p[(2 * q + 1) * a.ss_d]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void store8_state(const FwdArgs &a, int line, int c0, int col, uint4 v) {
    uint16_t *p = a.st + line * a.ss_l + c0 * a.ss_d + col * a.ss_t;
    if (a.st_vec) {
        *reinterpret_cast<uint4 *>(p) = v;
        return;
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        p[(2 * q) * a.ss_d] = uint16_t(w[q] & 0xffffu);
        p[(2 * q + 1) * a.ss_d] = uint16_t(w[q] >> 16);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// One output row of 8 channels: taps over ring[0..W-2] (oldest first) and v.
template <int W, bool SILU>
__device__ __forceinline__ uint4 ca_row(const uint4 (&wpk)[W], const float (&bs)[8],
                                        const uint4 (&ring)[W - 1], const uint4 &v) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        fma_bf16x2_init(acc[2 * q], acc[2 * q + 1], word_of(ring[0], q), word_of(wpk[0], q),
                        bs[2 * q], bs[2 * q + 1]);
#pragma unroll
    for (int k = 1; k < W; ++k) {
        const uint4 &u = k < W - 1 ? ring[k < W - 1 ? k : 0] : v;
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

// Three blocks per SM; W = 5 with SiLU does not fit their register share
// without spilling, so it runs at two (measured faster).
template <int W, bool SILU>
__global__ void __launch_bounds__(kCaThreads, W == 5 ? 2 : 3) fwd_cl_async_kernel(const FwdArgs a) {
    extern __shared__ __align__(16) uint4 s_ring[];  // [kCaSlots][kCaThreads]
    __shared__ __align__(16) uint16_t s_w[W * kCaTileC];
    __shared__ __align__(16) uint16_t s_b[kCaTileC];
    wait_prior_grid();  // no early release: see the note on the streaming kernels' launches
    // One-dimensional grid, block = slot * tiles + tile: channel tiles vary
    // fastest in launch order, so the blocks resident at one time read whole
    // token rows (3% faster than chunk-major order, measured).
    const int ntiles = (a.dim + kCaTileC - 1) / kCaTileC;
    const int tile = static_cast<int>(blockIdx.x % static_cast<unsigned>(ntiles));
    const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(ntiles));
    validate_sequence_at(a, slot, tile == 0 && threadIdx.x == 0);
    ChunkInfo ci;
    if (!locate_chunk(a, kCaChunk, slot, ci)) return;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int c0 = tile * kCaTileC + lane * 8;
    const int cbeg = ci.start + ci.chunk * kCaChunk;
    const int cend = ci.start + min(ci.len, (ci.chunk + 1) * kCaChunk);
    const int r0 = cbeg + warp * kCaRun;
    const int r1 = min(r0 + kCaRun, cend);
    const bool first = ci.chunk == 0 && warp == 0;
    const int h = first ? 0 : W - 1;  // halo rows streamed before the run
    const int row_base = r0 - h;
    const int nrows = r1 > r0 ? r1 - row_base : 0;
    const bool active = c0 < a.dim && nrows > 0;
    const int64_t xs = a.xs_t;
    const uint16_t *src = a.x + c0 + row_base * xs;
    uint4 *ring_base = s_ring + tid;

    // Start the stream before anything else; slot j % kCaSlots holds row j
    // (rows j < h are the halo).
#pragma unroll
    for (int j = 0; j < kCaSlots - 1; ++j) {
        if (active && j < nrows) {
            if (j < h) cp_async16_keep(ring_base + j * kCaThreads, src + j * xs);
            else cp_async16(ring_base + j * kCaThreads, src + j * xs);
        }
        cp_async_commit();
    }
    // The state line is looked up while the stream is in flight; a skipped
    // sequence waits for its copies so that nothing lands after it exits.
    int line;
    if (!sequence_line(a, ci, line)) {
        cp_async_wait<0>();
        return;
    }
    // The state line and the has_initial_state flag do not depend on each
    // other: both loads go out with the stream, before the weights.
    uint4 prior[W - 1];
    bool init = false;
    if (first && active && a.st != nullptr) {
        init = a.has_init != nullptr && a.has_init[ci.seq] != 0;
#pragma unroll
        for (int j = 0; j < W - 1; ++j) prior[j] = load8_state(a, line, c0, j);
    }
    stage_weights<W>(a.w, a.ws_d, a.ws_k, a.bias, a.dim, tile * kCaTileC, kCaTileC, s_w, s_b);
    if (!active) return;

    uint4 wpk[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wpk[k] = reinterpret_cast<const uint4 *>(s_w + k * kCaTileC)[lane];
    float bs[8];
    reinterpret_cast<const Raw<8> *>(s_b)[lane].to_float(bs);

    uint4 ring[W - 1];
    if (first) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            if (!init) prior[j] = make_uint4(0u, 0u, 0u, 0u);
            ring[j] = prior[j];
        }
        if (a.st != nullptr) {
            // New state = last W-1 entries of prior ++ x[sequence].
            uint4 nw[W - 1];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) {
                const int idx = ci.len + j;
                if (idx < W - 1) {
#pragma unroll
                    for (int q = 0; q < W - 1; ++q)
                        if (q == idx) nw[j] = prior[q];
                } else {
                    nw[j] = *reinterpret_cast<const uint4 *>(a.x + c0 + (ci.start + idx - (W - 1)) * xs);
                }
            }
#pragma unroll
            for (int j = 0; j < W - 1; ++j) store8_state(a, line, c0, j, nw[j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) ring[j] = make_uint4(0u, 0u, 0u, 0u);
    }

    const int64_t os = a.os_t;
    uint16_t *dst = a.out + c0 + row_base * os;
    const uint16_t *nxt = src + (kCaSlots - 1) * xs;  // next row to stream in
    // One row: wait for it, refill the slot read in the previous step, compute.
    auto step = [&](int j, int slot) {
        cp_async_wait<kCaSlots - 2>();
        const uint4 v = ring_base[slot * kCaThreads];
        if (j + kCaSlots - 1 < nrows)
            cp_async16(ring_base + ((slot + kCaSlots - 1) % kCaSlots) * kCaThreads, nxt);
        cp_async_commit();
        nxt += xs;
        if (j >= h) __stcs(reinterpret_cast<uint4 *>(dst), ca_row<W, SILU>(wpk, bs, ring, v));
        dst += os;
#pragma unroll
        for (int k = 0; k < W - 2; ++k) ring[k] = ring[k + 1];
        ring[W - 2] = v;
    };
    int j = 0;
    for (; j + kCaSlots <= nrows; j += kCaSlots) {
#pragma unroll
        for (int u = 0; u < kCaSlots; ++u) step(j + u, u);
    }
    for (int u = 0; j < nrows; ++j, ++u) step(j, u);
}

// ----------------------------------------- channel-first, cp.async ----
//
// One warp owns one channel row of one sequence chunk of kCfaChunk tokens (a
// block holds kCfaWarps consecutive rows).  The chunk is kCfaSegs warp-wide
// segments of 256 tokens (512 bytes) that start on a 256-byte boundary of
// the row's memory, at or before the first token needed (the chunk length
// leaves room for the halo and the alignment): every warp access then covers
// whole 32-byte sectors and exactly two 256-byte blocks of memory (about 4%
// faster than 16-byte alignment, measured).  Lane l owns tokens 8l..8l+7
// of a segment.  Each lane streams its 16-byte vectors through a private
// ring of kCfaSlots shared-memory slots with cp.async, started as soon as
// the chunk is known, edge segments included: the tokens outside the chunk
// that a vector carries feed no stored output, and the W-1 tokens before a
// sequence's first chunk take the prior when segment 0 is read.  The chunk
// search returns the sequence's state line and flag with its offsets in one
// round trip for up to 128 sequences, so the prior and the x entries of the
// new state load while the ring fills (with the edges assembled from scalar
// loads after the prior and the search taking up to three round trips, 64
// sequences of 1024 tokens ran at half the copy rate).
// The 4 tokens before a lane's vector come from lane l-1 by shuffle (lane 0:
// lane 31 of the previous segment).  Taps are native bf16 x bf16 + fp32
// FMAs on the packed 12-token window; segments wholly inside the chunk run
// without per-lane checks.  Outputs are written with plain stores, not the
// evict-first hint of the channel-last kernel: with plain stores the prefill
// parts and the whole step ran 1.7% faster (measured; for the channel-last
// kernel the hint is the faster choice).
//
// The chunk length CHUNK is chosen on the host from total_tokens and batch
// (cf_long_chunks) and the grid has total_tokens / CHUNK + batch chunk slots
// per row group, an upper bound computed without reading query_start_loc;
// the surplus slots exit after the chunk search.  Sequences of up to 16384
// tokens on average take one kCfaChunk-token chunk (128 segments) each and
// leave few surplus slots (8056-token chunks left a third of the blocks
// empty on 4 x 4096 tokens and split 11027-token sequences unevenly:
// 83.4 -> 82.1 us and 67.7 -> 59.7 us, measured); longer sequences keep
// 8056-token chunks (one 32632-token chunk plus a short one took 1 x 40000
// tokens from 197 to 214 us).

constexpr int kCfaThreads = 256;
constexpr int kCfaWarps = kCfaThreads / 32;
constexpr int kCfaSegs = 128;
constexpr int kCfaAlign = 128;  // tokens: segments start on a 256-byte boundary
constexpr int kCfaChunk = kCfaSegs * 256 - kCfaAlign - 8;  // + halo (<= 4) + alignment (< 128)
constexpr int kCfaChunkSplit = 32 * 256 - kCfaAlign - 8;      // 8056: chunks of long sequences
constexpr int kCfaSlots = 8;
constexpr int kCfaPer = 4;  // sequences per lane in the chunk search: one round trip up to 128
constexpr size_t kCfaSmem = sizeof(uint4) * kCfaSlots * kCfaThreads;
static_assert(kCfaChunk + kMaxWidth - 1 + kCfaAlign - 1 <= kCfaSegs * 256, "a chunk must fit its segments");
// Segment 1 must start after the chunk's first token (it runs unchecked).
static_assert(256 - (kCfaAlign - 1) - (kMaxWidth - 1) > 0, "segment 1 must lie inside the chunk");

__device__ __forceinline__ void cfa_store(uint16_t *p, const uint4 &v) { *reinterpret_cast<uint4 *>(p) = v; }

// The 8 inputs at tokens t0..t0+7 of one row where the 16-byte vector
// crosses an end of the row (rows that do not start on a 16-byte boundary):
// x inside [0, total), 0 outside.
__device__ __noinline__ uint4 cfa_ragged_vector(const uint16_t *xc, int t0, int total) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t pair = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = t0 + 2 * q + e;
            if (t >= 0 && t < total) pair |= uint32_t(xc[t]) << (16 * e);
        }
        w[q] = pair;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// A sequence's first chunk: tokens cbeg-(W-1) .. cbeg-1 of the vector at
// t0 take the prior (its W-1 columns packed oldest first, 0 without an
// initial state) in place of the x of whatever precedes the sequence.
template <int W>
__device__ __forceinline__ uint4 cfa_with_prior(const uint4 &v, int t0, int cbeg, uint32_t prior01,
                                                uint32_t prior23) {
    if (t0 + 8 <= cbeg - (W - 1) || t0 >= cbeg) return v;
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = t0 + 2 * q + e - cbeg + (W - 1);  // prior column
            if (i >= 0 && i < W - 1) {
                const uint32_t src = i < 2 ? prior01 : prior23;
                const uint32_t val = (i & 1) ? (src >> 16) : (src & 0xffffu);
                w[q] = (w[q] & (0xffff0000u >> (16 * e))) | (val << (16 * e));
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// f(std::integral_constant<int, i>{}) for i = 0 .. N-1, in order: a loop
// whose index is a compile-time constant inside the body.
template <typename F, int... I>
__device__ __forceinline__ void static_for_seq(F &&f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    static_for_seq(f, std::make_integer_sequence<int, N>{});
}

// One accumulator from one bf16 half of a packed word: half H (0 = low,
// 1 = high) of x times the low half of w, fp32 accumulate, one rounding.
// INIT: acc = x_H * w + b; otherwise acc += x_H * w.
template <int H, bool INIT>
__device__ __forceinline__ void fma_bf16_half(float &acc, uint32_t x, uint32_t w, float b) {
    static_assert(H == 0 || H == 1, "a bf16x2 word has two halves");
    if constexpr (INIT && H == 0)
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xl, wl, %3;\n\t}" : "=f"(acc) : "r"(x), "r"(w), "f"(b));
    else if constexpr (INIT)
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xh, wl, %3;\n\t}" : "=f"(acc) : "r"(x), "r"(w), "f"(b));
    else if constexpr (H == 0)
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t}" : "+f"(acc) : "r"(x), "r"(w));
    else
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, xh, wl, %0;\n\t}" : "+f"(acc) : "r"(x), "r"(w));
}

// One segment's worth of outputs for one lane: tokens t0..t0+7 from the
// 12-token window E (6 bf16x2 words, tokens t0-4 .. t0+7).  Output 2p takes
// tap k from window token i = 2p+5-W+k and output 2p+1 from token i+1; each
// token is read as its half of its word, so a pair that straddles two words
// needs no permute.  Native bf16 x bf16 + fp32 FMAs (bias first, then taps
// 0..W-1, one rounding each).
template <int W, bool SILU>
__device__ __forceinline__ uint4 cfa_outputs(const uint32_t (&E)[6], const uint32_t (&wb)[W], float bs) {
    uint32_t ow[4];
    static_for<4>([&](auto P) {
        constexpr int p = decltype(P)::value;
        float lo, hi;
        static_for<W>([&](auto K) {
            constexpr int k = decltype(K)::value;
            constexpr int i = 2 * p + 5 - W + k;
            fma_bf16_half<i & 1, k == 0>(lo, E[i >> 1], wb[k], bs);
            fma_bf16_half<(i + 1) & 1, k == 0>(hi, E[(i + 1) >> 1], wb[k], bs);
        });
        f32x2 r = pack2(lo, hi);
        if (SILU) r = silu2(r);
        ow[p] = f32x2_to_bf16x2(r);
    });
    return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

template <int W, bool SILU, int CHUNK>
__global__ void __launch_bounds__(kCfaThreads, 4) fwd_cf_async_kernel(const FwdArgs a) {
    extern __shared__ __align__(16) uint4 s_ring[];  // [kCfaSlots][kCfaThreads]
    wait_prior_grid();  // no early release: see the note on the streaming kernels' launches
    validate_sequence(a);
    SeqChunk sc;  // the chunk, its sequence's state line and flag: one round trip
    if (!locate_seq<kCfaPer>(a, CHUNK, blockIdx.x, sc)) return;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int c = blockIdx.y * kCfaWarps + (tid >> 5);
    if (c >= a.dim) return;  // warp-uniform

    const uint16_t *const xc = a.x + c * a.xs_d;
    const int cbeg = sc.start + sc.chunk * CHUNK;
    const int cend = sc.start + min(sc.len, (sc.chunk + 1) * CHUNK);
    const bool chunk0 = sc.chunk == 0;
    const bool keep = chunk0 && a.st != nullptr;  // this chunk reads and writes the state line
    // where the row starts within its 256-byte block of memory, in tokens
    const int phase = static_cast<int>((reinterpret_cast<uintptr_t>(xc) >> 1) & (kCfaAlign - 1));
    // first token of segment 0: aligned, at or before the first token needed
    const int need0 = cbeg - (W - 1);
    const int a0 = need0 - ((phase + need0) & (kCfaAlign - 1));
    const int nseg = (cend - a0 + 255) / 256;
    // Segments [1, jin1) lie wholly inside [cbeg, cend) (segment 0 starts at
    // a0 <= cbeg - (W-1), segment 1 at a0 + 256 > cbeg).
    const int jin1 = max(1, (cend - a0) / 256);
    uint4 *const ring_base = s_ring + tid;

    // Every segment streams in whole: the tokens of a vector outside the
    // chunk feed no stored output, except the W-1 before a sequence's first
    // chunk, which take the prior when segment 0 is read.  Only a vector
    // that crosses an end of the row is assembled with scalar loads.
    auto issue = [&](int seg) {
        if (seg >= nseg) return;
        const int t0 = a0 + seg * 256 + lane * 8;
        uint4 *slot = ring_base + (seg % kCfaSlots) * kCfaThreads;
        if (t0 >= 0 && t0 + 8 <= a.total) cp_async16(slot, xc + t0);
        else *slot = cfa_ragged_vector(xc, t0, a.total);
    };
    // Segments 0..kCfaSlots-2 form one commit group each, in order; segment
    // j goes to slot j % kCfaSlots.
#pragma unroll
    for (int j = 0; j < kCfaSlots - 1; ++j) {
        issue(j);
        cp_async_commit();
    }
    // The prior and the x entries of the new state load while the ring fills.
    uint32_t prior01 = 0, prior23 = 0;  // prior columns 0..3, packed
    uint16_t xnew = 0;                  // lane < W-1: x entry of new state column lane
    if (keep) {
        if (sc.init) {
            const uint16_t *sp = a.st + sc.line * a.ss_l + c * a.ss_d;
            uint32_t p[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < W - 1; ++j) p[j] = sp[j * a.ss_t];
            prior01 = p[0] | (p[1] << 16);
            prior23 = p[2] | (p[3] << 16);
        }
        const int idx = sc.len + lane;
        if (lane < W - 1 && idx >= W - 1) xnew = xc[sc.start + idx - (W - 1)];
    }

    uint32_t wt[W];  // tap k's bf16 weight in both halves
#pragma unroll
    for (int k = 0; k < W; ++k) wt[k] = 0x10001u * __ldg(a.w + c * a.ws_d + k * a.ws_k);
    const float bs = a.bias ? bf16_bits(__ldg(a.bias + c)) : 0.0f;
    uint32_t prev_z = 0, prev_w = 0;  // tokens before segment 0 are never needed
    uint16_t *const oc = a.out + c * a.os_d;

    auto window = [&](const uint4 &v, uint32_t (&E)[6]) {
        const uint32_t up_z = __shfl_up_sync(kFullMask, v.z, 1);
        const uint32_t up_w = __shfl_up_sync(kFullMask, v.w, 1);
        const uint32_t pv_z = __shfl_sync(kFullMask, prev_z, 31);
        const uint32_t pv_w = __shfl_sync(kFullMask, prev_w, 31);
        prev_z = v.z;
        prev_w = v.w;
        E[0] = lane ? up_z : pv_z;
        E[1] = lane ? up_w : pv_w;
        E[2] = v.x;
        E[3] = v.y;
        E[4] = v.z;
        E[5] = v.w;
    };
    auto step_checked = [&](int j) {
        cp_async_wait<kCfaSlots - 2>();
        uint4 v = ring_base[(j % kCfaSlots) * kCfaThreads];
        issue(j + kCfaSlots - 1);
        cp_async_commit();
        const int t0 = a0 + j * 256 + lane * 8;
        if (j == 0 && chunk0) v = cfa_with_prior<W>(v, t0, cbeg, prior01, prior23);
        uint32_t E[6];
        window(v, E);
        if (t0 + 8 <= cbeg || t0 >= cend) return;
        const uint4 o = cfa_outputs<W, SILU>(E, wt, bs);
        if (t0 >= cbeg && t0 + 8 <= cend) {
            cfa_store(oc + t0, o);
        } else {
            const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + i;
                if (t >= cbeg && t < cend)
                    oc[t] = uint16_t((i & 1) ? (ow[i >> 1] >> 16) : (ow[i >> 1] & 0xffffu));
            }
        }
    };

    step_checked(0);
    int j = 1;
    // Lean steps: this segment and the one streamed in lie inside [cbeg, cend).
    const uint16_t *nxt = xc + a0 + (j + kCfaSlots - 1) * 256 + lane * 8;
    uint16_t *dst = oc + a0 + j * 256 + lane * 8;
    // Groups of kCfaSlots lean steps starting at j = 1 (mod kCfaSlots):
    // segment j+u sits in slot (1+u) % kCfaSlots and the segment streamed
    // in goes to slot u, so every slot offset is a constant.  A step's
    // outputs are stored after the next step's wait, so its taps and SiLU
    // can overlap the next segment's shared-memory read.
    uint4 pend = make_uint4(0u, 0u, 0u, 0u);
    bool have = false;  // pend holds the outputs of segment j-1
    for (; j + 2 * kCfaSlots - 2 < jin1; j += kCfaSlots) {
#pragma unroll
        for (int u = 0; u < kCfaSlots; ++u) {
            cp_async_wait<kCfaSlots - 2>();
            const uint4 v = ring_base[((1 + u) % kCfaSlots) * kCfaThreads];
            cp_async16(ring_base + u * kCfaThreads, nxt + u * 256);
            cp_async_commit();
            if (u > 0 || have) cfa_store(dst + (u - 1) * 256, pend);
            uint32_t E[6];
            window(v, E);
            pend = cfa_outputs<W, SILU>(E, wt, bs);
        }
        have = true;
        nxt += kCfaSlots * 256;
        dst += kCfaSlots * 256;
    }
    if (have) cfa_store(dst - 256, pend);
    for (; j + kCfaSlots - 1 < jin1; ++j) {
        cp_async_wait<kCfaSlots - 2>();
        const uint4 v = ring_base[(j % kCfaSlots) * kCfaThreads];
        cp_async16(ring_base + ((j + kCfaSlots - 1) % kCfaSlots) * kCfaThreads, nxt);
        cp_async_commit();
        nxt += 256;
        uint32_t E[6];
        window(v, E);
        cfa_store(dst, cfa_outputs<W, SILU>(E, wt, bs));
        dst += 256;
    }
    // Interior segments whose streamed-in successor may cross the chunk's
    // edge: checked issue, lean compute and store.
    for (; j < jin1; ++j) {
        cp_async_wait<kCfaSlots - 2>();
        const uint4 v = ring_base[(j % kCfaSlots) * kCfaThreads];
        issue(j + kCfaSlots - 1);
        cp_async_commit();
        uint32_t E[6];
        window(v, E);
        cfa_store(dst, cfa_outputs<W, SILU>(E, wt, bs));
        dst += 256;
    }
    for (; j < nseg; ++j) step_checked(j);

    if (keep) {
        // New state = last W-1 entries of prior ++ x[sequence]; the prior was
        // read by every lane above, before any lane writes the line.
        uint16_t nb = xnew;
        const int idx = sc.len + lane;
        if (idx < W - 1) {
            const uint32_t src = idx < 2 ? prior01 : prior23;
            nb = uint16_t((idx & 1) ? (src >> 16) : (src & 0xffffu));
        }
        __syncwarp();
        if (lane < W - 1) a.st[sc.line * a.ss_l + c * a.ss_d + lane * a.ss_t] = nb;
    }
}

// ------------------------------- channel-first, cp.async, short chunks ----
//
// Sequences of a few thousand tokens give a warp of the kernel above one
// short row: a chunk search, a ring fill and a few segments, a few round
// trips for a few KB (64 sequences of 1024 tokens ran at half the copy
// rate).  Here a block takes ROWS channel rows of one chunk and each warp
// streams its ROWS / kCfaWarps rows (warp w: rows w, w + 8, ...) through
// one ring that runs on from one row into the next, so the ring stays full
// for the whole block.  The rows' weights, bias, prior and the x entries of
// their new state are staged in shared memory once, while the ring fills.
// Steps have the same arithmetic and edge handling as the kernel above; slot
// indices and row positions are counters rather than constants.

constexpr int kCfrRows = 64;        // channel rows per block
constexpr int kCfrRowsMid = 128;    // for sequences of about a thousand tokens
constexpr int kCfrRowsShort = 256;  // for sequences of a few hundred tokens
// Segments start on a 32-byte boundary (whole sectors), not 256 bytes as in
// the kernel above: a short row then wastes at most 15 tokens in front, and
// a sequence's first chunk starts at its first token, its prior coming from
// the window before segment 0 (1024-token sequences take 4 segments, not 5).
constexpr int kCfrAlign = 16;
static_assert(kCfaSlots == 8, "ring slot counters wrap with a mask");

template <int W, bool SILU, int CHUNK, int ROWS>
__global__ void __launch_bounds__(kCfaThreads, 4) fwd_cf_rows_kernel(const FwdArgs a) {
    constexpr int kRowsPerWarp = ROWS / kCfaWarps;
    extern __shared__ __align__(16) uint4 s_ring[];  // [kCfaSlots][kCfaThreads]
    __shared__ uint32_t s_w[ROWS * W];               // [row][tap], bf16 weight in both halves
    __shared__ float s_b[ROWS];
    __shared__ uint32_t s_p[ROWS * 2];               // prior columns 0..3, packed
    __shared__ uint32_t s_pre[ROWS * 2];             // the 4 tokens before segment 0, packed
    __shared__ uint16_t s_n[ROWS * 4];               // x entries of the new state
    wait_prior_grid();  // no early release: see the note on the streaming kernels' launches
    validate_sequence(a);
    SeqChunk sc;  // block-uniform: every warp finds the same chunk
    if (!locate_seq<kCfaPer>(a, CHUNK, blockIdx.x, sc)) return;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cbase = blockIdx.y * ROWS;
    const int cbeg = sc.start + sc.chunk * CHUNK;
    const int cend = sc.start + min(sc.len, (sc.chunk + 1) * CHUNK);
    const bool chunk0 = sc.chunk == 0;
    const bool keep = chunk0 && a.st != nullptr;
    // first token read: a first chunk takes its prior from the state, a
    // later chunk its W-1 halo tokens from x
    const int need0 = chunk0 ? cbeg : cbeg - (W - 1);
    // this warp's rows: cbase + warp + kCfaWarps * r, r < nr
    const int nr = max(0, min(kRowsPerWarp, (a.dim - cbase - warp + kCfaWarps - 1) / kCfaWarps));
    uint4 *const ring_base = s_ring + tid;

    // Channel row c's input row, first aligned token and segment count.
    auto geom_of = [&](int c, const uint16_t *&xc, int &a0, int &nseg) {
        xc = a.x + c * a.xs_d;
        const int phase = static_cast<int>((reinterpret_cast<uintptr_t>(xc) >> 1) & (kCfrAlign - 1));
        a0 = need0 - ((phase + need0) & (kCfrAlign - 1));
        nseg = (cend - a0 + 255) / 256;
    };
    // The same for this warp's row r.
    auto geom = [&](int r, const uint16_t *&xc, int &a0, int &nseg) {
        geom_of(cbase + warp + kCfaWarps * r, xc, a0, nseg);
    };
    // Issue side: the next (row, segment) to stream in and its slot.
    int ir = 0, ij = 0, islot = 0, i_a0 = 0, i_nseg = 0;
    const uint16_t *i_xc = a.x;
    if (nr > 0) geom(0, i_xc, i_a0, i_nseg);
    auto issue_next = [&]() {
        if (ir < nr) {
            const int t0 = i_a0 + ij * 256 + lane * 8;
            uint4 *slot = ring_base + islot * kCfaThreads;
            if (t0 >= 0 && t0 + 8 <= a.total) cp_async16(slot, i_xc + t0);
            else *slot = cfa_ragged_vector(i_xc, t0, a.total);
            if (++ij == i_nseg) {
                ij = 0;
                if (++ir < nr) geom(ir, i_xc, i_a0, i_nseg);
            }
        }
        islot = (islot + 1) & (kCfaSlots - 1);
        cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kCfaSlots - 1; ++j) issue_next();

    // Stage the block's row parameters: thread = (row, part tid % 4).
    for (int k = tid >> 2; k < ROWS; k += kCfaThreads / 4) {
        const int part = tid & 3;
        const int c = cbase + k;
        if (c < a.dim) {
            if (part == 0) {
#pragma unroll
                for (int t = 0; t < W; ++t) s_w[k * W + t] = 0x10001u * __ldg(a.w + c * a.ws_d + t * a.ws_k);
            } else if (part == 1) {
                s_b[k] = a.bias ? bf16_bits(__ldg(a.bias + c)) : 0.0f;
            } else if (part == 2) {
                uint32_t p[4] = {0, 0, 0, 0};
                if (keep && sc.init) {
                    const uint16_t *sp = a.st + sc.line * a.ss_l + c * a.ss_d;
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) p[j] = sp[j * a.ss_t];
                }
                const uint32_t p01 = p[0] | (p[1] << 16), p23 = p[2] | (p[3] << 16);
                s_p[2 * k] = p01;
                s_p[2 * k + 1] = p23;
                // The 4 tokens before segment 0: x before a later chunk's
                // halo (never needed), the prior's last columns before a
                // first chunk.
                uint4 before = make_uint4(0u, 0u, 0u, 0u);
                if (chunk0) {
                    const uint16_t *xr;
                    int a0, nseg;
                    geom_of(c, xr, a0, nseg);
                    before = cfa_with_prior<W>(before, a0 - 8, cbeg, p01, p23);
                }
                s_pre[2 * k] = before.z;
                s_pre[2 * k + 1] = before.w;
            } else if (keep) {
                const uint16_t *xr = a.x + c * a.xs_d;
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    const int idx = sc.len + j;
                    s_n[4 * k + j] = idx >= W - 1 ? xr[sc.start + idx - (W - 1)] : uint16_t(0);
                }
            }
        }
    }
    __syncthreads();

    uint32_t wt[W];
    float bs = 0.0f;
    uint32_t prior01 = 0, prior23 = 0;
    uint32_t prev_z = 0, prev_w = 0;
    auto window = [&](const uint4 &v, uint32_t (&E)[6]) {
        const uint32_t up_z = __shfl_up_sync(kFullMask, v.z, 1);
        const uint32_t up_w = __shfl_up_sync(kFullMask, v.w, 1);
        const uint32_t pv_z = __shfl_sync(kFullMask, prev_z, 31);
        const uint32_t pv_w = __shfl_sync(kFullMask, prev_w, 31);
        prev_z = v.z;
        prev_w = v.w;
        E[0] = lane ? up_z : pv_z;
        E[1] = lane ? up_w : pv_w;
        E[2] = v.x;
        E[3] = v.y;
        E[4] = v.z;
        E[5] = v.w;
    };

    int cr = 0, cj = 0, cslot = 0, c_a0 = 0, c_nseg = 0;
    const uint16_t *c_xc = a.x;
    uint16_t *oc = a.out;
    while (cr < nr) {
        cp_async_wait<kCfaSlots - 2>();
        uint4 v = ring_base[cslot * kCfaThreads];
        cslot = (cslot + 1) & (kCfaSlots - 1);
        issue_next();
        const int k = warp + kCfaWarps * cr;
        if (cj == 0) {  // a new row: its geometry and parameters
            geom(cr, c_xc, c_a0, c_nseg);
            oc = a.out + (cbase + k) * a.os_d;
#pragma unroll
            for (int t = 0; t < W; ++t) wt[t] = s_w[k * W + t];
            bs = s_b[k];
            prior01 = s_p[2 * k];
            prior23 = s_p[2 * k + 1];
            prev_z = s_pre[2 * k];
            prev_w = s_pre[2 * k + 1];
        }
        const int t0 = c_a0 + cj * 256 + lane * 8;
        if (cj == 0 && chunk0) v = cfa_with_prior<W>(v, t0, cbeg, prior01, prior23);
        uint32_t E[6];
        window(v, E);
        if (t0 + 8 > cbeg && t0 < cend) {
            const uint4 o = cfa_outputs<W, SILU>(E, wt, bs);
            if (t0 >= cbeg && t0 + 8 <= cend) {
                cfa_store(oc + t0, o);
            } else {
                const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = t0 + i;
                    if (t >= cbeg && t < cend)
                        oc[t] = uint16_t((i & 1) ? (ow[i >> 1] >> 16) : (ow[i >> 1] & 0xffffu));
                }
            }
        }
        if (++cj == c_nseg) {
            if (keep && lane < W - 1) {
                // New state = last W-1 entries of prior ++ x[sequence]; the
                // block read every prior before its barrier.
                const int idx = sc.len + lane;
                uint16_t nb = s_n[4 * k + lane];
                if (idx < W - 1) {
                    const uint32_t src = idx < 2 ? prior01 : prior23;
                    nb = uint16_t((idx & 1) ? (src >> 16) : (src & 0xffffu));
                }
                a.st[sc.line * a.ss_l + (cbase + k) * a.ss_d + lane * a.ss_t] = nb;
            }
            cj = 0;
            ++cr;
        }
    }
}

// ------------------------------------------------------ short problems ----
//
// A problem too small to fill the machine with streaming chunks is set by
// latency, not bandwidth: the dependent round trips before the first store
// (sequence search, state line, state columns, inputs) and the ring
// prologue.  These kernels cut that chain to two round trips for up to 32
// sequences.  A warp owns one short chunk of one sequence and one channel
// tile (channel-last) or channel row (channel-first); its lanes look up the
// chunk's sequence together with every candidate's end, state line and
// has_initial_state flag in one round trip, then load the chunk's inputs
// and the state columns straight into registers and compute.

constexpr int kShortThreads = 128;
constexpr int kShortWarps = kShortThreads / 32;
constexpr int kShortRun = 8;  // channel-last: tokens per warp (one run)
constexpr int kShortSegs = 5;  // channel-first: 256-token segments per warp
// channel-first chunk: a window of kShortSegs * 256 tokens that starts on the
// 16-byte boundary at or before the chunk's first token covers it
constexpr int kShortCfChunk = kShortSegs * 256 - 8;

// Channel-last: warp = (run of kShortRun tokens, 256-channel tile), lane =
// 8 channels; global warp g = slot * tiles + tile.  Every input row of the
// run goes to shared memory by asynchronous copies (no registers held while
// in flight, so a full grid fits the machine in one wave): slot rows
// [0, W-1) the inputs before the run, [W-1, W-1+n) the run, and for a
// sequence's first run [kShortRun+W-1, kShortRun+2W-2) the rows its new
// state takes from x.
constexpr int kShortClSlots = kShortRun + 2 * (kMaxWidth - 1);

template <int W, bool SILU>
__global__ void __launch_bounds__(kShortThreads, 7) fwd_cl_short_kernel(const FwdArgs a, int nslots) {
    __shared__ __align__(16) uint4 s_rows[kShortClSlots * kShortThreads];
    release_next_grid();
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const int ntiles = (a.dim + 255) / 256;
    const int g = blockIdx.x * kShortWarps + (threadIdx.x >> 5);
    const int tile = g % ntiles;
    const int slot = g / ntiles;
    if (slot >= nslots) return;  // warp-uniform
    validate_sequence_at(a, slot, tile == 0 && lane == 0);
    SeqChunk sc;
    if (!locate_short(a, kShortRun, slot, sc)) return;
    const int c0 = tile * 256 + lane * 8;
    if (c0 >= a.dim) return;

    const int64_t xs = a.xs_t;
    const uint16_t *xc = a.x + c0;
    uint4 *rows = s_rows + threadIdx.x;  // slot m at rows[m * kShortThreads]
    const int r0 = sc.start + sc.chunk * kShortRun;
    const int n = min(kShortRun, sc.len - sc.chunk * kShortRun);
    const bool first = sc.chunk == 0;
    const bool write_state = first && a.st != nullptr;
#pragma unroll
    for (int m = 0; m < kShortRun; ++m)
        if (m < n) cp_async16(rows + (W - 1 + m) * kShortThreads, xc + (r0 + m) * xs);
    if (!first) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
            cp_async16(rows + j * kShortThreads, xc + (r0 - (W - 1) + j) * xs);
    }
    if (write_state) {
        // New state = last W-1 entries of prior ++ x[sequence]; the entries
        // that come from x are copied in here.
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            const int idx = sc.len + j;
            if (idx >= W - 1)
                cp_async16(rows + (kShortRun + W - 1 + j) * kShortThreads,
                           xc + (sc.start + idx - (W - 1)) * xs);
        }
    }
    cp_async_commit();
    uint4 ring[W - 1];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
        ring[j] = make_uint4(0u, 0u, 0u, 0u);
        if (first && sc.init) ring[j] = load8_state(a, sc.line, c0, j);
    }
    uint4 wpk[W];
    const bool w_vec = a.ws_k == 1 && a.ws_d == W && (reinterpret_cast<uintptr_t>(a.w) & 15u) == 0;
    load_weights8<W>(a.w, a.ws_d, a.ws_k, c0, a.dim, w_vec, wpk);
    float bs[8];
    load_bias8(a.bias, c0, a.dim, (reinterpret_cast<uintptr_t>(a.bias) & 15u) == 0, bs);
    cp_async_wait<0>();

    uint4 nw[W - 1];
    if (write_state) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            const int idx = sc.len + j;
            if (idx < W - 1) {
#pragma unroll
                for (int q = 0; q < W - 1; ++q)
                    if (q == idx) nw[j] = ring[q];
            } else {
                nw[j] = rows[(kShortRun + W - 1 + j) * kShortThreads];
            }
        }
    }
    if (!first) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) ring[j] = rows[j * kShortThreads];
    }
    uint16_t *dst = a.out + c0 + static_cast<int64_t>(r0) * a.os_t;
#pragma unroll
    for (int m = 0; m < kShortRun; ++m) {
        if (m >= n) break;
        const uint4 v = rows[(W - 1 + m) * kShortThreads];
        __stcs(reinterpret_cast<uint4 *>(dst), ca_row<W, SILU>(wpk, bs, ring, v));
        dst += a.os_t;
#pragma unroll
        for (int k = 0; k < W - 2; ++k) ring[k] = ring[k + 1];
        ring[W - 2] = v;
    }
    if (write_state) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) store8_state(a, sc.line, c0, j, nw[j]);
    }
}

// The 8 inputs at tokens t0..t0+7 of a sequence's first chunk as its
// outputs see them: the prior (packed, oldest first) at the W-1 tokens
// before cbeg, `raw` (x as loaded) elsewhere.  Tokens further back feed no
// output of the chunk, nor do tokens at or past its end, so they keep
// whatever `raw` holds.  Only the one or two vectors that reach before cbeg
// get here, out of line.
template <int W>
__device__ __noinline__ uint4 short_prior_edge(uint4 raw, int t0, int cbeg, uint32_t prior01,
                                               uint32_t prior23) {
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = t0 + 2 * q + e - cbeg + (W - 1);  // prior column, if in [0, W-1)
            if (i >= 0 && i < W - 1) {
                const uint32_t src = i < 2 ? prior01 : prior23;
                const uint32_t val = (i & 1) ? (src >> 16) : (src & 0xffffu);
                w[q] = e ? ((w[q] & 0x0000ffffu) | (val << 16)) : ((w[q] & 0xffff0000u) | val);
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int W>
__device__ __forceinline__ uint4 short_prior(uint4 raw, int t0, int cbeg, uint32_t prior01,
                                             uint32_t prior23) {
    if (t0 >= cbeg || t0 + 8 <= cbeg - (W - 1)) return raw;
    return short_prior_edge<W>(raw, t0, cbeg, prior01, prior23);
}

// Tokens t0..t0+7 of a row that starts or ends inside them, element by
// element (0 outside [0, total)); out of line, like the edge masking.
__device__ __noinline__ uint4 short_load_edge(const uint16_t *xc, int t0, int total) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int t = t0 + 2 * q;
        const uint32_t lo = t >= 0 && t < total ? xc[t] : 0u;
        const uint32_t hi = t + 1 >= 0 && t + 1 < total ? xc[t + 1] : 0u;
        w[q] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Tokens t0..t0+7 of row xc as loaded: one 16-byte load when all lie inside
// [0, total) (t0 is on a 16-byte boundary), else element by element.
__device__ __forceinline__ uint4 short_load(const uint16_t *xc, int t0, int total) {
    if (t0 >= 0 && t0 + 8 <= total) return __ldg(reinterpret_cast<const uint4 *>(xc + t0));
    return short_load_edge(xc, t0, total);
}

// Channel-first: warp = (chunk of kShortCfChunk tokens, channel row), as
// kShortSegs segments of 256 tokens from the 16-byte boundary at or before
// the chunk's first token; lane l owns tokens 8l..8l+7 of each segment, and
// the W-1 tokens before them come from lane l-1 by shuffle (lane 0: lane 31
// of the segment before, or the vector before the window).
template <int W, bool SILU>
__global__ void __launch_bounds__(kShortThreads) fwd_cf_short_kernel(const FwdArgs a) {
    release_next_grid();
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const int slot = blockIdx.x;
    const int c = blockIdx.y * kShortWarps + (threadIdx.x >> 5);
    validate_sequence_at(a, slot, blockIdx.y == 0 && threadIdx.x == 0);
    if (c >= a.dim) return;  // warp-uniform
    SeqChunk sc;
    if (!locate_short(a, kShortCfChunk, slot, sc)) return;

    const uint16_t *const xc = a.x + c * a.xs_d;
    const int cbeg = sc.start + sc.chunk * kShortCfChunk;
    const int cend = sc.start + min(sc.len, (sc.chunk + 1) * kShortCfChunk);
    const bool chunk0 = sc.chunk == 0;
    const int phase = static_cast<int>((reinterpret_cast<uintptr_t>(xc) >> 1) & 7u);
    const int a0 = cbeg - ((phase + cbeg) & 7);  // on a 16-byte boundary, a0 > cbeg - 8
    // Every load goes out at once: the window's vectors, the vector before
    // it (lane 0), the state columns and the inputs the new state takes.
    uint4 raw[kShortSegs];
#pragma unroll
    for (int sg = 0; sg < kShortSegs; ++sg) {
        raw[sg] = make_uint4(0u, 0u, 0u, 0u);
        if (a0 + sg * 256 < cend) raw[sg] = short_load(xc, a0 + sg * 256 + lane * 8, a.total);  // warp-uniform
    }
    uint4 raw_before = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) raw_before = short_load(xc, a0 - 8, a.total);
    uint32_t p[4] = {0, 0, 0, 0};
    if (chunk0 && sc.init) {
        const uint16_t *sp = a.st + sc.line * a.ss_l + c * a.ss_d;
#pragma unroll
        for (int j = 0; j < W - 1; ++j) p[j] = sp[j * a.ss_t];
    }
    const bool write_state = chunk0 && a.st != nullptr;
    uint32_t from_x = 0;  // the new state's column `lane` when it comes from x
    const int idx = sc.len + lane;
    if (write_state && lane < W - 1 && idx >= W - 1) from_x = xc[sc.start + idx - (W - 1)];
    uint32_t wt[W];  // tap k's bf16 weight in both halves
#pragma unroll
    for (int k = 0; k < W; ++k) wt[k] = 0x10001u * __ldg(a.w + c * a.ws_d + k * a.ws_k);
    const float bs = a.bias ? bf16_bits(__ldg(a.bias + c)) : 0.0f;

    const uint32_t prior01 = p[0] | (p[1] << 16), prior23 = p[2] | (p[3] << 16);
    uint32_t prev_z = 0, prev_w = 0;  // lane 0: tokens a0-4 .. a0-1
    if (lane == 0) {
        const uint4 before = chunk0 ? short_prior<W>(raw_before, a0 - 8, cbeg, prior01, prior23) : raw_before;
        prev_z = before.z;
        prev_w = before.w;
    }
    uint16_t *const oc = a.out + c * a.os_d;
#pragma unroll
    for (int sg = 0; sg < kShortSegs; ++sg) {
        if (a0 + sg * 256 >= cend) break;  // warp-uniform: the chunk ends before this segment
        const int t0 = a0 + sg * 256 + lane * 8;
        const uint4 v = chunk0 && sg == 0 ? short_prior<W>(raw[sg], t0, cbeg, prior01, prior23) : raw[sg];
        const uint32_t up_z = __shfl_up_sync(kFullMask, v.z, 1);
        const uint32_t up_w = __shfl_up_sync(kFullMask, v.w, 1);
        const uint32_t pv_z = __shfl_sync(kFullMask, prev_z, sg == 0 ? 0 : 31);
        const uint32_t pv_w = __shfl_sync(kFullMask, prev_w, sg == 0 ? 0 : 31);
        prev_z = v.z;
        prev_w = v.w;
        const uint32_t E[6] = {lane ? up_z : pv_z, lane ? up_w : pv_w, v.x, v.y, v.z, v.w};
        if (t0 + 8 <= cbeg || t0 >= cend) continue;
        const uint4 o = cfa_outputs<W, SILU>(E, wt, bs);
        if (t0 >= cbeg && t0 + 8 <= cend) {
            __stcs(reinterpret_cast<uint4 *>(oc + t0), o);
        } else {
            const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + i;
                if (t >= cbeg && t < cend)
                    oc[t] = uint16_t((i & 1) ? (ow[i >> 1] >> 16) : (ow[i >> 1] & 0xffffu));
            }
        }
    }
    if (write_state) {
        // New state = last W-1 entries of prior ++ x[sequence]; every lane
        // read the prior above, before any lane writes the line.
        uint16_t nb = 0;
        if (lane < W - 1) {
            if (idx < W - 1) {
                const uint32_t src = idx < 2 ? prior01 : prior23;
                nb = uint16_t((idx & 1) ? (src >> 16) : (src & 0xffffu));
            } else {
                nb = uint16_t(from_x);
            }
        }
        __syncwarp();
        if (lane < W - 1) a.st[sc.line * a.ss_l + c * a.ss_d + lane * a.ss_t] = nb;
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

// Chunk length of the channel-first streaming kernel, from the sizes alone
// (the grid must not depend on query_start_loc): sequences of at most
// kCfaOneChunk tokens on average take one kCfaChunk-token chunk each, so few
// surplus slots remain; longer ones are cut into kCfaChunkSplit-token
// chunks, so no block streams a very long row.  The length is a template
// argument: as a runtime value the kernel measured 2.3 us slower.
constexpr int kCfaOneChunk = 16384;

bool cf_long_chunks(int total, int batch) {
    return (static_cast<int64_t>(total) + batch - 1) / batch <= kCfaOneChunk;
}


// Sequences of at most kCfrMaxAvg tokens on average go to the multi-row
// kernel, in chunks of kCfrChunk tokens, with more rows per block the
// shorter they are: a block's fixed cost (chunk search, ring fill, staging)
// then spreads over more data.  Measured at dim 8192, width 4 (us per call,
// 64 / 128 / 256 rows per block): 16 x 2048 tokens 172 / 178 / 210, 64 x 1024
// 369 / 359 / 373, 128 x 512 463 / 441 / 436, 256 x 256 665 / 613 / 593; the
// single-row kernel took 206, 607, 999 and 1870.  At 16 x 3072 the two
// kernels tie (248 and 251 us); at 16 x 4096 the single-row one wins (305
// against 334).
constexpr int kCfrMaxAvg = 3072;
constexpr int kCfrMidAvg = 1024;
constexpr int kCfrShortAvg = 512;
constexpr int kCfrChunk = kCfaChunkSplit;

int64_t average_length(int total, int batch) { return (static_cast<int64_t>(total) + batch - 1) / batch; }
bool cf_short_rows(int total, int batch) { return average_length(total, batch) <= kCfrMaxAvg; }

template <int W, bool SILU>
int launch_cl_async_w(const FwdArgs &a, cudaStream_t stream) {
    int dev = 0;
    current_device_sms(&dev);
    cudaError_t e;
    if (resident_blocks<fwd_cl_async_kernel<W, SILU>>(kCaThreads, kCaSmem, dev, &e) == 0)
        return static_cast<int>(e);
    const int64_t blocks = (static_cast<int64_t>(a.total) / kCaChunk + a.batch) *
                           ((a.dim + kCaTileC - 1) / kCaTileC);
    if (blocks > 0x7fffffff) return CCV_ERR_SIZE;
    return launch_pdl(fwd_cl_async_kernel<W, SILU>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kCaThreads), kCaSmem, stream, a);
}

template <int W, bool SILU, int CHUNK>
int launch_cf_async_chunk(const FwdArgs &a, cudaStream_t stream) {
    int dev = 0;
    current_device_sms(&dev);
    cudaError_t e;
    if (resident_blocks<fwd_cf_async_kernel<W, SILU, CHUNK>>(kCfaThreads, kCfaSmem, dev, &e) == 0)
        return static_cast<int>(e);
    const dim3 grid(static_cast<unsigned>(a.total / CHUNK + a.batch),
                    static_cast<unsigned>((a.dim + kCfaWarps - 1) / kCfaWarps));
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    return launch_pdl(fwd_cf_async_kernel<W, SILU, CHUNK>, grid, dim3(kCfaThreads), kCfaSmem, stream, a);
}

template <int W, bool SILU, int CHUNK, int ROWS>
int launch_cf_rows_chunk(const FwdArgs &a, cudaStream_t stream) {
    int dev = 0;
    current_device_sms(&dev);
    cudaError_t e;
    if (resident_blocks<fwd_cf_rows_kernel<W, SILU, CHUNK, ROWS>>(kCfaThreads, kCfaSmem, dev, &e) == 0)
        return static_cast<int>(e);
    const dim3 grid(static_cast<unsigned>(a.total / CHUNK + a.batch),
                    static_cast<unsigned>((a.dim + ROWS - 1) / ROWS));
    return launch_pdl(fwd_cf_rows_kernel<W, SILU, CHUNK, ROWS>, grid, dim3(kCfaThreads), kCfaSmem, stream,
                      a);
}

template <int W, bool SILU>
int launch_cf_async_w(const FwdArgs &a, cudaStream_t stream) {
    if (cf_short_rows(a.total, a.batch)) {
        const int64_t avg = average_length(a.total, a.batch);
        if (avg <= kCfrShortAvg) return launch_cf_rows_chunk<W, SILU, kCfrChunk, kCfrRowsShort>(a, stream);
        if (avg <= kCfrMidAvg) return launch_cf_rows_chunk<W, SILU, kCfrChunk, kCfrRowsMid>(a, stream);
        return launch_cf_rows_chunk<W, SILU, kCfrChunk, kCfrRows>(a, stream);
    }
    return cf_long_chunks(a.total, a.batch) ? launch_cf_async_chunk<W, SILU, kCfaChunk>(a, stream)
                                            : launch_cf_async_chunk<W, SILU, kCfaChunkSplit>(a, stream);
}

template <int W, bool SILU>
int launch_cl_short_w(const FwdArgs &a, cudaStream_t stream) {
    const int64_t nslots = static_cast<int64_t>(a.total) / kShortRun + a.batch;
    const int64_t warps = nslots * ((a.dim + 255) / 256);
    const int64_t blocks = (warps + kShortWarps - 1) / kShortWarps;
    if (nslots > 0x7fffffff || blocks > 0x7fffffff) return CCV_ERR_SIZE;
    return launch_pdl(fwd_cl_short_kernel<W, SILU>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kShortThreads), 0, stream, a, static_cast<int>(nslots));
}

template <int W, bool SILU>
int launch_cf_short_w(const FwdArgs &a, cudaStream_t stream) {
    const int64_t nslots = static_cast<int64_t>(a.total) / kShortCfChunk + a.batch;
    const dim3 grid(static_cast<unsigned>(nslots),
                    static_cast<unsigned>((a.dim + kShortWarps - 1) / kShortWarps));
    return launch_pdl(fwd_cf_short_kernel<W, SILU>, grid, dim3(kShortThreads), 0, stream, a);
}

int launch_cl_short(const FwdArgs &a, int width, bool silu, cudaStream_t stream) {
    switch (width) {
        case 2: return silu ? launch_cl_short_w<2, true>(a, stream) : launch_cl_short_w<2, false>(a, stream);
        case 3: return silu ? launch_cl_short_w<3, true>(a, stream) : launch_cl_short_w<3, false>(a, stream);
        case 4: return silu ? launch_cl_short_w<4, true>(a, stream) : launch_cl_short_w<4, false>(a, stream);
        case 5: return silu ? launch_cl_short_w<5, true>(a, stream) : launch_cl_short_w<5, false>(a, stream);
    }
    return CCV_ERR_WIDTH;
}

int launch_cf_short(const FwdArgs &a, int width, bool silu, cudaStream_t stream) {
    switch (width) {
        case 2: return silu ? launch_cf_short_w<2, true>(a, stream) : launch_cf_short_w<2, false>(a, stream);
        case 3: return silu ? launch_cf_short_w<3, true>(a, stream) : launch_cf_short_w<3, false>(a, stream);
        case 4: return silu ? launch_cf_short_w<4, true>(a, stream) : launch_cf_short_w<4, false>(a, stream);
        case 5: return silu ? launch_cf_short_w<5, true>(a, stream) : launch_cf_short_w<5, false>(a, stream);
    }
    return CCV_ERR_WIDTH;
}

// Which prefill kernels serve a problem of `elems` = total_tokens * dim
// elements: the short kernels up to kShortMaxElems, the streaming kernels
// above.  The environment variable CCV_PREFILL_PATH=short or =stream forces
// one family (both compute the same results; for tests and tuning).
constexpr int64_t kShortMaxElems = int64_t(1) << 23;

bool use_short_path(int64_t elems) {
    const char *force = std::getenv("CCV_PREFILL_PATH");
    if (force != nullptr && std::strcmp(force, "short") == 0) return true;
    if (force != nullptr && std::strcmp(force, "stream") == 0) return false;
    return elems <= kShortMaxElems;
}

int launch_cl_async(const FwdArgs &a, int width, bool silu, cudaStream_t stream) {
    switch (width) {
        case 2: return silu ? launch_cl_async_w<2, true>(a, stream) : launch_cl_async_w<2, false>(a, stream);
        case 3: return silu ? launch_cl_async_w<3, true>(a, stream) : launch_cl_async_w<3, false>(a, stream);
        case 4: return silu ? launch_cl_async_w<4, true>(a, stream) : launch_cl_async_w<4, false>(a, stream);
        case 5: return silu ? launch_cl_async_w<5, true>(a, stream) : launch_cl_async_w<5, false>(a, stream);
    }
    return CCV_ERR_WIDTH;
}

int launch_cf_async(const FwdArgs &a, int width, bool silu, cudaStream_t stream) {
    switch (width) {
        case 2: return silu ? launch_cf_async_w<2, true>(a, stream) : launch_cf_async_w<2, false>(a, stream);
        case 3: return silu ? launch_cf_async_w<3, true>(a, stream) : launch_cf_async_w<3, false>(a, stream);
        case 4: return silu ? launch_cf_async_w<4, true>(a, stream) : launch_cf_async_w<4, false>(a, stream);
        case 5: return silu ? launch_cf_async_w<5, true>(a, stream) : launch_cf_async_w<5, false>(a, stream);
    }
    return CCV_ERR_WIDTH;
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
        // With a single token the token strides are never used.
        const bool tok_ok = total_tokens <= 1 || (x_stride_tok % 8 == 0 && out_stride_tok % 8 == 0);
        const bool vec = dim % 8 == 0 && aligned16(x) && aligned16(out) && tok_ok;
        a.st_vec = vec && conv_states != nullptr && s_stride_dim == 1 && aligned16(conv_states) &&
                   s_stride_line % 8 == 0 && s_stride_tok % 8 == 0;
        if (vec) {
            return use_short_path(static_cast<int64_t>(total_tokens) * dim)
                       ? launch_cl_short(a, width, is_silu, stream)
                       : launch_cl_async(a, width, is_silu, stream);
        }
        fn = pick_kernel<1, true>(width, is_silu);
        grid = dim3(static_cast<unsigned>(total_tokens / kClChunk + batch),
                    static_cast<unsigned>((dim + 31) / 32));
    } else if (x_stride_tok == 1 && out_stride_tok == 1) {
        const uintptr_t xo = (reinterpret_cast<uintptr_t>(x) >> 1) & 7u;
        const uintptr_t oo = (reinterpret_cast<uintptr_t>(out) >> 1) & 7u;
        const bool same_phase = (reinterpret_cast<uintptr_t>(x) & 1u) == 0 &&
                                (reinterpret_cast<uintptr_t>(out) & 1u) == 0 && xo == oo &&
                                (x_stride_dim - out_stride_dim) % 8 == 0;
        if (same_phase) {
            const bool fits = (dim + kShortWarps - 1) / kShortWarps <= 65535;
            return fits && use_short_path(static_cast<int64_t>(total_tokens) * dim)
                       ? launch_cf_short(a, width, is_silu, stream)
                       : launch_cf_async(a, width, is_silu, stream);
        }
        fn = pick_kernel<1, false>(width, is_silu);
        grid = dim3(static_cast<unsigned>(total_tokens / (kCfSegs * 32) + batch),
                    static_cast<unsigned>((dim + kWarps - 1) / kWarps));
    } else {
        fn = pick_kernel<1, true>(width, is_silu);
        grid = dim3(static_cast<unsigned>(total_tokens / kClChunk + batch),
                    static_cast<unsigned>((dim + 31) / 32));
    }
    if (grid.y > 65535u) return CCV_ERR_SIZE;
    return launch_pdl(fn, grid, dim3(kThreads), 0, stream, a);
}
