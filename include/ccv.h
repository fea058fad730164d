/*
 * ccv.h -- C ABI of the GB300 (sm_103a) causal depthwise conv1d forward
 * library, libccv.so.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *   allocates no memory, never synchronises the device or the stream, and
 *   only enqueues kernels on `stream`, so each call can be captured into a
 *   CUDA graph.  Launch grids depend only on the integer size arguments,
 *   never on device-resident data.
 * - bf16 tensors are passed as `const void*` / `void*` pointing at IEEE
 *   bfloat16 values.  Index tensors are int32 except positions and slot
 *   mappings (int64).  Strides are in ELEMENTS and must be >= 0
 *   (CCV_ERR_STRIDE otherwise); an output's strides must map distinct
 *   elements to distinct addresses.  The fast kernels are picked when the
 *   innermost stride is 1 and the pointers/strides are 16-byte aligned; a
 *   generic strided kernel handles everything else with the same results.
 * - Return value: 0 (CCV_OK) on success; a negative ccv_status for an
 *   argument error detected on the host (nothing is launched); a positive
 *   value is the cudaError_t of a failed launch.
 * - Size 0 work (no tokens, no rows) returns CCV_OK without launching.
 * - Kernels are launched with programmatic stream serialization: a kernel's
 *   blocks may be scheduled while the previous kernel on the stream is still
 *   finishing, but each waits for that kernel to complete before it reads or
 *   writes any memory, so stream order holds exactly as for plain launches
 *   (and under CUDA-graph capture).
 * - `err_count` (nullable) is a device int the kernels atomically increment
 *   when they skip data-dependent invalid indices (a query_start_loc that
 *   decreases or leaves [0, total_tokens], a state line outside
 *   [0, num_cache_lines) that is not the pad id, a block id outside the
 *   cache, ...).  Only zero vs non-zero is meaningful.  Kernels never trap.
 *
 * Sources: the semantics are those of three pages -- tokenspeed
 * "causal_conv1d.py" (`causal_conv1d_fn`, `causal_conv1d_update`), vLLM
 * Inkling "sconv.py" (`fused_sconv`, `sconv_seq_metadata`) and atrex-bench
 * operator #003 "causal_conv1d" (reference formulation).
 */
#ifndef CCV_H_
#define CCV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ccv_stream_t; /* same type as cudaStream_t */

enum ccv_status {
    CCV_OK = 0,
    CCV_ERR_NULL_POINTER = -1,  /* a required pointer is NULL */
    CCV_ERR_WIDTH = -2,         /* width outside 2..5 */
    CCV_ERR_SIZE = -3,          /* a negative or inconsistent size */
    CCV_ERR_STATE_LEN = -4,     /* state storage narrower than the method needs */
    CCV_ERR_ALIAS = -5,         /* out overlaps x where that is not allowed */
    CCV_ERR_STRIDE = -6,        /* a stride the method requires to be 1 is not */
    CCV_ERR_RANGE = -7,         /* stream D-range outside the cache or overlapping another */
    CCV_ERR_CAPACITY = -8,      /* an output buffer has fewer entries than needed */
    CCV_ERR_ARGUMENT = -9       /* an argument combination the pages reject */
};

/* Human-readable name of a status code (static storage, never NULL). */
const char *ccv_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int ccv_version(void);

/*
 * ccv_fwd -- varlen causal depthwise conv1d prefill with conv_state
 * (continuous batching).  tokenspeed causal_conv1d.py, `causal_conv1d_fn`
 * and `_causal_conv1d_fwd_kernel`; reference formulation atrex-bench #003.
 *
 * x, out        logical (dim, total_tokens); element (c, t) at
 *               x[c*x_stride_dim + t*x_stride_tok].  Both channel-last
 *               (x_stride_dim == 1) and channel-first (x_stride_tok == 1)
 *               layouts are fast.  out must not overlap x (chunks read
 *               their neighbours' inputs as halo).
 * weight        (dim, width); bias (dim) or NULL.
 * conv_states   pool (num_cache_lines, dim, state_len >= width-1), column 0
 *               the oldest; NULL means a zero prior and no write-back.
 *               Updated in place: columns [0, width-1) of each processed
 *               sequence's line receive the sequence's last width-1 inputs
 *               (for a sequence shorter than width-1 the old columns shift
 *               left).  Columns >= width-1 are never touched.
 * query_start_loc  int32 [batch+1], cumulative token offsets with a leading
 *               0; sequence i owns tokens [qsl[i], qsl[i+1]).  Tokens past
 *               qsl[batch] are not processed.
 * cache_indices int32 [batch] or NULL (line i for sequence i).  An entry equal
 *               to pad_slot_id skips the sequence: its out tokens and every
 *               state line stay untouched.
 * has_initial_state  uint8/bool [batch] or NULL (all false).  When false the
 *               prior is zeros; the state is written back either way.
 *               Requires conv_states.
 * A zero-length sequence writes nothing.  silu != 0 applies v/(1+exp(-v)).
 * Two non-pad sequences that share a state line race (undefined result).
 * Problems of up to 2^23 elements (total_tokens * dim) run on kernels built
 * for latency, larger ones on streaming kernels; both compute the same
 * results.  In the channel-first layout the streaming family has a kernel
 * for sequences of a few thousand tokens or fewer on average (several
 * channel rows per warp) and one for longer ones.  Every choice and every
 * grid follows from the sizes (total_tokens, batch, dim, width), the strides
 * and the buffers' alignment, never from query_start_loc, so a captured
 * graph stays valid for any offsets of the same sizes.  The environment variable CCV_PREFILL_PATH=short or =stream,
 * read at each call, forces one family (for testing and tuning).
 */
int ccv_fwd(const void *x, int64_t x_stride_dim, int64_t x_stride_tok,
            void *out, int64_t out_stride_dim, int64_t out_stride_tok,
            const void *weight, int64_t w_stride_dim, int64_t w_stride_w,
            const void *bias,
            void *conv_states, int64_t s_stride_line, int64_t s_stride_dim,
            int64_t s_stride_tok, int num_cache_lines, int state_len,
            const int32_t *query_start_loc, int batch,
            const int32_t *cache_indices, const uint8_t *has_initial_state,
            int dim, int total_tokens, int width, int pad_slot_id, int silu,
            int *err_count, ccv_stream_t stream);

/*
 * ccv_update -- decode step: causal conv over `seqlen` new tokens per row
 * with the row's conv_state as the window prefix, state shifted in place.
 * tokenspeed causal_conv1d.py, `causal_conv1d_update` and
 * `_causal_conv1d_update_kernel` (non-speculative path; ccv_update_spec
 * below adds the speculative-decoding extras).
 *
 * x, out        (batch, dim, seqlen) with strides (b, d, t); out may be
 *               exactly x (same pointer and strides: in-place, as the page's
 *               wrapper does) or must not overlap it.
 * conv_state    pool (num_cache_lines, dim, state_len); row b uses line
 *               conv_state_indices[b] (or b when NULL); a line equal to
 *               pad_slot_id skips the row (out and state untouched).
 *               out[b,c,t] = act(bias[c] + sum_k w[c,k] * u[t+k]) with
 *               u = state[line,c,0..width-2] ++ x[b,c,0..seqlen-1]; then
 *               state[line,c,j] = u[1+j] for j < width-2+seqlen, so
 *               state_len >= width-2+seqlen is required (CCV_ERR_STATE_LEN).
 */
int ccv_update(const void *x, int64_t x_stride_b, int64_t x_stride_dim, int64_t x_stride_tok,
               void *out, int64_t out_stride_b, int64_t out_stride_dim, int64_t out_stride_tok,
               const void *weight, int64_t w_stride_dim, int64_t w_stride_w,
               const void *bias,
               void *conv_state, int64_t s_stride_line, int64_t s_stride_dim,
               int64_t s_stride_tok, int num_cache_lines, int state_len,
               const int32_t *conv_state_indices, int batch, int dim, int seqlen,
               int width, int pad_slot_id, int silu, int *err_count,
               ccv_stream_t stream);

/*
 * ccv_update_spec -- ccv_update with the speculative-decoding extras of
 * tokenspeed causal_conv1d.py, `causal_conv1d_update` (num_accepted_tokens,
 * intermediate_conv_window, output_state_indices).  Every argument shared
 * with ccv_update means the same.
 *
 * num_accepted_tokens  int32 [batch] or NULL.  Row b reads its window from
 *               state columns off .. off+width-2, off = num_accepted_tokens[b]
 *               - 1 (0 when NULL): after a verify step that kept k drafts the
 *               state holds [history.., drafts..] and the window starts k-1
 *               columns in.  A row with off < 0 or off+width-1 > state_len is
 *               skipped and counted in err_count.
 * intermediate_conv_window  bf16 or NULL, element (b, step, c, j) at
 *               b*i_stride_b + step*i_stride_step + c*i_stride_dim +
 *               j*i_stride_win, inter_steps >= seqlen steps: after token t
 *               it receives the window u[t+1 .. t+width-1] (the last width-1
 *               inputs), indexed by batch position, not by state line.  Must
 *               not overlap x, out or conv_state.
 * output_state_indices  int32 or NULL, element (b, step) at b*oi_stride_b +
 *               step*oi_stride_step, oidx_steps >= seqlen: when the entry for
 *               (b, t) is >= 0 the same window is written to columns
 *               0..width-2 of that state line (a line outside the pool is
 *               counted and skipped).  Output lines must not be lines that
 *               other rows of the same call read (they would race).
 * When either buffer is given the state line is NOT shifted in place and
 * state_len >= width-1 suffices; otherwise the line is shifted exactly as
 * in ccv_update (state_len >= width-2+seqlen).  inter_steps or oidx_steps
 * below seqlen gives CCV_ERR_CAPACITY.
 */
int ccv_update_spec(const void *x, int64_t x_stride_b, int64_t x_stride_dim, int64_t x_stride_tok,
                    void *out, int64_t out_stride_b, int64_t out_stride_dim,
                    int64_t out_stride_tok, const void *weight, int64_t w_stride_dim,
                    int64_t w_stride_w, const void *bias,
                    void *conv_state, int64_t s_stride_line, int64_t s_stride_dim,
                    int64_t s_stride_tok, int num_cache_lines, int state_len,
                    const int32_t *conv_state_indices, const int32_t *num_accepted_tokens,
                    void *intermediate_conv_window, int64_t i_stride_b, int64_t i_stride_step,
                    int64_t i_stride_dim, int64_t i_stride_win, int inter_steps,
                    const int32_t *output_state_indices, int64_t oi_stride_b,
                    int64_t oi_stride_step, int oidx_steps,
                    int batch, int dim, int seqlen, int width, int pad_slot_id, int silu,
                    int *err_count, ccv_stream_t stream);

/*
 * paged_sconv_seq_metadata -- per-token request id and first x-row.
 * vLLM Inkling sconv.py, `sconv_seq_metadata` / `_seq_metadata_kernel`.
 *
 * query_start_loc  int32, at least num_reqs entries (only [0, num_reqs) are
 *               read).
 * For t < num_actual_tokens: seq_idx_out[t] = the largest j in [0, num_reqs)
 * with query_start_loc[j] <= t (0 if none), query_start_out[t] =
 * query_start_loc[seq_idx_out[t]].  Rows num_actual_tokens <= t <
 * num_padded_tokens get 0 in both (they must carry slot -1).  Rows past
 * num_padded_tokens are not written.  Errors: num_padded_tokens <
 * num_actual_tokens (CCV_ERR_SIZE); out_capacity < num_padded_tokens
 * (CCV_ERR_CAPACITY).
 */
int paged_sconv_seq_metadata(const int32_t *query_start_loc, int num_reqs,
                             int num_actual_tokens, int num_padded_tokens,
                             int32_t *seq_idx_out, int32_t *query_start_out,
                             int out_capacity, ccv_stream_t stream);

/*
 * paged_sconv_fwd -- single-launch insert + depthwise causal conv over a
 * paged sliding-window cache.  vLLM Inkling sconv.py, `fused_sconv` and
 * `_fused_sconv_kernel`.
 *
 * x             [T, C] bf16, C = H*ws channels head-major, channel stride 1,
 *               row stride x_stride_t; also the residual.
 * cache         [num_blocks, H, N, D] bf16, D stride 1; the stream occupies
 *               D-range [off_s, off_s+ws) (CCV_ERR_RANGE otherwise).
 * weight        [C, width]; no bias.
 * out           [T, C], channel stride 1, row stride out_stride_t; must not
 *               overlap x or the cache.
 * positions     int64 [T] absolute position per token.
 * seq_idx, query_start  int32 [T] (from paged_sconv_seq_metadata).
 * slot_mapping  int64 [T]: flat slot block*N + offset; < 0 marks a PAD row.
 * block_table   int32 [bt_rows, max_blocks], row stride bt_stride_r.
 * For each token t and tap iw = 0..width-1: src = pos[t]-(width-1)+iw,
 * row = t-(width-1)+iw; the tap is 0 for PAD rows or src < 0, x[row] when
 * row >= query_start[t] (in this forward), else the cache entry at
 * block_table[seq_idx[t], min(src/N, max_blocks-1)], offset src%N.
 * out = act(sum of taps * w) (+ x[t] when residual).  Every real token's x
 * is also written to its slot.  The caller guarantees that no slot written
 * by this call is read as a pre-forward tap in the same call (the pages'
 * race-freedom condition); then one launch is race-free and deterministic.
 */
int paged_sconv_fwd(const void *x, int64_t x_stride_t,
                    void *cache, int64_t c_stride_blk, int64_t c_stride_h,
                    int64_t c_stride_n, int num_blocks, int H, int N, int D,
                    const void *weight, int64_t w_stride_c, int64_t w_stride_w,
                    void *out, int64_t out_stride_t,
                    const int64_t *positions, const int32_t *seq_idx,
                    const int64_t *slot_mapping, const int32_t *block_table,
                    int64_t bt_stride_r, int bt_rows, int max_blocks,
                    const int32_t *query_start, int T, int off_s, int ws,
                    int width, int silu, int residual, int *err_count,
                    ccv_stream_t stream);

/*
 * paged_sconv_fwd_with_metadata -- paged_sconv_fwd in one launch, with the
 * token metadata resolved inside it.  vLLM Inkling sconv.py,
 * `sconv_seq_metadata` / `_seq_metadata_kernel` and `fused_sconv` /
 * `_fused_sconv_kernel`: each token's request and first x-row are computed
 * from query_start_loc exactly as paged_sconv_seq_metadata computes them,
 * then the insert and conv run as in paged_sconv_fwd.
 *
 * query_start_loc, num_reqs, num_actual_tokens  as for
 *               paged_sconv_seq_metadata, with T the padded token count:
 *               num_actual_tokens <= T, and num_reqs == 0 only with no real
 *               token (CCV_ERR_SIZE otherwise).
 * seq_idx_out, query_start_out  int32 [T] each, or NULL: when given they
 *               receive the metadata (the same values paged_sconv_seq_metadata
 *               writes), so that later calls of the same forward -- other
 *               layers, other streams -- can pass them to paged_sconv_fwd.
 *               They must not overlap any other argument.
 * Every other argument means what it means for paged_sconv_fwd.  out, the
 * cache and err_count end up as after paged_sconv_seq_metadata followed by
 * paged_sconv_fwd.
 */
int paged_sconv_fwd_with_metadata(const void *x, int64_t x_stride_t,
                                  void *cache, int64_t c_stride_blk, int64_t c_stride_h,
                                  int64_t c_stride_n, int num_blocks, int H, int N, int D,
                                  const void *weight, int64_t w_stride_c, int64_t w_stride_w,
                                  void *out, int64_t out_stride_t,
                                  const int64_t *positions, const int32_t *query_start_loc,
                                  int num_reqs, int num_actual_tokens,
                                  int32_t *seq_idx_out, int32_t *query_start_out,
                                  const int64_t *slot_mapping, const int32_t *block_table,
                                  int64_t bt_stride_r, int bt_rows, int max_blocks,
                                  int T, int off_s, int ws, int width, int silu, int residual,
                                  int *err_count, ccv_stream_t stream);

/*
 * One conv stream of a layer for paged_sconv_fwd_streams: its input, its
 * weights, its output and the D-range [off_s, off_s + ws) of the shared
 * cache it owns.  Fields mean what the same-named arguments of
 * paged_sconv_fwd mean.
 */
typedef struct ccv_paged_stream {
    const void *x;
    int64_t x_stride_t;
    const void *weight;
    int64_t w_stride_c;
    int64_t w_stride_w;
    void *out;
    int64_t out_stride_t;
    int off_s;
    int ws;
} ccv_paged_stream;

/*
 * paged_sconv_fwd_streams -- paged_sconv_fwd for up to 8 conv streams of one
 * layer in a single launch.  vLLM Inkling sconv.py, module docstring: a
 * layer's streams (K, V, attn-output, mlp-output) share one paged cache,
 * each in its own D-sub-range, and each is one `fused_sconv` call; the
 * result equals calling paged_sconv_fwd once per stream, in any order.
 *
 * streams       HOST array of num_streams (1..8) descriptors, read during the
 *               call only.  The streams' D-ranges must be pairwise disjoint
 *               (CCV_ERR_RANGE otherwise); no out may overlap any x, another
 *               out or the cache (CCV_ERR_ALIAS).
 * Every other argument is shared by all streams and means what it means for
 * paged_sconv_fwd (silu and residual apply to every stream).  When every
 * stream allows 16-byte vectors one grid covers them all; otherwise each
 * stream is launched on its own, in order, with the same results.
 */
int paged_sconv_fwd_streams(const ccv_paged_stream *streams, int num_streams,
                            void *cache, int64_t c_stride_blk, int64_t c_stride_h,
                            int64_t c_stride_n, int num_blocks, int H, int N, int D,
                            const int64_t *positions, const int32_t *seq_idx,
                            const int64_t *slot_mapping, const int32_t *block_table,
                            int64_t bt_stride_r, int bt_rows, int max_blocks,
                            const int32_t *query_start, int T, int width, int silu,
                            int residual, int *err_count, ccv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CCV_H_ */
