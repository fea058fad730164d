/*
 * ccv_oracle.c -- plain, slow CPU oracle for the causal depthwise conv1d
 * forward family.  TEST INFRASTRUCTURE ONLY: the library's product path never
 * links, loads or calls this file.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may use it.
 *
 * Every routine is a scalar loop over (sequence, channel, token, tap) written
 * from the definitions on these pages:
 *   [P1] tokenspeed "causal_conv1d.py" (linear-attention layers): the varlen
 *        prefill kernel `_causal_conv1d_fwd_kernel` / wrapper `causal_conv1d_fn`
 *        and the decode kernel `_causal_conv1d_update_kernel` / wrapper
 *        `causal_conv1d_update`.
 *   [P2] vLLM Inkling "sconv.py": `_fused_sconv_kernel` / `fused_sconv` (paged
 *        sliding-window short conv) and `_seq_metadata_kernel` /
 *        `sconv_seq_metadata`.
 *   [P3] atrex-bench operator #003 "causal_conv1d": the reference formulation
 *        `Model.forward` (concatenate the state, grouped conv1d, keep the last
 *        T outputs, SiLU).
 *
 * Arithmetic.  Storage is bf16 (passed as raw uint16 bit patterns).  The pages
 * accumulate in fp32 ([P1] `acc_preload ... .to(tl.float32)`, [P2]
 * `acc = tl.zeros(..., tl.float32)`), so the oracle does too:
 *   acc = bias; for k = 0..W-1: acc = acc + w[k] * u[k]      (fp32, this order)
 * A bf16 x bf16 product is exact in fp32, so only the additions round.  The
 * file must be compiled with -ffp-contract=off so no compiler turns the
 * separate multiply and add into an fma.  SiLU v/(1+exp(-v)) ([P1] token loop;
 * [P2] uses v*sigmoid(v), the same function) is evaluated in double from the
 * fp32 value and rounded back to fp32.  The final value is rounded once to
 * bf16 with round-to-nearest-even.
 *
 * This file shares no code with the CUDA library.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 is the upper half of an IEEE-754 binary32, so widening is a shift. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even.  NaN stays NaN (quiet
 * bit forced so a payload in the dropped half cannot turn it into inf). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

static float silu_f32(float v) {
    double d = (double)v;
    return (float)(d / (1.0 + exp(-d)));
}

/* Exported so a test can pin the rounding rule against an independent
 * implementation (torch's float -> bfloat16 cast). */
void oracle_f32_to_bf16(const float *src, uint16_t *dst, int64_t n) {
    for (int64_t i = 0; i < n; i++) dst[i] = f32_to_bf16(src[i]);
}

void oracle_silu_f32(const float *src, float *dst, int64_t n) {
    for (int64_t i = 0; i < n; i++) dst[i] = silu_f32(src[i]);
}

static void count_error(int *err_count) {
    if (err_count) (*err_count)++;
}

/* ------------------------------------------------------- varlen prefill ---- */

/*
 * oracle_ccv_fwd -- [P1] `causal_conv1d_fn` / `_causal_conv1d_fwd_kernel`.
 *
 * x and out are logically (dim, total_tokens); element (c, t) sits at
 * x[c*xs_dim + t*xs_tok].  Sequence i owns tokens [qsl[i], qsl[i+1]) ([P1]
 * docstring: query_start_loc is the cumulative length with a leading 0).
 * Its state line is cache_indices[i] (or i when cache_indices is NULL); a
 * line equal to pad_slot_id means the sequence is not processed at all
 * ([P1] docstring, "cache_indices = [pad_slot_id, 1, 20, pad_slot_id]").
 *
 * For channel c of a processed sequence of length L >= 1:
 *   prior[j]  = conv_states[line, c, j] if has_initial_state[i] else 0,
 *               j = 0..W-2  (column 0 is the oldest; [P1] chunk-0 state read)
 *   u         = prior ++ x[c, qsl[i] .. qsl[i+1]-1]           (length W-1+L)
 *   out[c, qsl[i]+t] = act(bias[c] + sum_k w[c,k] * u[t+k]),  t = 0..L-1
 *   conv_states[line, c, j] = u[L+j],  j = 0..W-2              ([P1] state
 *               update: the last W-1 inputs, shifting the old state left
 *               when L < W-1)
 * A zero-length sequence launches no program in [P1], so it leaves both out
 * and its state line untouched.  conv_states == NULL means a zero prior and
 * no write-back.  Columns >= W-1 of a wider state line are not touched.
 *
 * Data-dependent invalid input (decreasing or out-of-range query_start_loc,
 * a state line outside [0, num_cache_lines)) skips the sequence and bumps
 * *err_count.  Returns 0.
 */
int oracle_ccv_fwd(const uint16_t *x, int64_t xs_dim, int64_t xs_tok,
                   uint16_t *out, int64_t os_dim, int64_t os_tok,
                   const uint16_t *weight, int64_t ws_dim, int64_t ws_w,
                   const uint16_t *bias,
                   uint16_t *conv_states, int64_t ss_line, int64_t ss_dim, int64_t ss_tok,
                   int num_cache_lines,
                   const int32_t *query_start_loc, int batch,
                   const int32_t *cache_indices, const uint8_t *has_initial_state,
                   int dim, int total_tokens, int width, int pad_slot_id, int silu,
                   int *err_count) {
    const int W = width;
    for (int i = 0; i < batch; i++) {
        int line = cache_indices ? cache_indices[i] : i;
        if (line == pad_slot_id) continue;
        int start = query_start_loc[i];
        int end = query_start_loc[i + 1];
        if (start < 0 || end < start || end > total_tokens) {
            count_error(err_count);
            continue;
        }
        int L = end - start;
        if (L == 0) continue;
        if (conv_states && (line < 0 || line >= num_cache_lines)) {
            count_error(err_count);
            continue;
        }
        int use_prior = conv_states && has_initial_state && has_initial_state[i];

        uint16_t *u_bits = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(W - 1 + L));
        for (int c = 0; c < dim; c++) {
            for (int j = 0; j < W - 1; j++)
                u_bits[j] = use_prior
                    ? conv_states[line * ss_line + c * ss_dim + j * ss_tok]
                    : (uint16_t)0;
            for (int t = 0; t < L; t++)
                u_bits[W - 1 + t] = x[c * xs_dim + (int64_t)(start + t) * xs_tok];

            float b = bias ? bf16_to_f32(bias[c]) : 0.0f;
            for (int t = 0; t < L; t++) {
                float acc = b;
                for (int k = 0; k < W; k++)
                    acc = acc + bf16_to_f32(weight[c * ws_dim + k * ws_w]) *
                                    bf16_to_f32(u_bits[t + k]);
                if (silu) acc = silu_f32(acc);
                out[c * os_dim + (int64_t)(start + t) * os_tok] = f32_to_bf16(acc);
            }
            if (conv_states)
                for (int j = 0; j < W - 1; j++)
                    conv_states[line * ss_line + c * ss_dim + j * ss_tok] = u_bits[L + j];
        }
        free(u_bits);
    }
    return 0;
}

/* ------------------------------------------------------------- decode ---- */

/*
 * oracle_ccv_update -- [P1] `causal_conv1d_update` / `_causal_conv1d_update_kernel`
 * without the speculative-decoding extras.
 *
 * x and out are (batch, dim, seqlen); out may be the very same buffer as x
 * ([P1] wrapper: out = x).  Row b uses state line conv_state_indices[b] (or b);
 * a pad line skips the row, leaving out and the state untouched.  The state
 * is always read (there is no has_initial_state in decode):
 *   u = conv_state[line, c, 0..W-2] ++ x[b, c, 0..seqlen-1]
 *   out[b, c, t] = act(bias[c] + sum_k w[c,k] * u[t+k])
 * and the state is shifted left by one column and the new inputs appended
 * ([P1] update kernel, STEP 2):
 *   conv_state[line, c, j] = u[1 + j],  j = 0 .. W-3+seqlen
 * which needs state_len >= W-2+seqlen columns of storage (checked by the
 * caller).  For seqlen == 1 this is the classic [s1..s_{W-2}, x].
 */
int oracle_ccv_update(const uint16_t *x, int64_t xs_b, int64_t xs_d, int64_t xs_t,
                      uint16_t *out, int64_t os_b, int64_t os_d, int64_t os_t,
                      const uint16_t *weight, int64_t ws_dim, int64_t ws_w,
                      const uint16_t *bias,
                      uint16_t *conv_state, int64_t ss_line, int64_t ss_dim, int64_t ss_tok,
                      int num_cache_lines,
                      const int32_t *conv_state_indices, int batch, int dim, int seqlen,
                      int width, int pad_slot_id, int silu, int *err_count) {
    const int W = width;
    uint16_t *u_bits = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(W - 1 + seqlen));
    for (int b = 0; b < batch; b++) {
        int line = conv_state_indices ? conv_state_indices[b] : b;
        if (line == pad_slot_id) continue;
        if (line < 0 || line >= num_cache_lines) {
            count_error(err_count);
            continue;
        }
        for (int c = 0; c < dim; c++) {
            for (int j = 0; j < W - 1; j++)
                u_bits[j] = conv_state[line * ss_line + c * ss_dim + j * ss_tok];
            for (int t = 0; t < seqlen; t++)
                u_bits[W - 1 + t] = x[b * xs_b + c * xs_d + t * xs_t];

            float bc = bias ? bf16_to_f32(bias[c]) : 0.0f;
            for (int t = 0; t < seqlen; t++) {
                float acc = bc;
                for (int k = 0; k < W; k++)
                    acc = acc + bf16_to_f32(weight[c * ws_dim + k * ws_w]) *
                                    bf16_to_f32(u_bits[t + k]);
                if (silu) acc = silu_f32(acc);
                out[b * os_b + c * os_d + t * os_t] = f32_to_bf16(acc);
            }
            for (int j = 0; j < W - 2 + seqlen; j++)
                conv_state[line * ss_line + c * ss_dim + j * ss_tok] = u_bits[1 + j];
        }
    }
    free(u_bits);
    return 0;
}

/*
 * oracle_ccv_update_spec -- [P1] `causal_conv1d_update` with its
 * speculative-decoding extras (`num_accepted_tokens`,
 * `intermediate_conv_window`, `output_state_indices`).
 *
 * Row b reads its window from state columns off .. off+W-2 of its line, where
 * off = num_accepted_tokens[b] - 1 (0 without it): [P1] rolls the state as
 * [history.., draft1..draftN] and a verify step that accepted k drafts starts
 * k-1 columns in.  With u = those W-1 columns ++ x[b, c, 0..seqlen-1]:
 *   out[b, c, t] = act(bias[c] + sum_k w[c,k] * u[t+k])
 * and the window after token t is u[t+1 .. t+W-1].  For each t that window
 * is written to intermediate_conv_window[b, t, c, 0..W-2] (indexed by the
 * batch position, not the state line) and, when output_state_indices[b, t]
 * >= 0, to columns 0..W-2 of that state line.  When neither buffer is given
 * the state is shifted in place instead, as in the plain update:
 *   conv_state[line, c, j] = u[1 + j],  j = 0 .. W-3+seqlen.
 * A row whose offset leaves no room for W-1 columns (off < 0 or off+W-1 >
 * state_len), or an output line outside the pool, is counted in err_count
 * and skipped (the row, or that one window write).  Output lines must not be
 * lines that other rows of the same call read.
 */
int oracle_ccv_update_spec(const uint16_t *x, int64_t xs_b, int64_t xs_d, int64_t xs_t,
                           uint16_t *out, int64_t os_b, int64_t os_d, int64_t os_t,
                           const uint16_t *weight, int64_t ws_dim, int64_t ws_w,
                           const uint16_t *bias,
                           uint16_t *conv_state, int64_t ss_line, int64_t ss_dim, int64_t ss_tok,
                           int num_cache_lines, int state_len,
                           const int32_t *conv_state_indices, const int32_t *num_accepted_tokens,
                           uint16_t *inter, int64_t is_b, int64_t is_t, int64_t is_d, int64_t is_w,
                           const int32_t *out_state_idx, int64_t ois_b, int64_t ois_t,
                           int batch, int dim, int seqlen,
                           int width, int pad_slot_id, int silu, int *err_count) {
    const int W = width;
    const int shift = inter == NULL && out_state_idx == NULL;
    uint16_t *u_bits = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(W - 1 + seqlen));
    for (int b = 0; b < batch; b++) {
        int line = conv_state_indices ? conv_state_indices[b] : b;
        if (line == pad_slot_id) continue;
        if (line < 0 || line >= num_cache_lines) {
            count_error(err_count);
            continue;
        }
        int off = num_accepted_tokens ? num_accepted_tokens[b] - 1 : 0;
        if (off < 0 || off + W - 1 > state_len) {
            count_error(err_count);
            continue;
        }
        for (int t = 0; t < seqlen && out_state_idx; t++) {
            int o = out_state_idx[b * ois_b + t * ois_t];
            if (o >= num_cache_lines) count_error(err_count);
        }
        for (int c = 0; c < dim; c++) {
            for (int j = 0; j < W - 1; j++)
                u_bits[j] = conv_state[line * ss_line + c * ss_dim + (off + j) * ss_tok];
            for (int t = 0; t < seqlen; t++)
                u_bits[W - 1 + t] = x[b * xs_b + c * xs_d + t * xs_t];

            float bc = bias ? bf16_to_f32(bias[c]) : 0.0f;
            for (int t = 0; t < seqlen; t++) {
                float acc = bc;
                for (int k = 0; k < W; k++)
                    acc = acc + bf16_to_f32(weight[c * ws_dim + k * ws_w]) *
                                    bf16_to_f32(u_bits[t + k]);
                if (silu) acc = silu_f32(acc);
                out[b * os_b + c * os_d + t * os_t] = f32_to_bf16(acc);
                for (int j = 0; j < W - 1; j++) {
                    uint16_t v = u_bits[t + 1 + j];
                    if (inter) inter[b * is_b + t * is_t + c * is_d + j * is_w] = v;
                    if (out_state_idx) {
                        int o = out_state_idx[b * ois_b + t * ois_t];
                        if (o >= 0 && o < num_cache_lines)
                            conv_state[o * ss_line + c * ss_dim + j * ss_tok] = v;
                    }
                }
            }
            if (shift)
                for (int j = 0; j < W - 2 + seqlen; j++)
                    conv_state[line * ss_line + c * ss_dim + j * ss_tok] = u_bits[1 + j];
        }
    }
    free(u_bits);
    return 0;
}

/* ------------------------------------------------------ paged metadata ---- */

/*
 * oracle_paged_sconv_seq_metadata -- [P2] `sconv_seq_metadata`.
 * For token t < num_actual_tokens: seq_idx[t] is the largest j in
 * [0, num_reqs) with query_start_loc[j] <= t (0 if there is none) and
 * query_start[t] = query_start_loc[seq_idx[t]].  Padded rows
 * num_actual_tokens <= t < num_padded_tokens get 0 in both.  Rows at or past
 * num_padded_tokens are not written.
 */
int oracle_paged_sconv_seq_metadata(const int32_t *query_start_loc, int num_reqs,
                                    int num_actual_tokens, int num_padded_tokens,
                                    int32_t *seq_idx_out, int32_t *query_start_out) {
    for (int t = 0; t < num_padded_tokens; t++) {
        if (t >= num_actual_tokens) {
            seq_idx_out[t] = 0;
            query_start_out[t] = 0;
            continue;
        }
        int owner = 0;
        for (int j = 0; j < num_reqs; j++)
            if (query_start_loc[j] <= t) owner = j;
        seq_idx_out[t] = owner;
        query_start_out[t] = query_start_loc[owner];
    }
    return 0;
}

/* --------------------------------------------------- paged short conv ---- */

/*
 * oracle_paged_sconv_fwd -- [P2] `_fused_sconv_kernel` / `fused_sconv`.
 *
 * x and out are [T, C] with C = H*ws channels, head-major (channel c belongs
 * to head c/ws and lives at cache D-index off_s + c%ws).  The cache is
 * [num_blocks, H, N, D] with D contiguous and holds the conv input at every
 * absolute position.  Token t with slot_mapping[t] >= 0 is real; a negative
 * slot marks a PAD row.
 *
 * Step 2 (convolve), for every token t and channel c, taps iw = 0..W-1:
 *   src = positions[t] - (W-1) + iw        absolute window position
 *   row = t - (W-1) + iw                   x row holding src in this forward
 *   value = 0                         if PAD or src < 0
 *         = x[row, c]                 if row >= query_start[t]   (in-forward)
 *         = cache[block_table[seq_idx[t], min(src/N, max_blocks-1)],
 *                 c/ws, src%N, off_s + c%ws]   otherwise        (pre-forward)
 *   acc = sum_iw value * w[c, iw]      (fp32, no bias), then SiLU, then
 *   + x[t, c] when residual is on; out[t, c] = bf16(acc).
 * Pre-forward taps are read from the cache as it was before this forward.
 *
 * Step 1 (insert): for every real token, cache[slot/N, c/ws, slot%N,
 * off_s + c%ws] = x[t, c] (a bit copy).
 *
 * The pages run both steps in one launch and rely on the just-written slots
 * never being pre-forward taps of the same forward; reading the pre-forward
 * cache and inserting afterwards is the same thing under that assumption.
 *
 * Invalid data-dependent indices (request outside the block table, physical
 * block outside [0, num_blocks), negative x row) read 0 / skip the write and
 * bump *err_count.
 */
int oracle_paged_sconv_fwd(const uint16_t *x, int64_t xs_t,
                           uint16_t *cache, int64_t cs_blk, int64_t cs_h, int64_t cs_n,
                           int num_blocks, int H, int N, int D,
                           const uint16_t *weight, int64_t ws_c, int64_t ws_w,
                           uint16_t *out, int64_t os_t,
                           const int64_t *positions, const int32_t *seq_idx,
                           const int64_t *slot_mapping, const int32_t *block_table,
                           int64_t bt_stride_r, int bt_rows, int max_blocks,
                           const int32_t *query_start, int T, int off_s, int ws,
                           int width, int silu, int residual, int *err_count) {
    const int W = width;
    const int C = H * ws;
    (void)D;
    /* Step 2 first: every cache read sees the pre-forward cache. */
    for (int t = 0; t < T; t++) {
        int real = slot_mapping[t] >= 0;
        for (int c = 0; c < C; c++) {
            int head = c / ws;
            int cd = off_s + c % ws;
            float acc = 0.0f;
            for (int iw = 0; iw < W; iw++) {
                int64_t src = positions[t] - (W - 1) + iw;
                int64_t row = (int64_t)t - (W - 1) + iw;
                float v = 0.0f;
                if (real && src >= 0) {
                    if (row >= query_start[t]) {
                        if (row < 0) {
                            count_error(err_count);
                        } else {
                            v = bf16_to_f32(x[row * xs_t + c]);
                        }
                    } else {
                        int req = seq_idx[t];
                        int64_t lblk = src / N;
                        if (lblk > max_blocks - 1) lblk = max_blocks - 1;
                        if (req < 0 || req >= bt_rows) {
                            count_error(err_count);
                        } else {
                            int64_t blk = block_table[req * bt_stride_r + lblk];
                            if (blk < 0 || blk >= num_blocks) {
                                count_error(err_count);
                            } else {
                                v = bf16_to_f32(cache[blk * cs_blk + head * cs_h +
                                                      (src % N) * cs_n + cd]);
                            }
                        }
                    }
                }
                acc = acc + v * bf16_to_f32(weight[c * ws_c + iw * ws_w]);
            }
            if (silu) acc = silu_f32(acc);
            if (residual) acc = acc + bf16_to_f32(x[(int64_t)t * xs_t + c]);
            out[(int64_t)t * os_t + c] = f32_to_bf16(acc);
        }
    }
    /* Step 1: insert every real token's input at its slot. */
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / N;
        if (blk >= num_blocks) {
            count_error(err_count);
            continue;
        }
        for (int c = 0; c < C; c++)
            cache[blk * cs_blk + (c / ws) * cs_h + (slot % N) * cs_n + off_s + c % ws] =
                x[(int64_t)t * xs_t + c];
    }
    return 0;
}
