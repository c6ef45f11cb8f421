/*
 * CPU oracle for the batched speculative-verify causal depthwise conv1d update.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the bench's CPU-baseline leg
 * may call this file; the product path never does.  It shares no code, header, table or helper
 * with the CUDA library: it is a plain, slow, single-threaded loop that states the definition.
 *
 * What it computes, with the passages it follows:
 *
 *   - Causal depthwise conv1d update over T draft tokens (sglang PR #46184, "Motivation": chain
 *     verify runs the conv update with an intermediate window; Atlas fn
 *     gdn_verify_fused_conv_kn_batched: the K draft positions of a batch are handled by a single
 *     launch).  For one channel c the
 *     sequence is full = [state[o .. o+W-2], x_0 .. x_{T-1}] (W-1 committed inputs, then the T new
 *     ones) and token t sees the W inputs full[t .. t+W-1]:
 *         acc_t = bias[c] + sum_{j=0}^{W-1} w[c][j] * full[t+j]
 *     so w[c][W-1] multiplies the newest input x_t (the textbook causal convolution).  fp32
 *     accumulate, bias first, taps in ascending j, every product rounded before its add (no fused
 *     multiply-add: this file is built with -ffp-contract=off).
 *   - SiLU fused into the conv (glm5next_kda mod.rs, module doc: the decode conv is followed by
 *     SiLU and then by an L2 normalisation of q and k alone):
 *         y_t = acc_t / (1 + exp(-acc_t))            in fp32.
 *   - L2 normalisation of the q|k channels only, per head_dim group, exactly once, V never
 *     (mod.rs module doc: the decode conv applies the normalisation to q and k a single time and
 *     leaves V alone), with the eps inside the square root (mod.rs Glm5NextKdaConfig::l2_eps: eps
 *     is added to the sum of squares under the root, it is not a floor on the norm):
 *         y_t[c] *= 1 / sqrt(sum_{c' in group(c)} y_t[c']^2 + eps)     for c < qk_channels.
 *     The sum runs over the group's channels in ascending order.  The result is rounded once to
 *     the output type (round to nearest even for bf16).
 *   - Per-token rollback snapshots (Atlas fn gdn_verify_fused_conv_kn_batched: the kernel also
 *     stores, for each draft token, the conv state a rollback would return to; mod.rs decode_k:
 *     snapshot t is the state AFTER row t).  Snapshot t of channel c is the committed window after token t, full[t+1 .. t+W-1],
 *     copied as raw bits.  Dense layout: element (s, t, c, k) at
 *         s*seq + t*step + c*ch + k*col.
 *     Deduplicated layout (sglang PR #46184, "Motivation" and "Modifications"): one
 *     [dim, T+W-2] row per sequence seen as an overlapping [T, dim, W-1] view whose step stride
 *     equals its column stride, so element (s, t, c, k) lives at s*seq + (t+k)*col + c*ch.  The
 *     oracle writes every (t, k) of the view one by one: this is the per-token store path, which
 *     the PR shows to hit the same addresses with the same values as the row written once.
 *   - The state is left holding the committed window after the last token, full[T .. T+W-2]
 *     (Atlas fn doc: after the call the state holds the window past the final draft position),
 *     written to state columns [0, W-1).  Columns at and above W-1 are not touched.
 *   - Padded sequences (cache index < 0) touch nothing (PR #46184, "Modifications": padded rows
 *     leave the kernel before storing anything).
 *   - An optional per-sequence offset o into the state row says where the committed window is
 *     read (PR #46184, "Modifications", test coverage: an offset into the state given by the
 *     number of accepted tokens).
 *   - History-row state (a reading, not a printed kernel): PR #46184's slots hold one [dim, T+K-2]
 *     window row, and its tests cover an accepted-token offset into the state.  In the
 *     history layout the state row itself is that row: the call reads its committed window at
 *     columns [o, o+W-1) and then writes columns [0, T+W-2) of the same row with the row
 *     [full[1 .. W-2], x_0 .. x_{T-1}], through the same per-token view (element (t, k) at column
 *     t+k) the dedup layout uses.  Snapshot a-1 then sits at columns [a-1, a+W-2), so the next
 *     call passes o = a-1 and no commit is needed.  No separate window buffer is written; columns
 *     at and above T+W-2 are not touched.
 *   - Recompute rollback (memra-engine Engine doc, ssm_conv_ring_rebuild_dc: the conv state is rebuilt
 *     from the ring kept from before the verify, the verify's inputs and the device-side accept
 *     count).  In the recompute layout the verify writes the outputs only: no snapshots, and the
 *     state keeps the pre-verify window.  The commit then sets state[k] = full[a+k] for k < W-1,
 *     with full = [state[0 .. W-2], x_0 .. x_{T-1}] read at commit time -- the same value snapshot
 *     a-1 holds.
 *   - Commit: restore the state to the snapshot of the accepted prefix (PR #46184, "Motivation":
 *     the window exists so the state can be rolled back to the accepted prefix after verify;
 *     mod.rs decode_k:
 *     snapshot t is what a partial accept rewinds to).  With a accepted tokens (1 <= a <= T) the
 *     state becomes snapshot a-1.
 *
 *   - Mixed dtypes (sglang PR #46184, "Accuracy Tests": its extra check covers mixed input and state
 *     dtypes).  The state and the snapshots may be stored in the other dtype than x, out, weight and
 *     bias.  The arithmetic widens every input exactly to fp32; the snapshots and the state hold
 *     the inputs converted to the state dtype: raw bits when the dtypes agree, an exact widening
 *     for bf16 inputs into fp32 state, and round-to-nearest-even (any NaN to the quiet NaN) for
 *     fp32 inputs into bf16 state.
 *   - Tree verify (sglang PR #46184, "Scope": tree verify keeps dense windows and per-token stores).
 *     Draft token t has a parent p(t) in [-1, t) (-1: the committed window).  Its conv sees the
 *     parent's window followed by x_t, and its snapshot is that window shifted by one with x_t
 *     appended: window(t) = [window(p)[1 .. W-2], x_t], window(-1) = the committed window.  A
 *     chain (p(t) = t-1) is the plain verify.  The state is left on window(T-1), as for a chain;
 *     the commit restores the window of the accepted path's last token (accept_len = its index + 1).
 *     Only the dense layout holds tree snapshots.  A parent outside [-1, t) flags the sequence (32).
 *   - Packed ragged verify (sglang PR #46184, "Related upstream work": a packed variable-length
 *     update, and target verify run on packed ragged tokens with the tile store covering the
 *     packed rows).  Sequence s owns draft tokens [cu[s], cu[s+1]) of x and out, packed back to
 *     back (row cu[s]+t holds its token t); its draft count T_s = cu[s+1]-cu[s] lies in [0, T],
 *     where T is the call's maximum and sizes the window buffer.  Everything above holds with T_s
 *     in place of T for that sequence: outputs for its T_s rows, snapshots t < T_s (snapshot steps
 *     t >= T_s are not written, and in the deduplicated layout only columns [0, T_s+W-2), the ones
 *     the per-token stores write, are), the state left on full[T_s .. T_s+W-2].  T_s = 0 writes no
 *     output and no snapshot; the state then receives the committed window itself.  A span that
 *     is reversed, leaves [0, total_tokens) or is longer than T flags the sequence (16).  The commit
 *     accepts a in 1..T_s; a sequence with T_s = 0 has nothing to commit and is skipped.
 *   - Prefill (glm5next_kda mod.rs, the prefill path of the layer: the conv over all T prompt
 *     tokens with SiLU, then the L2 normalisation of q|k, which that code runs as a second launch;
 *     here the normalisation is applied to the fp32 SiLU values and rounded once, as in decode).
 *     Packed variable-length sequences: sequence s owns tokens [cu[s], cu[s+1]) of x and out.
 *     full = [initial window, x_0 .. x_{L-1}], the initial window being state[0 .. W-2] when the
 *     sequence has an initial state and zeros otherwise; out_t is the verify's output for token t;
 *     the state is left holding the last W-1 entries of full.
 *
 * Status codes written per sequence (same meaning as the library's): 1 = cache slot out of range,
 * 2 = state offset out of range, 4 = accept count out of range, 16 = token span invalid (prefill,
 * packed ragged verify),
 * 32 = a draft token's parent outside [-1, t) (tree verify).
 * A flagged sequence is untouched.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t n_seq, T, dim, width, qk_channels, head_dim;
    int32_t is_bf16; /* 0: fp32 elements, 1: bf16 elements (every buffer) */
    float l2_eps;
    const void *x;
    int64_t x_seq, x_tok;
    void *out;
    int64_t out_seq, out_tok;
    void *state;
    int32_t n_slots, state_cols;
    int64_t st_slot, st_ch;
    const int32_t *cache_idx; /* NULL: sequence s uses slot s */
    const int32_t *state_off; /* NULL: offset 0 */
    const void *weight;       /* [dim][W] */
    const void *bias;         /* [dim] or NULL */
    void *window;
    int32_t dedup;
    int64_t w_seq, w_step, w_ch, w_col;
    int32_t *status; /* [n_seq] or NULL */
    int32_t history;   /* 1: the state row is the snapshot row (no window buffer) */
    int32_t recompute; /* 1: outputs only; no snapshots and the state is not written */
    int32_t state_is_bf16; /* dtype of state and window: 0 fp32, 1 bf16 (may differ from is_bf16) */
    const int32_t *parent; /* [n_seq][T] parent of each draft token (-1: the committed window) or NULL */
    const int32_t *cu_draft; /* [n_seq + 1] packed draft rows of x and out, or NULL (T each) */
    int32_t total_tokens;    /* rows of x and out when cu_draft is given */
} oracle_verify_args;

typedef struct {
    int32_t n_seq, T, dim, width, is_bf16;
    void *state;
    int32_t n_slots;
    int64_t st_slot, st_ch;
    const int32_t *cache_idx;
    const void *window;
    int32_t dedup;
    int64_t w_seq, w_step, w_ch, w_col;
    const int32_t *accept_len;
    int32_t *status;
    int32_t recompute; /* 1: rebuild from the state's window and x (no window buffer) */
    const void *x;
    int64_t x_seq, x_tok;
    const int32_t *cu_draft; /* [n_seq + 1] as in the verify, or NULL (T tokens each) */
    int32_t total_tokens;
} oracle_commit_args;

/* ---- element access: raw bits, so copies keep NaN payloads and signed zeros ---- */

static uint32_t get_bits(const void *base, int is_bf16, int64_t i) {
    if (is_bf16) return ((const uint16_t *)base)[i];
    return ((const uint32_t *)base)[i];
}

static void put_bits(void *base, int is_bf16, int64_t i, uint32_t v) {
    if (is_bf16)
        ((uint16_t *)base)[i] = (uint16_t)v;
    else
        ((uint32_t *)base)[i] = v;
}

static float bits_to_float(uint32_t v, int is_bf16) {
    /* bf16 is the upper half of an IEEE binary32: widening is exact. */
    uint32_t u = is_bf16 ? (v << 16) : v;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t float_to_bits(float f, int is_bf16) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (!is_bf16) return u;
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u; /* any NaN -> quiet NaN */
    /* round to nearest, ties to even, on the 16 dropped bits */
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return u >> 16;
}

/* An element of x (dtype xbf) in the state's dtype (sbf): raw bits when they agree, else widened
 * exactly (bf16 -> fp32) or rounded to nearest even (fp32 -> bf16). */
static uint32_t to_state_bits(uint32_t v, int xbf, int sbf) {
    if (xbf == sbf) return v;
    if (xbf) return v << 16;
    return float_to_bits(bits_to_float(v, 0), 1);
}

static int64_t win_index(const oracle_verify_args *a, int s, int t, int c, int k) {
    int64_t step = a->dedup ? a->w_col : a->w_step;
    return (int64_t)s * a->w_seq + (int64_t)t * step + (int64_t)c * a->w_ch + (int64_t)k * a->w_col;
}

/* Returns 0; per-sequence problems go to status[]. */
int oracle_conv_verify(const oracle_verify_args *a) {
    const int W = a->width, T = a->T, dim = a->dim, bf = a->is_bf16, sbf = a->state_is_bf16;
    uint32_t full[1024];  /* W-1 + T elements of one channel, as bits of the state's dtype */
    float fullf[1024];    /* the same inputs widened to fp32 (exact) */
    if (W < 1 || T < 1 || dim < 1 || W - 1 + T > 1024) return -1;
    if (a->history && T + W - 2 > a->state_cols) return -3;
    if (a->cu_draft && a->parent) return -4; /* packed rows are chains only */
    /* y[t*dim + c]: post-SiLU fp32 values of one sequence, normalised in place below */
    float *y = (float *)malloc(sizeof(float) * (size_t)T * (size_t)dim);
    if (!y) return -2;

    for (int s = 0; s < a->n_seq; ++s) {
        const int slot = a->cache_idx ? a->cache_idx[s] : s;
        const int o = a->state_off ? a->state_off[s] : 0;
        int st = 0;
        if (slot >= 0 && slot >= a->n_slots) st |= 1;
        if (slot >= 0 && (o < 0 || o + W - 1 > a->state_cols)) st |= 2;
        if (slot >= 0 && a->parent)
            for (int t = 0; t < T; ++t) {
                const int par = a->parent[(int64_t)s * T + t];
                if (par < -1 || par >= t) st |= 32;
            }
        /* the sequence's draft rows: T rows at x[s] (sequence stride), or its packed span
           [cu[s], cu[s+1]) of T_s rows (token stride only) */
        int Ts = T;
        int64_t xrow = (int64_t)s * a->x_seq, orow = (int64_t)s * a->out_seq;
        if (a->cu_draft) {
            const int b = a->cu_draft[s], e = a->cu_draft[s + 1];
            if (slot >= 0 && (b < 0 || e < b || e > a->total_tokens || e - b > T)) st |= 16;
            Ts = e - b;
            xrow = (int64_t)b * a->x_tok;
            orow = (int64_t)b * a->out_tok;
        }
        if (a->status) a->status[s] = st;
        if (slot < 0 || st) continue;

        if (a->parent) {
            /* wbits[(t+1)*(W-1) + k]: window after token t (entry 0: the committed window), as bits of
               the state's dtype; wf: the same values widened */
            const int R = W - 1;
            uint32_t *wbits = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(T + 1) * (size_t)R + 4);
            float *wf = (float *)malloc(sizeof(float) * (size_t)(T + 1) * (size_t)R + 4);
            if (!wbits || !wf) {
                free(wbits);
                free(wf);
                free(y);
                return -2;
            }
            for (int c = 0; c < dim; ++c) {
                const int64_t srow = (int64_t)slot * a->st_slot + (int64_t)c * a->st_ch;
                for (int k = 0; k < R; ++k) {
                    wbits[k] = get_bits(a->state, sbf, srow + o + k);
                    wf[k] = bits_to_float(wbits[k], sbf);
                }
                for (int t = 0; t < T; ++t) {
                    const int base = (a->parent[(int64_t)s * T + t] + 1) * R;
                    const uint32_t xv = get_bits(a->x, bf, xrow + (int64_t)t * a->x_tok + c);
                    const float xf = bits_to_float(xv, bf);
                    float acc = a->bias ? bits_to_float(get_bits(a->bias, bf, c), bf) : 0.0f;
                    for (int j = 0; j < W; ++j) {
                        const float wj = bits_to_float(get_bits(a->weight, bf, (int64_t)c * W + j), bf);
                        const float prod = wj * (j < R ? wf[base + j] : xf);
                        acc = acc + prod;
                    }
                    y[(int64_t)t * dim + c] = acc / (1.0f + expf(-acc));
                    const int nb = (t + 1) * R;
                    for (int k = 0; k + 1 < R; ++k) {
                        wbits[nb + k] = wbits[base + k + 1];
                        wf[nb + k] = wf[base + k + 1];
                    }
                    wbits[nb + R - 1] = to_state_bits(xv, bf, sbf);
                    wf[nb + R - 1] = xf;
                    for (int k = 0; k < R; ++k) put_bits(a->window, sbf, win_index(a, s, t, c, k), wbits[nb + k]);
                }
                for (int k = 0; k < R; ++k) put_bits(a->state, sbf, srow + k, wbits[T * R + k]);
            }
            free(wbits);
            free(wf);
        } else
        for (int c = 0; c < dim; ++c) {
            const int64_t srow = (int64_t)slot * a->st_slot + (int64_t)c * a->st_ch;
            for (int k = 0; k < W - 1; ++k) {
                full[k] = get_bits(a->state, sbf, srow + o + k);
                fullf[k] = bits_to_float(full[k], sbf);
            }
            for (int t = 0; t < Ts; ++t) {
                const uint32_t xv = get_bits(a->x, bf, xrow + (int64_t)t * a->x_tok + c);
                full[W - 1 + t] = to_state_bits(xv, bf, sbf);
                fullf[W - 1 + t] = bits_to_float(xv, bf);
            }

            for (int t = 0; t < Ts; ++t) {
                float acc = a->bias ? bits_to_float(get_bits(a->bias, bf, c), bf) : 0.0f;
                for (int j = 0; j < W; ++j) {
                    const float wj = bits_to_float(get_bits(a->weight, bf, (int64_t)c * W + j), bf);
                    const float prod = wj * fullf[t + j];
                    acc = acc + prod;
                }
                y[(int64_t)t * dim + c] = acc / (1.0f + expf(-acc));
            }

            if (a->recompute) continue; /* outputs only: the state keeps the pre-verify window */

            if (a->history) {
                /* snapshot t into the state row itself, at columns t .. t+W-2 (after every read) */
                for (int t = 0; t < Ts; ++t)
                    for (int k = 0; k < W - 1; ++k) put_bits(a->state, sbf, srow + t + k, full[t + 1 + k]);
                continue;
            }

            /* snapshot t = window after token t = full[t+1 .. t+W-1] */
            for (int t = 0; t < Ts; ++t)
                for (int k = 0; k < W - 1; ++k) put_bits(a->window, sbf, win_index(a, s, t, c, k), full[t + 1 + k]);

            /* committed window after the last token, written after every read of this row */
            for (int k = 0; k < W - 1; ++k) put_bits(a->state, sbf, srow + k, full[Ts + k]);
        }

        for (int t = 0; t < Ts; ++t) {
            float *yt = y + (int64_t)t * dim;
            if (a->qk_channels > 0) {
                const int hd = a->head_dim;
                for (int g = 0; g + hd <= a->qk_channels; g += hd) {
                    float ss = 0.0f;
                    for (int c = g; c < g + hd; ++c) {
                        const float sq = yt[c] * yt[c];
                        ss = ss + sq;
                    }
                    const float r = 1.0f / sqrtf(ss + a->l2_eps);
                    for (int c = g; c < g + hd; ++c) yt[c] = yt[c] * r;
                }
            }
            for (int c = 0; c < dim; ++c)
                put_bits(a->out, bf, orow + (int64_t)t * a->out_tok + c, float_to_bits(yt[c], bf));
        }
    }
    free(y);
    return 0;
}

int oracle_conv_commit(const oracle_commit_args *a) {
    const int W = a->width, bf = a->is_bf16;
    if (a->recompute && W - 1 + a->T > 1024) return -1;
    for (int s = 0; s < a->n_seq; ++s) {
        const int slot = a->cache_idx ? a->cache_idx[s] : s;
        int st = 0;
        if (slot >= 0 && slot >= a->n_slots) st |= 1;
        /* draft count and rows as in the verify (packed span, or T rows at x[s]) */
        int Ts = a->T;
        int64_t xrow = (int64_t)s * a->x_seq;
        if (a->cu_draft) {
            const int b = a->cu_draft[s], e = a->cu_draft[s + 1];
            if (slot >= 0 && (b < 0 || e < b || e > a->total_tokens || e - b > a->T)) st |= 16;
            Ts = e - b;
            xrow = (int64_t)b * a->x_tok;
        }
        const int acc = a->accept_len[s];
        if (slot >= 0 && !(st & 16) && Ts > 0 && (acc < 1 || acc > Ts)) st |= 4;
        if (a->status) a->status[s] = st;
        if (slot < 0 || st) continue;
        if (Ts == 0) continue; /* no draft token was verified: nothing to commit */
        const int t = acc - 1;
        if (a->recompute) {
            for (int c = 0; c < a->dim; ++c) {
                const int64_t srow = (int64_t)slot * a->st_slot + (int64_t)c * a->st_ch;
                uint32_t full[1024]; /* W-1 + T_s raw elements of one channel */
                for (int k = 0; k < W - 1; ++k) full[k] = get_bits(a->state, bf, srow + k);
                for (int u = 0; u < Ts; ++u)
                    full[W - 1 + u] = get_bits(a->x, bf, xrow + (int64_t)u * a->x_tok + c);
                /* snapshot acc-1 = full[acc .. acc+W-2], written after the row's reads */
                for (int k = 0; k < W - 1; ++k) put_bits(a->state, bf, srow + k, full[acc + k]);
            }
            continue;
        }
        const int64_t step = a->dedup ? a->w_col : a->w_step;
        for (int c = 0; c < a->dim; ++c)
            for (int k = 0; k < W - 1; ++k) {
                const int64_t src = (int64_t)s * a->w_seq + (int64_t)t * step + (int64_t)c * a->w_ch + (int64_t)k * a->w_col;
                const int64_t dst = (int64_t)slot * a->st_slot + (int64_t)c * a->st_ch + k;
                put_bits(a->state, bf, dst, get_bits(a->window, bf, src));
            }
    }
    return 0;
}

typedef struct {
    int32_t n_seq, dim, width, qk_channels, head_dim, is_bf16;
    float l2_eps;
    int32_t total_tokens;
    const void *x;
    int64_t x_tok;
    void *out;
    int64_t out_tok;
    const int32_t *cu_seqlens;        /* [n_seq + 1] */
    void *state;
    int32_t n_slots, state_cols;
    int64_t st_slot, st_ch;
    const int32_t *cache_idx;         /* NULL: sequence s uses slot s */
    const int32_t *has_initial_state; /* NULL: every sequence has one */
    const void *weight, *bias;
    int32_t *status;
} oracle_prefill_args;

int oracle_conv_prefill(const oracle_prefill_args *a) {
    const int W = a->width, dim = a->dim, bf = a->is_bf16;
    for (int s = 0; s < a->n_seq; ++s) {
        const int slot = a->cache_idx ? a->cache_idx[s] : s;
        const int b = a->cu_seqlens[s], e = a->cu_seqlens[s + 1];
        int st = 0;
        if (slot >= 0 && slot >= a->n_slots) st |= 1;
        if (slot >= 0 && (b < 0 || e < b || e > a->total_tokens)) st |= 16;
        if (a->status) a->status[s] = st;
        if (slot < 0 || st) continue;
        const int L = e - b;
        const int init = a->has_initial_state ? a->has_initial_state[s] != 0 : 1;
        uint32_t *full = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(W - 1 + L));
        float *y = (float *)malloc(sizeof(float) * ((size_t)L * (size_t)dim + 1));
        if (!full || !y) {
            free(full);
            free(y);
            return -2;
        }
        for (int c = 0; c < dim; ++c) {
            const int64_t srow = (int64_t)slot * a->st_slot + (int64_t)c * a->st_ch;
            for (int k = 0; k < W - 1; ++k) full[k] = init ? get_bits(a->state, bf, srow + k) : 0u;
            for (int t = 0; t < L; ++t) full[W - 1 + t] = get_bits(a->x, bf, (int64_t)(b + t) * a->x_tok + c);
            for (int t = 0; t < L; ++t) {
                float acc = a->bias ? bits_to_float(get_bits(a->bias, bf, c), bf) : 0.0f;
                for (int j = 0; j < W; ++j) {
                    const float wj = bits_to_float(get_bits(a->weight, bf, (int64_t)c * W + j), bf);
                    const float prod = wj * bits_to_float(full[t + j], bf);
                    acc = acc + prod;
                }
                y[(int64_t)t * dim + c] = acc / (1.0f + expf(-acc));
            }
            /* the last W-1 entries of full, after every read of this row */
            for (int k = 0; k < W - 1; ++k) put_bits(a->state, bf, srow + k, full[L + k]);
        }
        for (int t = 0; t < L; ++t) {
            float *yt = y + (int64_t)t * dim;
            if (a->qk_channels > 0) {
                const int hd = a->head_dim;
                for (int g = 0; g + hd <= a->qk_channels; g += hd) {
                    float ss = 0.0f;
                    for (int c = g; c < g + hd; ++c) {
                        const float sq = yt[c] * yt[c];
                        ss = ss + sq;
                    }
                    const float r = 1.0f / sqrtf(ss + a->l2_eps);
                    for (int c = g; c < g + hd; ++c) yt[c] = yt[c] * r;
                }
            }
            for (int c = 0; c < dim; ++c)
                put_bits(a->out, bf, (int64_t)(b + t) * a->out_tok + c, float_to_bits(yt[c], bf));
        }
        free(full);
        free(y);
    }
    return 0;
}

/* Exposed so the tests can pin the rounding against an independent library conversion. */
uint32_t oracle_round_f32_to_bf16(float f) { return float_to_bits(f, 1); }
