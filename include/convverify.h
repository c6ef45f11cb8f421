/*
 * convverify.h -- C ABI of the batched speculative-verify causal depthwise conv1d update.
 *
 * One verify call runs, for n_seq sequences of T draft tokens each, the conv update of a hybrid
 * GDN/KDA/Mamba2 layer over all T positions in one launch, and writes every per-token rollback
 * snapshot of the conv window; one commit call later restores the state of the accepted prefix.
 *
 * Sources (the pages this library follows):
 *   [atlas-batched]  Atlas spark_model API doc, fn gdn_verify_fused_conv_kn_batched: one launch
 *                    covers the K draft positions, the kernel itself stores each position's
 *                    rollback snapshot into a strided buffer, the state ends on the committed
 *                    window, and the batch over n_seq (per-sequence strides) matches n separate
 *                    calls bit for bit.
 *   [sglang-46184]   sglang pull request #46184 (dedup conv window tile store), sections
 *                    "Motivation" and "Modifications": the deduplicated [dim, T+K-2] window row
 *                    seen as an overlapping [T, dim, K-1] view whose step stride equals its
 *                    column stride; the window of step t starts at column t of the row that
 *                    follows the first committed column with x_0 .. x_{T-1}; padded rows store
 *                    nothing; the tests cover an accepted-token offset into the state.
 *   [kda-mod]        Atlas spark_model/layers/glm5next_kda/mod.rs: conv1d with SiLU, then an L2
 *                    normalisation of the q|k channels alone (V untouched), eps under the root; decode_k snapshot
 *                    t = state after row t, which a partial accept rewinds to.
 *
 * Conventions for every entry point:
 *   - Strides are in ELEMENTS and must be >= 0.  The channel stride of x, out and weight is 1, and
 *     the column stride of conv_state is 1.
 *   - Every data pointer is a DEVICE pointer (or managed memory) unless stated otherwise.  The
 *     caller owns every buffer: the library allocates, frees and synchronises nothing, launches
 *     asynchronously on `stream`, and keeps no pointer after it returns.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *   - Invalid arguments are reported by a negative status before anything is launched; nothing is
 *     written then.  Problems that only the device can see (a cache slot or state offset out of
 *     range, an accept count out of range) are reported per sequence through the optional `err`
 *     array, and that sequence is left untouched.  No kernel traps.  The kernels that stage data
 *     through bulk copies wait for them with bounded waits (wait_polls below): a wait that gives
 *     up flags CV_SEQ_TIMEOUT for every sequence the block did not finish, and the kernel returns
 *     with its context intact.
 */
#ifndef CONVVERIFY_H
#define CONVVERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CV_API __attribute__((visibility("default")))
#else
#define CV_API
#endif

#define CV_ABI_VERSION 8
#define CV_MAX_T 128 /* draft tokens per verify call */

typedef enum cv_dtype {
    CV_F32 = 0,  /* IEEE binary32 */
    CV_BF16 = 1  /* bfloat16; arithmetic in fp32, outputs rounded to nearest even */
} cv_dtype;

/* cv_verify_args.state_dtype: the dtype of conv_state and the snapshots. */
#define CV_STATE_SAME 0 /* the dtype of x (a zero-initialised struct asks for no mixing) */
#define CV_STATE_F32 1  /* fp32 state with bf16 x */
#define CV_STATE_BF16 2 /* bf16 state with fp32 x */

typedef enum cv_window_layout {
    /* window element (s, t, c, k) at s*win_seq_stride + t*win_step_stride + c*win_ch_stride
       + k*win_col_stride: the [n_seq, T, dim, W-1] intermediates of [atlas-batched]. */
    CV_WINDOW_DENSE = 1,
    /* the deduplicated row of [sglang-46184]: element (s, t, c, k) at s*win_seq_stride
       + (t+k)*win_col_stride + c*win_ch_stride, i.e. one [dim, T+W-2] row per sequence whose
       column q holds input q+1 of [committed window, x_0 .. x_{T-1}].  win_step_stride must
       equal win_col_stride. */
    CV_WINDOW_DEDUP = 2,
    /* history-row state: no window buffer (window may be NULL; the win_* strides are ignored).
       The state row is the deduplicated row itself: the call reads the committed window at
       columns [o, o+W-1) of conv_state[slot][c] and then writes columns [0, T+W-2) of that row
       with [full[1 .. W-2], x_0 .. x_{T-1}], so snapshot t sits at columns [t, t+W-1).  The next
       call passes state_off[s] = accept_len[s] - 1 and no commit runs (a reading of the
       [sglang-46184] slot row together with its accepted-token state offset).  Needs
       state_cols >= T+W-2; columns at and above T+W-2 are not touched.  cv_conv_commit rejects
       this layout.  Only this layout accepts column-major state rows (state_col_stride != 1:
       [n_slots, state_cols, dim] storage seen as [n_slots, dim, state_cols], like the pool's
       axis-0 window layout of [sglang-46184]), with which the call reads W-1 columns and writes
       T+W-2 columns, each a contiguous run of channels. */
    CV_WINDOW_HISTORY = 3,
    /* recompute rollback ([memra-engine] ssm_conv_ring_rebuild_dc): no window buffer (window may
       be NULL; the win_* strides are ignored).  The verify writes the outputs only -- no
       snapshots, and conv_state is not written, so it keeps the pre-verify window.  The matching
       cv_conv_commit (same layout) then rebuilds the state from that window and the verify's x:
       conv_state[slot][c][k] = full[a+k], the value snapshot a-1 would hold. */
    CV_WINDOW_RECOMPUTE = 4
} cv_window_layout;

/* Status codes returned by the entry points. */
enum {
    CV_OK = 0,
    CV_ERR_NULL_ARGS = -1,    /* args pointer is NULL */
    CV_ERR_NULL_POINTER = -2, /* a required buffer pointer is NULL */
    CV_ERR_SHAPE = -3,        /* n_seq outside 0..65535, dim < 1, n_slots < 1, state_cols < W-1,
                                 or state_cols < T+W-2 in the history layout */
    CV_ERR_TOKENS = -4,       /* T outside 1..CV_MAX_T */
    CV_ERR_WIDTH = -5,        /* conv width outside 2..4 */
    CV_ERR_DTYPE = -6,        /* dtype not a cv_dtype */
    CV_ERR_HEAD_DIM = -7,     /* qk_channels > 0 and head_dim not a power of two in 8..256, or
                                 qk_channels not a multiple of head_dim, or qk_channels > dim */
    CV_ERR_LAYOUT = -8,       /* unknown layout, DEDUP with win_step_stride != win_col_stride,
                                 HISTORY passed to cv_conv_commit, or column-major state rows
                                 outside HISTORY */
    CV_ERR_STRIDE = -9,       /* a negative stride, or state rows that overlap (state_ch_stride <
                                 state_cols with dim > 1; column-major rows: state_ch_stride != 1
                                 or state_col_stride < dim) */
    CV_ERR_ALIAS = -10,       /* out or window has the same base address as x, conv_state or weight,
                                 or out and window share a base address */
    CV_ERR_LAUNCH = -11,      /* the CUDA launch failed (cudaGetLastError after the launch) */
    CV_ERR_SMEM = -12         /* the tile does not fit in shared memory for any block size */
};

/* Per-sequence bits written to err[s] (0 = fine or padded). */
#define CV_SEQ_BAD_SLOT 1   /* cache slot >= n_slots */
#define CV_SEQ_BAD_OFFSET 2 /* state offset < 0 or offset + W-1 > state_cols */
#define CV_SEQ_BAD_ACCEPT 4 /* accept count outside 1..T (commit only) */
#define CV_SEQ_TIMEOUT 8    /* a bounded wait for a bulk copy gave up: the sequence may be partly
                               written (every sequence whose data the block had not finished) */
#define CV_SEQ_BAD_SPAN 16  /* prefill: token span invalid or longer than max_seqlen; packed
                               verify / commit: draft span invalid or longer than T */
#define CV_SEQ_BAD_TREE 32  /* tree verify: a draft token's parent outside [-1, t) */

/*
 * cv_conv_verify -- [atlas-batched] fused multi-token verify, batched over sequences.
 *
 * For every sequence s with slot = cache_idx ? cache_idx[s] : s and slot >= 0, and every channel
 * c, let o = state_off ? state_off[s] : 0 and
 *     full = [conv_state[slot][c][o .. o+W-2], x[s][0][c], ..., x[s][T-1][c]]     (W-1+T values)
 * Then for every token t:
 *     acc   = bias[c] (or 0) + sum_{j=0}^{W-1} weight[c][j] * full[t+j]   fp32, bias first, taps in
 *                                                                         order, each product
 *                                                                         rounded (exact for bf16)
 *     y     = acc / (1 + exp(-acc))                                      SiLU [kda-mod]
 *     for c < qk_channels: y *= 1/sqrt(sum over c's head_dim group of y^2 + l2_eps)   [kda-mod]
 *     out[s][t][c] = y rounded once to dtype
 *                    (SiLU and the normalisation use fast hardware approximations: the outputs
 *                    match the exact expressions to within 1e-5 relative (+1e-7) in fp32 and
 *                    2 ulp in bf16, and are identical for every launch path and batch split)
 *     snapshot (s, t, c, k) = full[t+1+k], k < W-1      raw bit copy, dense or dedup layout
 * and finally conv_state[slot][c][0 .. W-2] = full[T .. T+W-2] (the committed window, equal to
 * snapshot T-1); state columns >= W-1 keep their values (packed rows wider than the window may be
 * written back whole with those columns' own bits, so nothing else may write them during the
 * call).  In the CV_WINDOW_HISTORY layout the
 * snapshots go into the state row instead (columns [0, T+W-2), see the layout) and no window
 * buffer is written; in the CV_WINDOW_RECOMPUTE layout neither snapshots nor the state are
 * written.  A sequence with slot < 0 is padding: its
 * out rows, window rows and every state slot are left untouched ([sglang-46184]).
 *
 * Arguments (all in cv_verify_args):
 *   n_seq, T, dim      sequences (0 = nothing to do), draft tokens 1..CV_MAX_T, channels >= 1
 *   width              conv width W in 2..4 (the window is held in registers)
 *   qk_channels        leading channels that are L2-normalised (0 = none); multiple of head_dim
 *   head_dim           L2 group size when qk_channels > 0: power of two, 8..256
 *   dtype              cv_dtype of x, out, weight and bias (and of conv_state and window unless
 *                      state_dtype says otherwise)
 *   l2_eps             added to the group's sum of squares inside the square root
 *   x                  [n_seq][T][dim] read-only; element (s,t,c) at s*x_seq_stride + t*x_tok_stride + c
 *                      (x may be a strided slice of a wider projection output)
 *   out                [n_seq][T][dim] write-only; (s,t,c) at s*out_seq_stride + t*out_tok_stride + c
 *   conv_state         [n_slots][dim][state_cols] read-modify-write in place;
 *                      (slot,c,k) at slot*state_slot_stride + c*state_ch_stride + k*state_col_stride
 *                      (state_col_stride 0 or 1: columns contiguous, state_ch_stride >= state_cols;
 *                      else only in CV_WINDOW_HISTORY, with state_ch_stride == 1 and
 *                      state_col_stride >= dim: column-major rows, else CV_ERR_STRIDE /
 *                      CV_ERR_LAYOUT)
 *   cache_idx          int32 [n_seq] device array or NULL (slot = s); negative = padded sequence
 *   state_off          int32 [n_seq] device array or NULL (0): column where the committed window is
 *                      read, the num_accept_tokens offset of [sglang-46184]
 *   weight             [dim][W] contiguous, read-only; weight[c][W-1] multiplies the newest input
 *   bias               [dim] read-only, or NULL
 *   window             snapshot buffer, write-only, laid out as window_layout says (NULL allowed
 *                      and ignored for CV_WINDOW_HISTORY and CV_WINDOW_RECOMPUTE)
 *   err                int32 [n_seq] device array or NULL: receives the CV_SEQ_* bits of each
 *                      sequence (0 for fine and for padded sequences).  On the pipelined path the
 *                      library clears it (an asynchronous memset on `stream`) before the kernel ORs
 *                      the bits in, since several blocks report for one sequence.
 *   wait_polls         limit of each unit's first wait for its bulk copies on the pipelined path
 *                      (path 3): 0 = the default (2^20 polls of mbarrier.try_wait, far beyond any
 *                      copy's latency), n > 0 = n polls, negative = no poll at all, so the wait
 *                      gives up at once.  Nonzero values exist to exercise the timeout path: the
 *                      block flags CV_SEQ_TIMEOUT for the unit's sequence and for those of every
 *                      later unit it owns, waits (with the default limit) for the copies it has in
 *                      flight, and returns; the other sequences are computed as usual.  Other paths
 *                      ignore it.
 *   state_dtype        CV_STATE_SAME, or the other dtype for conv_state and window (mixed dtypes,
 *                      [sglang-46184] "Accuracy Tests"): inputs are widened exactly for the
 *                      arithmetic; snapshots and state receive x converted to the state dtype
 *                      (exact widening bf16 -> fp32, or round to nearest even fp32 -> bf16 with any
 *                      NaN becoming the quiet NaN 0x7fc0).  Mixed calls take the pipelined kernel
 *                      (path 3) for T <= 8 with packed buffers, the general kernel otherwise.
 *   parent             int32 [n_seq][T] device array (row-major, contiguous) or NULL (a chain):
 *                      tree verify ([sglang-46184] "Scope": tree verify keeps dense windows).  Token
 *                      t's parent p in [-1, t) (-1: the committed window); its conv sees the
 *                      parent's window followed by x_t, and snapshot t is window(t) =
 *                      [window(p)[1 .. W-2], x_t].  The state is left on window(T-1).  The commit
 *                      restores the accepted path's last node: accept_len = its index + 1.  Needs
 *                      the dense layout and one dtype; a parent outside [-1, t) flags
 *                      CV_SEQ_BAD_TREE.
 *   cu_draft           int32 [n_seq + 1] device array or NULL: packed ragged drafts ([sglang-46184]
 *                      "Related upstream work": target verify on packed ragged tokens, the tile
 *                      store covering the packed rows).  Sequence s then owns rows
 *                      [cu_draft[s], cu_draft[s+1]) of x and out -- row r at r*x_tok_stride and
 *                      r*out_tok_stride; x_seq_stride and out_seq_stride are ignored -- and its T_s
 *                      rows are verified exactly as a verify of T_s tokens: T_s outputs, snapshots
 *                      t < T_s (dense steps >= T_s and dedup columns >= T_s+W-2 are not written),
 *                      and the state left on full[T_s .. T_s+W-2].  T is the largest T_s and sizes
 *                      the window buffer (dense [n_seq][T][dim][W-1], dedup [n_seq][dim][T+W-2],
 *                      history rows >= T+W-2).  T_s = 0 writes no output and no snapshot (the
 *                      state receives the committed window; in the history layout nothing is
 *                      written).  A span that is reversed, leaves [0, total_tokens) or holds more
 *                      than T rows flags CV_SEQ_BAD_SPAN and leaves the sequence untouched.  Chains
 *                      only: cu_draft with parent is CV_ERR_LAYOUT.  With packed 16-byte-aligned
 *                      buffers the pipelined kernel runs it (one dtype), otherwise the general one.
 *   total_tokens       rows of x and out with cu_draft (>= 0); x and out may be NULL when it is 0
 * Preconditions the library cannot check: distinct sequences use distinct slots; out and window do
 * not overlap themselves, each other, x, conv_state or weight.
 * Returns CV_OK after the launch is queued, or a negative CV_ERR_* code with nothing launched.
 */
typedef struct cv_verify_args {
    int32_t n_seq, T, dim, width, qk_channels, head_dim;
    int32_t dtype; /* cv_dtype */
    float l2_eps;
    const void *x;
    int64_t x_seq_stride, x_tok_stride;
    void *out;
    int64_t out_seq_stride, out_tok_stride;
    void *conv_state;
    int32_t n_slots, state_cols;
    int64_t state_slot_stride, state_ch_stride;
    const int32_t *cache_idx;
    const int32_t *state_off;
    const void *weight;
    const void *bias;
    void *window;
    int32_t window_layout; /* cv_window_layout */
    int32_t wait_polls;    /* limit of the bounded waits (see above); 0 = the default */
    int64_t win_seq_stride, win_step_stride, win_ch_stride, win_col_stride;
    int32_t *err;
    int32_t state_dtype; /* CV_STATE_* */
    const int32_t *parent;
    const int32_t *cu_draft; /* packed ragged drafts: int32 [n_seq + 1] device array, or NULL */
    int32_t total_tokens;    /* rows of x and out when cu_draft is given */
    int64_t state_col_stride; /* conv_state column stride; 0 or 1 = columns contiguous */
} cv_verify_args;

CV_API int cv_conv_verify(const cv_verify_args *args, void *stream);

/*
 * cv_conv_commit -- restore the state of the accepted prefix ([sglang-46184] "Motivation": the
 * window exists so the state can be rolled back to the accepted prefix; [kda-mod] decode_k:
 * snapshot t is the state after row t, which a partial accept rewinds to).
 *
 * For every sequence s with slot = cache_idx ? cache_idx[s] : s, slot >= 0, and a = accept_len[s]
 * read on the device (no host round trip), 1 <= a <= T:
 *     conv_state[slot][c][k] = snapshot (s, a-1, c, k)      for every c < dim, k < W-1
 * a = T rewrites the state with the value it already holds.  State columns >= W-1 keep their
 * values (packed rows wider than the window may be written back whole with those columns' own
 * bits, so nothing else may write them during the call).  A sequence whose a is out of range
 * gets CV_SEQ_BAD_ACCEPT in err[s] and is untouched.  Packed deduplicated rows are staged by a
 * bulk copy per block with a bounded wait (wait_polls, as in cv_verify_args; a timeout flags
 * CV_SEQ_TIMEOUT and leaves the block's channels unwritten); that kernel ORs its bits into err,
 * which the library clears first with an asynchronous memset on `stream`.  Rows laid out
 * transposed (win_ch_stride = 1, 16-byte-aligned columns) are read by plain loads of the accepted
 * columns alone.  The window must be the one the matching
 * cv_conv_verify wrote (same layout and strides).
 *
 * CV_WINDOW_RECOMPUTE: there is no window; x (with x_seq_stride, x_tok_stride, channel stride 1)
 * must be the input of the matching verify, unchanged since, and the state still holds the
 * pre-verify window in columns [0, W-1) (the verify leaves it alone in this layout).  With
 * full = [conv_state[slot][c][0 .. W-2], x[s][0][c] .. x[s][T-1][c]], the commit sets
 * conv_state[slot][c][k] = full[a+k] for k < W-1; each state row is read before it is written.
 * With cu_draft (the matching verify's packed spans) the accept count of sequence s must lie in
 * 1..T_s, an invalid span flags CV_SEQ_BAD_SPAN, and a sequence with T_s = 0 has nothing to commit
 * (skipped, err 0); in the recompute layout its x rows start at row cu_draft[s] (x_tok_stride;
 * total_tokens rows).
 * CV_WINDOW_HISTORY has nothing to commit and returns CV_ERR_LAYOUT.  dtype here is the dtype of
 * conv_state and window (with mixed dtypes, the state's); the recompute layout needs x in it too.
 */
typedef struct cv_commit_args {
    int32_t n_seq, T, dim, width;
    int32_t dtype; /* cv_dtype */
    int32_t n_slots;
    void *conv_state;
    int64_t state_slot_stride, state_ch_stride;
    int32_t state_cols;
    int32_t window_layout; /* cv_window_layout */
    const int32_t *cache_idx;
    const void *window;
    int64_t win_seq_stride, win_step_stride, win_ch_stride, win_col_stride;
    const int32_t *accept_len; /* int32 [n_seq] device array, required */
    int32_t *err;              /* int32 [n_seq] device array or NULL */
    /* CV_WINDOW_RECOMPUTE only (ignored otherwise): the verify's input [n_seq][T][dim] */
    const void *x;
    int64_t x_seq_stride, x_tok_stride;
    const int32_t *cu_draft; /* the matching verify's packed draft spans, or NULL */
    int32_t total_tokens;    /* rows of x (recompute layout) when cu_draft is given */
    int32_t wait_polls;      /* limit of the packed-dedup commit's bounded wait, as in cv_verify_args */
} cv_commit_args;

CV_API int cv_conv_commit(const cv_commit_args *args, void *stream);

/*
 * cv_conv_prefill -- the conv over whole prompts, packed back to back ([kda-mod], the layer's
 * prefill path: conv + SiLU over every prompt token, then the L2 normalisation of q|k).
 *
 * Sequence s owns tokens [cu_seqlens[s], cu_seqlens[s+1]) of x and out (L = its length, 0
 * allowed).  With slot = cache_idx ? cache_idx[s] : s and slot >= 0, for every channel c:
 *     full = [w0, x[cu_seqlens[s]][c], ..., x[cu_seqlens[s]+L-1][c]]      (W-1+L values)
 * where w0 = conv_state[slot][c][0 .. W-2] if has_initial_state[s] (or has_initial_state is
 * NULL), else W-1 zeros.  Token t's output is computed exactly as cv_conv_verify's output for
 * token t (conv, SiLU, the L2 normalisation of the q|k groups applied to the fp32 values, one
 * rounding), and afterwards conv_state[slot][c][0 .. W-2] = full[L .. L+W-2] (the last W-1
 * inputs, raw bits).  State columns >= W-1 are not touched; a sequence with slot < 0 touches
 * nothing.  Device-side problems go to err[s]: CV_SEQ_BAD_SLOT, or CV_SEQ_BAD_SPAN when the span
 * is reversed, leaves [0, total_tokens) or is longer than max_seqlen; that sequence is untouched.
 *
 * Arguments (all in cv_prefill_args):
 *   n_seq, dim, width, qk_channels, head_dim, dtype, l2_eps   as for cv_conv_verify
 *   total_tokens       rows of x and out (>= 0)
 *   max_seqlen         host-side bound on every L (sizes the grid), >= 0
 *   x                  [total_tokens][dim] read-only; token stride x_tok_stride, channel stride 1
 *   out                [total_tokens][dim] write-only; token stride out_tok_stride, channel stride 1
 *   cu_seqlens         int32 [n_seq + 1] device array (required)
 *   conv_state         [n_slots][dim][state_cols], column stride 1, read-modify-write
 *   cache_idx, has_initial_state, err   int32 [n_seq] device arrays or NULL
 *   weight, bias       [dim][W] and [dim] (bias may be NULL)
 * Returns CV_OK after the launch is queued, or a negative CV_ERR_* code with nothing launched.
 */
typedef struct cv_prefill_args {
    int32_t n_seq, dim, width, qk_channels, head_dim;
    int32_t dtype; /* cv_dtype */
    float l2_eps;
    int32_t total_tokens, max_seqlen;
    const void *x;
    int64_t x_tok_stride;
    void *out;
    int64_t out_tok_stride;
    const int32_t *cu_seqlens;
    void *conv_state;
    int32_t n_slots, state_cols;
    int64_t state_slot_stride, state_ch_stride;
    const int32_t *cache_idx;
    const int32_t *has_initial_state;
    const void *weight;
    const void *bias;
    int32_t *err;
} cv_prefill_args;

CV_API int cv_conv_prefill(const cv_prefill_args *args, void *stream);

/*
 * cv_verify_plan -- validate `args` exactly as cv_conv_verify does and report the launch it would
 * make, without touching the GPU.  grid = (grid_x, grid_y), block = threads, dynamic shared
 * memory = smem_bytes; a unit of work is channels_per_block channels of one sequence (one unit per
 * block, or, on the persistent paths 3 and 5, a stream of units per block).  path says
 * which kernel runs: 3 = persistent pipelined kernel (packed buffers and packed state rows, T a
 * compile-time constant; grid_y = 1 and each block walks (sequence, channel block) units),
 * 1 = packed buffers with T a compile-time constant (T <= 17 for bf16, <= 8 for fp32),
 * 2 = packed buffers, dense window, larger T in chunks of 8 tokens, 0 = the general kernel (any
 * strides), 5 = tree verify (parent given; persistent blocks of one or two warps walk (sequence,
 * 256 channels) units, staging each unit's committed windows, x rows and parents in one of `stages`
 * shared-memory buffers; grid_y = 1).  Host pointer `plan` must not be NULL.  Returns the same status
 * cv_conv_verify would return before launching.
 */
typedef struct cv_launch_plan {
    int32_t grid_x, grid_y, threads, smem_bytes, channels_per_block, path;
    int32_t stages; /* paths 3 and 5: unit buffers per block (loads in flight); 0 otherwise */
    int32_t token_groups; /* path 2: thread groups splitting the draft tokens (the block's y size); 1 otherwise */
} cv_launch_plan;

CV_API int cv_verify_plan(const cv_verify_args *args, cv_launch_plan *plan);

/* cv_status_string -- a static, NUL-terminated description of a status code (never NULL). */
CV_API const char *cv_status_string(int status);

/* cv_abi_version -- CV_ABI_VERSION of the built library. */
CV_API int cv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONVVERIFY_H */
