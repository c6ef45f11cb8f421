// C ABI of the verify/commit library: argument validation, launch planning and dispatch to the
// kernels.  Every check runs on the host before anything is launched; a failed check returns a
// negative status and launches nothing.
//
// Path selection for cv_conv_verify:
//   fast, static T  (path 1): packed, 16-byte aligned buffers, dim % 8 == 0, T <= the largest
//                             compiled static T (17 for bf16, 8 for fp32); either window layout.
//   fast, chunked   (path 2): the same buffers with a dense window and a larger T.
//   general         (path 0): everything else (any strides, any dim, dedup rows with a larger T).
//   pipelined       (path 3): path 1's buffers with packed state rows: persistent blocks walk
//                             (sequence, channel block) units and load each by bulk copy into
//                             double-buffered shared memory, two units ahead.  The history layout
//                             takes it when its state rows are the packed [dim][T+W-2] rows, and
//                             the general kernel otherwise.  Mixed dtypes (state and snapshots in
//                             the other dtype) take it for T <= 8, the general kernel otherwise.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "convverify.h"
#include "cv_launch.h"
#include "cv_verify_tree.cuh"  // tree_buffer_bytes

namespace {

constexpr int kFastThreads = 128;
constexpr int kFastThreadsMax = 256;   // the one-pass kernel's launch bound (threads x token groups)
constexpr int kMaxTokenGroups = 4;     // token groups of the chunked one-pass kernel, at most
constexpr int kFastMinWarpsPerSM = 8;  // below this the chunked one-pass kernel splits the tokens
constexpr int kPipeThreads = 128;
constexpr long long kFastRowsMaxBytes = 64 * 1024;  // staged wide state rows of a one-pass block
// blocks per SM the pipelined kernel's launch bounds provide registers for
constexpr int pipe_blocks_per_sm(int cpt, int T) { return (cpt == 4 && T <= 8) ? 4 : 2; }
constexpr int kSmemPerBlockReserved = 1024;
constexpr int kMinThreads = 32;
constexpr int kGenericSmemBudget = 96 * 1024;
constexpr int kTreeWarps = 2;         // tree verify: warps per block (tokens split among them)
constexpr int kTreeBlocksPerSM = 10;  // tree verify: resident blocks per SM at most
// commit block sizes per mode (measured on the steps they end): small blocks start beside the
// verify's resident blocks while it drains
constexpr int kCommitDenseThreads = 64;      // packed dense snapshot -> packed state (16-byte copies)
constexpr int kCommitElementThreads = 32;    // element by element
constexpr int kCommitWideThreads = 32;       // packed dense snapshot -> packed rows wider than the window
constexpr int kCommitRecomputeThreads = 64;  // recompute rollback
// dedup commit: 256 channels per block (small blocks fit beside the verify's resident blocks, so
// more of them start, under programmatic dependent launch, while the verify drains)
constexpr int kCommitRowThreads = 32;
constexpr int kCommitColThreads = 64;  // transposed dedup rows: 512 channels per block (measured: 4.4 us alone against 5.1 with 128)
// the same after a verify of packed ragged drafts, whose uneven tail leaves room for more, smaller
// blocks to start while it drains (measured, 128 drafts of 1..16 tokens: step 32.0 us against 33.1)
constexpr int kCommitColThreadsPacked = 32;
// the pipelined kernel lists the active sequences (or packed drafts' chunks) in shared memory up to
// this many entries
constexpr int kCompactMaxEntries = 1024;
constexpr int kPrefillMaxChunk = 128;  // tokens per prefill block, at most / at least (multiples of
constexpr int kPrefillMinChunk = 32;   // the kernel's 8-token batch, and >= W-1)
constexpr int kPrefillRing = 4;        // batches of staged x rows per prefill thread (as the kernel's)

// The device the launch plans size for: SM count (the persistent grids), shared memory per SM
// (residency) and per block (opt-in maximum), queried once per device and cached.  Without a
// usable device (cv_verify_plan on a host without a GPU) the plans are made for a GB300: 152 SMs,
// 228 KB per SM, 227 KB per block.
struct DeviceLimits {
    int sms, smem_per_sm, smem_per_block;
};
DeviceLimits device_limits() {
    constexpr DeviceLimits kGB300{152, 232448, 227 * 1024};
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached[kMaxDevices][3];  // zero until queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();  // clear the error the failed query recorded
        return kGB300;
    }
    if (dev < kMaxDevices && cached[dev][0].load(std::memory_order_acquire) > 0)
        return {cached[dev][0].load(std::memory_order_relaxed), cached[dev][1].load(std::memory_order_relaxed),
                cached[dev][2].load(std::memory_order_relaxed)};
    DeviceLimits d{0, 0, 0};
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        d.sms < 1) {
        cudaGetLastError();
        return kGB300;
    }
    if (dev < kMaxDevices) {
        cached[dev][1].store(d.smem_per_sm, std::memory_order_relaxed);
        cached[dev][2].store(d.smem_per_block, std::memory_order_relaxed);
        cached[dev][0].store(d.sms, std::memory_order_release);
    }
    return d;
}

// Tokens per unit of the pipelined kernel for packed drafts: the whole draft when T <= 8, else
// chunks of 8 (so any T runs with the registers of an 8-token unit); T otherwise.
constexpr int kVarlenChunk = 8;
int pipe_tokens(const cv_verify_args *a) {
    return a->cu_draft && a->T > kVarlenChunk ? kVarlenChunk : a->T;
}
// entries of the pipelined kernel's work list: sequences, or (packed drafts) chunks of them
long long pipe_list_len(const cv_verify_args *a) {
    const int ts = pipe_tokens(a);
    return (long long)a->n_seq * ((a->T + ts - 1) / ts);
}
// the list of active sequences (padded ones dropped; packed drafts as chunks ordered by size)
bool pipe_compacts(const cv_verify_args *a) {
    return (a->cache_idx != nullptr || a->cu_draft != nullptr) && pipe_list_len(a) <= kCompactMaxEntries;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride16(long long stride_elems, int esize) { return ((stride_elems * esize) & 15) == 0; }
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

const cvk::KernelSet &kernel_set(int dtype, int width) {
    if (dtype == CV_BF16) {
        if (width == 2) return cvk::kernels_bf16_w2();
        if (width == 3) return cvk::kernels_bf16_w3();
        return cvk::kernels_bf16_w4();
    }
    if (width == 2) return cvk::kernels_f32_w2();
    if (width == 3) return cvk::kernels_f32_w3();
    return cvk::kernels_f32_w4();
}

const cvk::VarlenSet &varlen_set(int dtype, int width) {
    if (dtype == CV_BF16) {
        if (width == 2) return cvk::varlen_bf16_w2();
        if (width == 3) return cvk::varlen_bf16_w3();
        return cvk::varlen_bf16_w4();
    }
    if (width == 2) return cvk::varlen_f32_w2();
    if (width == 3) return cvk::varlen_f32_w3();
    return cvk::varlen_f32_w4();
}

// State columns not contiguous (state_col_stride other than 0 or 1).
bool state_col_major(const cv_verify_args *a) { return a->state_col_stride > 1; }

int check_verify(const cv_verify_args *a) {
    if (!a) return CV_ERR_NULL_ARGS;
    if (a->dtype != CV_F32 && a->dtype != CV_BF16) return CV_ERR_DTYPE;
    if (a->state_dtype != CV_STATE_SAME && a->state_dtype != CV_STATE_F32 && a->state_dtype != CV_STATE_BF16)
        return CV_ERR_DTYPE;
    if (a->width < 2 || a->width > 4) return CV_ERR_WIDTH;
    if (a->T < 1 || a->T > CV_MAX_T) return CV_ERR_TOKENS;
    if (a->n_seq < 0 || a->n_seq > 65535 || a->dim < 1 || a->n_slots < 1 || a->state_cols < a->width - 1)
        return CV_ERR_SHAPE;
    const bool hist = a->window_layout == CV_WINDOW_HISTORY;
    const bool recomp = a->window_layout == CV_WINDOW_RECOMPUTE;
    const bool nowin = hist || recomp;  // no window buffer
    if (a->window_layout != CV_WINDOW_DENSE && a->window_layout != CV_WINDOW_DEDUP && !nowin) return CV_ERR_LAYOUT;
    if (a->window_layout == CV_WINDOW_DEDUP && a->win_step_stride != a->win_col_stride) return CV_ERR_LAYOUT;
    if (hist && a->state_cols < a->T + a->width - 2) return CV_ERR_SHAPE;
    // tree verify: dense snapshots only, one dtype; packed drafts are chains
    if (a->parent && a->window_layout != CV_WINDOW_DENSE) return CV_ERR_LAYOUT;
    if (a->parent && a->cu_draft) return CV_ERR_LAYOUT;
    if (a->cu_draft && a->total_tokens < 0) return CV_ERR_SHAPE;
    if (a->parent && a->state_dtype != CV_STATE_SAME && a->state_dtype - 1 != a->dtype) return CV_ERR_DTYPE;
    if (a->qk_channels < 0 || a->qk_channels > a->dim) return CV_ERR_HEAD_DIM;
    if (a->qk_channels > 0 && (!pow2(a->head_dim) || a->head_dim < 8 || a->head_dim > 256 ||
                               a->qk_channels % a->head_dim != 0))
        return CV_ERR_HEAD_DIM;
    if (a->x_seq_stride < 0 || a->x_tok_stride < 0 || a->out_seq_stride < 0 || a->out_tok_stride < 0 ||
        a->state_slot_stride < 0 || a->state_ch_stride < 0)
        return CV_ERR_STRIDE;
    if (!nowin && (a->win_seq_stride < 0 || a->win_step_stride < 0 || a->win_ch_stride < 0 || a->win_col_stride < 0))
        return CV_ERR_STRIDE;
    if (a->state_col_stride < 0) return CV_ERR_STRIDE;
    if (state_col_major(a)) {
        // column-major rows: the commit-free history layout only
        if (!hist) return CV_ERR_LAYOUT;
        if (a->state_ch_stride != 1 || a->state_col_stride < a->dim) return CV_ERR_STRIDE;
    } else if (a->dim > 1 && a->state_ch_stride < a->state_cols) {
        return CV_ERR_STRIDE;
    }
    // (packed drafts with no rows at all need no x or out)
    const bool rows = !a->cu_draft || a->total_tokens > 0;
    if (a->n_seq > 0 && ((rows && (!a->x || !a->out)) || !a->conv_state || !a->weight || (!nowin && !a->window)))
        return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0) {
        const void *outs[2] = {a->out, nowin ? nullptr : a->window};
        const void *ins[3] = {a->x, a->conv_state, a->weight};
        for (const void *o : outs)
            for (const void *i : ins)
                if (o && o == i) return CV_ERR_ALIAS;
        if (!nowin && a->out == a->window) return CV_ERR_ALIAS;
    }
    return CV_OK;
}

// x, out, taps and bias allow 16-byte vectors and bulk copies of whole channel blocks.
bool io_packed(const cv_verify_args *a, int esize) {
    if (a->dim % 8 != 0) return false;
    // (packed drafts ignore the sequence strides)
    const bool vl = a->cu_draft != nullptr;
    if (!aligned16(a->x) || !(vl || stride16(a->x_seq_stride, esize)) || !stride16(a->x_tok_stride, esize)) return false;
    if (!aligned16(a->out) || !(vl || stride16(a->out_seq_stride, esize)) || !stride16(a->out_tok_stride, esize))
        return false;
    return aligned16(a->weight) && (!a->bias || aligned16(a->bias));
}

// (esize: bytes of an x element; ssize: of a state and snapshot element)
bool fast_eligible(const cv_verify_args *a, int esize, int ssize, int max_static_t, int tokens) {
    const int R = a->width - 1;
    const long long Q = a->T + R - 1;
    if (a->window_layout == CV_WINDOW_HISTORY || a->window_layout == CV_WINDOW_RECOMPUTE || !io_packed(a, esize))
        return false;
    if (!aligned16(a->window) || !stride16(a->win_seq_stride, ssize) || a->win_col_stride != 1) return false;
    if (a->window_layout == CV_WINDOW_DEDUP) return a->win_ch_stride == Q && tokens <= max_static_t;
    return a->win_ch_stride == R && stride16(a->win_step_stride, ssize);
}

// Deduplicated rows laid out transposed (channel stride 1, every column a 16-byte-aligned run of
// channels), which only the pipelined kernel stores by bulk copies (one per column).
bool dedup_transposed_ok(const cv_verify_args *a, int ssize, int max_static_t) {
    return a->window_layout == CV_WINDOW_DEDUP && a->dim % 8 == 0 && a->win_ch_stride == 1 &&
           a->win_col_stride >= a->dim && aligned16(a->window) && stride16(a->win_seq_stride, ssize) &&
           stride16(a->win_col_stride, ssize) && pipe_tokens(a) <= max_static_t;
}

// Halve a block (down to 32 threads) while the launch would have fewer than two blocks per SM and
// the smaller block still holds whole L2 groups: small batches then still fill the GPU.
int shrink_for_parallelism(int threads, int cpt, const cv_verify_args *a, int sms) {
    const int min_bc = a->qk_channels > 0 ? a->head_dim : 8;
    auto units = [&](int t) { return (long long)a->n_seq * ((a->dim + (long long)cpt * t - 1) / ((long long)cpt * t)); };
    while (threads > 32 && units(threads) < 2LL * sms && cpt * (threads / 2) >= min_bc) threads /= 2;
    return threads;
}

// Units (sequence x channel block) per block of the pipelined kernel's persistent grid, for the
// block size it would use (an upper bound on its shared-memory residency of 4 blocks per SM).
double units_per_pipe_block(const cv_verify_args *a, int cpt, int sms) {
    int threads = kPipeThreads;
    while (threads > 32 && cpt * (threads / 2) >= a->dim) threads /= 2;
    while (a->qk_channels > 0 && cpt * threads < a->head_dim) threads *= 2;
    threads = shrink_for_parallelism(threads, cpt, a, sms);
    const long long bc = (long long)cpt * threads;
    const long long nblk = (a->dim + bc - 1) / bc;
    const long long units = (long long)a->n_seq * nblk;
    long long g = (long long)sms * pipe_blocks_per_sm(cpt, pipe_tokens(a));
    if (g >= nblk) g = g / nblk * nblk;
    if (g > units) g = units;
    return g > 0 ? (double)units / (double)g : 0.0;
}

bool state_packed(const void *state, long long slot_stride, long long ch_stride, int width, int esize) {
    return aligned16(state) && stride16(slot_stride, esize) && ch_stride == width - 1;
}

// Packed state rows wider than the window (read at a state offset): [dim][state_cols] per slot,
// 16-byte aligned.  The one-pass kernel then stages a block's rows whole in shared memory and
// stores them back whole, when they take at most kFastRowsMaxBytes.
bool fast_rows_staged(const cv_verify_args *a, int ssize, long long bc) {
    return !state_packed(a->conv_state, a->state_slot_stride, a->state_ch_stride, a->width, ssize) &&
           aligned16(a->conv_state) && stride16(a->state_slot_stride, ssize) && a->state_ch_stride == a->state_cols &&
           bc * a->state_cols * ssize <= kFastRowsMaxBytes;
}

// Validates verify arguments; on success fills the launch plan.
// dtype of conv_state and the snapshots
int state_dtype_of(const cv_verify_args *a) { return a->state_dtype == CV_STATE_SAME ? a->dtype : a->state_dtype - 1; }
bool mixed_dtypes(const cv_verify_args *a) { return state_dtype_of(a) != a->dtype; }

int plan_verify(const cv_verify_args *a, cv_launch_plan *pl) {
    const int rc = check_verify(a);
    if (rc != CV_OK) return rc;
    const int esize = a->dtype == CV_BF16 ? 2 : 4;
    const bool mixed = mixed_dtypes(a);
    const int R = a->width - 1;
    const DeviceLimits lim = device_limits();
    std::memset(pl, 0, sizeof *pl);
    pl->token_groups = 1;
    if (a->parent) {
        // tree verify: its own persistent kernel of kTreeWarps-warp blocks walking (sequence,
        // kTreeChannels channels) units; two unit buffers (the next unit loads while this one
        // computes) when they fit, else one; a grid of kTreeBlocksPerSM blocks per SM at most (as
        // shared memory allows), a multiple of the channel-block count so that a block keeps its taps
        const long long buf = cvk::tree_buffer_bytes(a->T, a->width, esize);
        const int nbuf = 2 * buf <= lim.smem_per_block ? 2 : 1;
        if (buf > lim.smem_per_block) return CV_ERR_SMEM;
        int per_sm = (int)(lim.smem_per_sm / (nbuf * buf + kSmemPerBlockReserved));
        if (per_sm > kTreeBlocksPerSM) per_sm = kTreeBlocksPerSM;
        if (per_sm < 1) per_sm = 1;
        const long long nblk = (a->dim + cvk::kTreeChannels - 1) / cvk::kTreeChannels;
        const long long units = (long long)a->n_seq * nblk;
        long long g = (long long)lim.sms * per_sm;
        if (g >= nblk) g = g / nblk * nblk;
        if (g > units) g = units;
        pl->threads = 32 * (a->T < kTreeWarps ? a->T : kTreeWarps);
        pl->channels_per_block = cvk::kTreeChannels;
        pl->smem_bytes = (int)(nbuf * buf);
        pl->stages = nbuf;
        pl->path = 5;
        pl->grid_x = (int)(g > 0 ? g : 1);
        pl->grid_y = 1;
        return CV_OK;
    }
    const int min_threads =
        (a->qk_channels > 0 && a->head_dim / 8 > kMinThreads) ? a->head_dim / 8 : kMinThreads;
    const cvk::KernelSet &ks = kernel_set(a->dtype, a->width);
    std::memset(pl, 0, sizeof *pl);
    pl->token_groups = 1;

    const bool hist = a->window_layout == CV_WINDOW_HISTORY;
    const bool recomp = a->window_layout == CV_WINDOW_RECOMPUTE;
    const int ssize = state_dtype_of(a) == CV_BF16 ? 2 : 4;
    const bool fast = fast_eligible(a, esize, ssize, ks.max_static_t, pipe_tokens(a));
    const int cpt = (a->qk_channels > 0 && a->head_dim / 4 > 32) ? 8 : 4;
    // the pipelined kernel stages packed state rows whole (state_ch_stride == state_cols): the
    // committed windows of [dim][W-1] rows, or wider rows read at an offset; the history layout
    // needs rows of exactly T+W-2 columns
    const bool hist_t = hist && state_col_major(a);  // column-major history rows
    const bool rows_packed = hist_t ? a->dim % 8 == 0 && aligned16(a->conv_state) &&
                                          stride16(a->state_slot_stride, ssize) && stride16(a->state_col_stride, ssize)
                                    : aligned16(a->conv_state) && stride16(a->state_slot_stride, ssize) &&
                                          a->state_ch_stride == a->state_cols;
    const bool varlen = a->cu_draft != nullptr;
    const int ts = pipe_tokens(a);             // tokens per unit
    const bool chunked = varlen && a->T > ts;  // packed drafts cut into chunks
    const bool dedup_t = dedup_transposed_ok(a, ssize, ks.max_static_t);
    // (mixed dtypes: compiled for T <= kMaxMixedT; packed drafts: one dtype, and the chunks of a
    // longer draft need the work list and no history rows)
    bool pipe_ok = (!mixed || a->T <= cvk::kMaxMixedT) && !(mixed && varlen) && io_packed(a, esize) &&
                   ts <= ks.max_static_t && rows_packed &&
                   (hist ? (hist_t || a->state_cols == a->T + R - 1) : (recomp || fast || dedup_t)) &&
                   !(chunked && (hist || !pipe_compacts(a)));
    const bool wide = !hist && a->state_cols != R;
    // The pipeline pays for its prologue only when every block walks several units; with fewer the
    // one-pass kernel wins (measured: 8 x 17 tokens x 8192 channels, 2 units per block, 6.8 us
    // one-pass against 9.4 pipelined; 4 x 4 x 4096, 1 unit per block, 4.0 against 4.0 and a shorter
    // step), from 3 units per block the pipeline does (the 128 x 8 x 10240 benchmark: 3.8).  Wide
    // rows cost the one-pass kernel whole-row reads and element stores of the window, so for them
    // the pipeline wins from 2 units per block.  (Mixed dtypes have no one-pass kernel.)
    if (pipe_ok && fast && !mixed && !varlen && units_per_pipe_block(a, cpt, lim.sms) < (wide ? 2.0 : 3.0))
        pipe_ok = false;
    if (pipe_ok) {
        auto part = [](long long b) { return (b + 127) / 128 * 128; };
        int threads = kPipeThreads;
        while (threads > 32 && cpt * (threads / 2) >= a->dim) threads /= 2;
        while (a->qk_channels > 0 && cpt * threads < a->head_dim) threads *= 2;
        threads = shrink_for_parallelism(threads, cpt, a, lim.sms);
        const long long bc = (long long)cpt * threads;
        const long long Q = ts + R - 1;
        // two stages (x rows -- with a halo or tail of W-1 more for chunks of packed drafts --
        // + committed windows, or whole history rows) and two image buffers (dedup row + committed
        // windows, or the history row alone; none for the recompute rollback), the state parts in
        // the state's dtype; 2 mbarriers, 2 slots, 2 offsets
        const long long stage = part((long long)(ts + (chunked ? R : 0)) * bc * esize) +
                                part((long long)(hist_t ? R : a->state_cols) * bc * ssize);
        // (mixed dtypes and packed drafts store the committed windows straight from registers: no
        // state image)
        long long image =
            (hist || recomp || ((mixed || varlen) && !wide)) ? 0 : part((wide ? a->state_cols : R) * bc * ssize);
        if (a->window_layout == CV_WINDOW_DEDUP || hist) image += part(Q * bc * ssize);
        const long long smem = 2 * stage + 2 * image + cvk::kPipeInfoBytes +
                               (pipe_compacts(a) ? 4LL * cvk::pipe_aux_ints(varlen, ts) + (varlen ? 4LL : 12LL) * pipe_list_len(a) : 0);
        int per_sm = (int)(lim.smem_per_sm / (smem + kSmemPerBlockReserved));
        if (per_sm > pipe_blocks_per_sm(cpt, ts)) per_sm = pipe_blocks_per_sm(cpt, ts);
        const int nst = (smem <= lim.smem_per_block && per_sm >= 1) ? 2 : 0;
        if (nst > 0) {
            const long long nblk = (a->dim + bc - 1) / bc;
            const long long units = (long long)a->n_seq * nblk;
            // a multiple of the channel-block count keeps each block on one channel block
            long long g = (long long)lim.sms * per_sm;
            if (g >= nblk) g = g / nblk * nblk;
            if (g > units) g = units;
            pl->threads = threads;
            pl->channels_per_block = (int)bc;
            pl->smem_bytes = (int)smem;
            pl->path = 3;
            pl->stages = nst;
            pl->grid_x = (int)(g > 0 ? g : 1);
            pl->grid_y = 1;
            return CV_OK;
        }
    }
    if (fast && !mixed && !varlen) {
        // 4 channels per thread (twice the threads of 8) unless an L2 group would span more than a warp
        int threads = kFastThreads;
        while (threads > 32 && cpt * (threads / 2) >= a->dim) threads /= 2;
        while (a->qk_channels > 0 && cpt * threads < a->head_dim) threads *= 2;
        threads = shrink_for_parallelism(threads, cpt, a, lim.sms);
        const long long bc = (long long)cpt * threads;
        // committed-window image, or the staged wide rows
        long long smem = bc * (fast_rows_staged(a, ssize, bc) ? a->state_cols : R) * esize;
        if (a->window_layout == CV_WINDOW_DEDUP) smem += bc * (a->T + R - 1) * esize;
        // Small dense batches: split the draft tokens among thread groups (the chunked kernel, the
        // block's y dimension) while the launch would hold fewer than kFastMinWarpsPerSM warps per
        // SM, each group keeping at least W-1 tokens (its first W-1 inputs are the x rows before it)
        int groups = 1;
        if (a->window_layout == CV_WINDOW_DENSE) {
            const long long warps = (long long)a->n_seq * ((a->dim + bc - 1) / bc) * ((threads + 31) / 32);
            while (groups < kMaxTokenGroups && threads * groups * 2 <= kFastThreadsMax &&
                   warps * groups < (long long)kFastMinWarpsPerSM * lim.sms && (a->T + 2 * groups - 1) / (2 * groups) >= R)
                groups *= 2;
        }
        pl->threads = threads;
        pl->channels_per_block = (int)bc;
        pl->smem_bytes = (int)smem;
        pl->path = (a->T <= ks.max_static_t && groups == 1) ? 1 : 2;
        pl->token_groups = groups;
    } else {
        // (with mixed dtypes the tile holds fp32 bits)
        const int tsize = mixed ? 4 : esize;
        const int rows = a->T + a->width - 1;
        const int pad = 16 / tsize;  // one 16-byte vector of padding per tile row
        int threads = 128;
        while (threads > min_threads && 8 * (threads / 2) >= a->dim) threads /= 2;
        long long smem = (long long)rows * (8 * threads + pad) * tsize;
        while (smem > kGenericSmemBudget && threads > min_threads) {
            threads /= 2;
            smem = (long long)rows * (8 * threads + pad) * tsize;
        }
        if (smem > lim.smem_per_block) return CV_ERR_SMEM;
        pl->threads = threads;
        pl->channels_per_block = 8 * threads;
        pl->smem_bytes = (int)smem;
        pl->path = 0;
    }
    pl->grid_x = (a->dim + pl->channels_per_block - 1) / pl->channels_per_block;
    pl->grid_y = a->n_seq;
    return CV_OK;
}

// Launch with programmatic stream serialization: the kernel may be scheduled while the previous
// grid in the stream finishes; every kernel waits (griddepcontrol.wait) for that grid's completion
// before its first global-memory access, so the order of the stream's work is kept.
template <typename P>
cudaError_t launch_pdl(void (*kernel)(P), dim3 grid, dim3 block, int smem, cudaStream_t stream, const P &p) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    std::memset(attr, 0, sizeof attr);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Opt a kernel into more than 48 KB of dynamic shared memory (once per kernel and device).
cudaError_t ensure_smem(const void *kernel, int bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    static std::atomic<unsigned long long> done_cache[64][4];  // tiny open-addressing cache
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long key = reinterpret_cast<uintptr_t>(kernel) ^ ((unsigned long long)dev << 56);
    const unsigned h = (unsigned)((key >> 4) * 0x9E3779B1u) & 63u;
    for (auto &slot : done_cache[h])
        if (slot.load(std::memory_order_relaxed) == key) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, device_limits().smem_per_block);
    if (e != cudaSuccess) return e;
    for (auto &slot : done_cache[h]) {
        unsigned long long z = 0;
        if (slot.compare_exchange_strong(z, key)) break;
    }
    return cudaSuccess;
}

int launch_verify(const cv_verify_args *a, const cv_launch_plan &pl, cudaStream_t stream) {
    const int esize = a->dtype == CV_BF16 ? 2 : 4;
    cvk::VerifyParams p;
    std::memset(&p, 0, sizeof p);
    p.x = a->x;
    p.x_seq = a->x_seq_stride;
    p.x_tok = a->x_tok_stride;
    p.out = a->out;
    p.out_seq = a->out_seq_stride;
    p.out_tok = a->out_tok_stride;
    p.state = a->conv_state;
    p.st_slot = a->state_slot_stride;
    p.st_ch = a->state_ch_stride;
    p.st_col = state_col_major(a) ? a->state_col_stride : 1;
    p.cache_idx = a->cache_idx;
    p.state_off = a->state_off;
    p.weight = a->weight;
    p.bias = a->bias;
    p.win = a->window;
    p.dedup = a->window_layout == CV_WINDOW_DEDUP;
    p.dedup_t = pl.path == 3 && dedup_transposed_ok(a, state_dtype_of(a) == CV_BF16 ? 2 : 4,
                                                    kernel_set(a->dtype, a->width).max_static_t);
    p.hist = a->window_layout == CV_WINDOW_HISTORY;
    p.recomp = a->window_layout == CV_WINDOW_RECOMPUTE;
    p.parent = a->parent;
    p.compact = pl.path == 3 && pipe_compacts(a);
    if (p.hist || p.recomp) p.win = nullptr;
    p.w_seq = a->win_seq_stride;
    p.w_step = p.dedup ? a->win_col_stride : a->win_step_stride;
    p.w_ch = a->win_ch_stride;
    p.w_col = a->win_col_stride;
    p.err = a->err;
    p.wait_polls = a->wait_polls;
    p.cu_draft = a->cu_draft;
    p.total_tokens = a->total_tokens;
    p.n_seq = a->n_seq;
    p.T = a->T;
    p.dim = a->dim;
    p.n_slots = a->n_slots;
    p.state_cols = a->state_cols;
    p.qk_channels = a->qk_channels;
    p.head_dim = a->qk_channels > 0 ? a->head_dim : 8;
    const bool mixed = mixed_dtypes(a);
    const int ssize = state_dtype_of(a) == CV_BF16 ? 2 : 4;
    p.pitch = pl.channels_per_block + 16 / (mixed ? 4 : esize);
    p.eps = a->l2_eps;
    const bool vl = a->cu_draft != nullptr;  // (packed drafts ignore the sequence strides)
    p.x_vec = aligned16(a->x) && (vl || stride16(a->x_seq_stride, esize)) && stride16(a->x_tok_stride, esize);
    p.out_vec = aligned16(a->out) && (vl || stride16(a->out_seq_stride, esize)) && stride16(a->out_tok_stride, esize);
    p.st_vec = !state_col_major(a) &&
               state_packed(a->conv_state, a->state_slot_stride, a->state_ch_stride, a->width, ssize);
    p.st_rows = (pl.path == 1 || pl.path == 2) && fast_rows_staged(a, ssize, pl.channels_per_block);
    p.w_vec = aligned16(a->weight);
    p.b_vec = a->bias ? aligned16(a->bias) : 0;
    if (pl.path == 5) {
        // tree verify: pitch = unit buffers (1 or 2); st_vec -> packed 16-byte dense snapshot runs of
        // 8 channels x (W-1) columns; st_packed -> the committed windows read as 16-byte runs
        p.pitch = pl.stages;
        p.st_vec = a->dim % 8 == 0 && aligned16(a->window) && a->win_ch_stride == a->width - 1 &&
                   a->win_col_stride == 1 && stride16(a->win_seq_stride, esize) && stride16(a->win_step_stride, esize);
        p.st_packed = aligned16(a->conv_state) && stride16(a->state_slot_stride, esize) &&
                      a->state_ch_stride == a->width - 1 && a->state_cols == a->width - 1;
    }

    const cvk::KernelSet &ks = kernel_set(a->dtype, a->width);
    const int ci = pl.channels_per_block / pl.threads == 8 ? 1 : 0;
    cvk::VerifyKernel k = pl.path == 0   ? (mixed ? ks.generic_mixed : ks.generic)
                          : pl.path == 1 ? ks.fast[ci][a->T]
                          : pl.path == 2 ? ks.fast[ci][0]
                          : pl.path == 3 ? (mixed ? ks.pipe_mixed[ci][a->T]
                                            : a->cu_draft ? varlen_set(a->dtype, a->width).pipe[ci][pipe_tokens(a)]
                                                          : ks.pipe[ci][a->T])
                                         : ks.tree;
    if (ensure_smem(reinterpret_cast<const void *>(k), pl.smem_bytes) != cudaSuccess) return CV_ERR_LAUNCH;
    // the pipelined kernel ORs the per-sequence bits into err (several blocks share a sequence)
    if (pl.path == 3 && a->err && cudaMemsetAsync(a->err, 0, sizeof(int32_t) * (size_t)a->n_seq, stream) != cudaSuccess)
        return CV_ERR_LAUNCH;
    if (launch_pdl(k, dim3(pl.grid_x, pl.grid_y), dim3(pl.threads, pl.token_groups > 1 ? pl.token_groups : 1),
                   pl.smem_bytes, stream, p) != cudaSuccess)
        return CV_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
}

int check_commit(const cv_commit_args *a) {
    if (!a) return CV_ERR_NULL_ARGS;
    if (a->dtype != CV_F32 && a->dtype != CV_BF16) return CV_ERR_DTYPE;
    if (a->width < 2 || a->width > 4) return CV_ERR_WIDTH;
    if (a->T < 1 || a->T > CV_MAX_T) return CV_ERR_TOKENS;
    if (a->n_seq < 0 || a->n_seq > 65535 || a->dim < 1 || a->n_slots < 1 || a->state_cols < a->width - 1)
        return CV_ERR_SHAPE;
    // (the history layout has nothing to commit: the next verify reads at accept_len - 1)
    const bool recomp = a->window_layout == CV_WINDOW_RECOMPUTE;
    if (a->window_layout != CV_WINDOW_DENSE && a->window_layout != CV_WINDOW_DEDUP && !recomp) return CV_ERR_LAYOUT;
    if (a->window_layout == CV_WINDOW_DEDUP && a->win_step_stride != a->win_col_stride) return CV_ERR_LAYOUT;
    if (a->state_slot_stride < 0 || a->state_ch_stride < 0) return CV_ERR_STRIDE;
    if (!recomp && (a->win_seq_stride < 0 || a->win_step_stride < 0 || a->win_ch_stride < 0 || a->win_col_stride < 0))
        return CV_ERR_STRIDE;
    if (recomp && (a->x_seq_stride < 0 || a->x_tok_stride < 0)) return CV_ERR_STRIDE;
    if (a->cu_draft && a->total_tokens < 0) return CV_ERR_SHAPE;
    if (a->dim > 1 && a->state_ch_stride < a->state_cols) return CV_ERR_STRIDE;
    if (a->n_seq > 0 && (!a->conv_state || !a->accept_len)) return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0 && (recomp ? (!a->x && !(a->cu_draft && a->total_tokens == 0)) : !a->window))
        return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0 && (recomp ? a->conv_state == a->x : a->conv_state == a->window)) return CV_ERR_ALIAS;
    return CV_OK;
}

int launch_commit(const cv_commit_args *a, cudaStream_t stream) {
    const int esize = a->dtype == CV_BF16 ? 2 : 4;
    const int R = a->width - 1;
    const long long Q = a->T + R - 1;
    cvk::CommitParams p;
    std::memset(&p, 0, sizeof p);
    p.state = a->conv_state;
    p.st_slot = a->state_slot_stride;
    p.st_ch = a->state_ch_stride;
    p.cache_idx = a->cache_idx;
    p.win = a->window;
    p.w_seq = a->win_seq_stride;
    p.w_step = a->window_layout == CV_WINDOW_DEDUP ? a->win_col_stride : a->win_step_stride;
    p.w_ch = a->win_ch_stride;
    p.w_col = a->win_col_stride;
    p.accept_len = a->accept_len;
    p.err = a->err;
    p.wait_polls = a->wait_polls;
    p.cu_draft = a->cu_draft;
    p.total_tokens = a->total_tokens;
    p.n_seq = a->n_seq;
    p.T = a->T;
    p.dim = a->dim;
    p.n_slots = a->n_slots;

    if (a->window_layout == CV_WINDOW_RECOMPUTE) {
        p.mode = 3;
        p.win = nullptr;
        p.x = a->x;
        p.x_seq = a->x_seq_stride;
        p.x_tok = a->x_tok_stride;
        // 8 channels per thread with 16-byte vectors when the rows and x allow it
        const bool vec = a->dim % 8 == 0 &&
                         state_packed(a->conv_state, a->state_slot_stride, a->state_ch_stride, a->width, esize) &&
                         aligned16(a->x) && (a->cu_draft || stride16(a->x_seq_stride, esize)) &&
                         stride16(a->x_tok_stride, esize);
        const int threads = kCommitRecomputeThreads;
        const int per_block = vec ? 8 * threads : threads;
        auto kr = vec ? kernel_set(a->dtype, a->width).commit_recompute_vec : kernel_set(a->dtype, a->width).commit_recompute;
        if (launch_pdl(kr, dim3((a->dim + per_block - 1) / per_block, a->n_seq), threads, 0, stream, p) != cudaSuccess)
            return CV_ERR_LAUNCH;
        return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
    }

    const bool packed_state = state_packed(a->conv_state, a->state_slot_stride, a->state_ch_stride, a->width, esize);
    const bool win_base = a->dim % 8 == 0 && aligned16(a->window) && stride16(a->win_seq_stride, esize);
    const bool win_ok = win_base && a->win_col_stride == 1;
    const bool dedup = a->window_layout == CV_WINDOW_DEDUP;
    int smem = 0;
    if (packed_state && win_ok && a->window_layout == CV_WINDOW_DENSE && a->win_ch_stride == R &&
        stride16(a->win_step_stride, esize)) {
        p.mode = 1;
    } else if (!packed_state && win_ok && a->window_layout == CV_WINDOW_DENSE && a->win_ch_stride == R &&
               stride16(a->win_step_stride, esize) && aligned16(a->conv_state) &&
               stride16(a->state_slot_stride, esize) && a->state_ch_stride == a->state_cols &&
               8LL * kCommitWideThreads * a->state_cols * esize <= device_limits().smem_per_block) {
        // rows wider than the window: staged whole, the new window written over their first columns
        p.mode = 5;
        int wt = kCommitWideThreads;
        while (wt > kMinThreads && 8 * (wt / 2) >= a->dim) wt /= 2;
        const int sm = 8 * wt * a->state_cols * esize;
        auto kr = kernel_set(a->dtype, a->width).commit_wide;
        if (ensure_smem(reinterpret_cast<const void *>(kr), sm) != cudaSuccess) return CV_ERR_LAUNCH;
        if (launch_pdl(kr, dim3((a->dim + 8 * wt - 1) / (8 * wt), a->n_seq), wt, sm, stream, p) != cudaSuccess)
            return CV_ERR_LAUNCH;
        return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
    } else if (packed_state && win_base && dedup && a->win_ch_stride == 1 && stride16(a->win_col_stride, esize)) {
        // transposed rows: each thread reads its W-1 accepted column pieces
        p.mode = 4;
        const int threads = a->cu_draft ? kCommitColThreadsPacked : kCommitColThreads;
        auto kr = kernel_set(a->dtype, a->width).commit_cols;
        if (launch_pdl(kr, dim3((a->dim + 8 * threads - 1) / (8 * threads), a->n_seq), threads, 0, stream, p) !=
            cudaSuccess)
            return CV_ERR_LAUNCH;
        return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
    } else if (packed_state && win_ok && dedup && a->win_ch_stride == Q) {
        // one block of 8*kCommitRowThreads channels per sequence, its rows staged by one bulk copy
        int rt = kCommitRowThreads;
        while (rt > kMinThreads && 8 * (rt / 2) >= a->dim) rt /= 2;
        const long long sm = (8LL * rt * Q * esize + 127) / 128 * 128 + 8;
        if (sm <= device_limits().smem_per_block) {
            p.mode = 2;
            const int bc = 8 * rt;
            auto kr = kernel_set(a->dtype, a->width).commit_rows;
            if (ensure_smem(reinterpret_cast<const void *>(kr), (int)sm) != cudaSuccess) return CV_ERR_LAUNCH;
            // commit_rows ORs its bits into err
            if (a->err && cudaMemsetAsync(a->err, 0, sizeof(int32_t) * (size_t)a->n_seq, stream) != cudaSuccess)
                return CV_ERR_LAUNCH;
            if (launch_pdl(kr, dim3((a->dim + bc - 1) / bc, a->n_seq), rt, (int)sm, stream, p) != cudaSuccess)
                return CV_ERR_LAUNCH;
            return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
        }
        p.mode = 0;
    } else {
        p.mode = 0;
    }
    int threads = p.mode == 1 ? kCommitDenseThreads : kCommitElementThreads;
    while (threads > kMinThreads && 8 * (threads / 2) >= a->dim) threads /= 2;
    const int bc = 8 * threads;
    auto k = p.mode == 1 ? kernel_set(a->dtype, a->width).commit_packed : kernel_set(a->dtype, a->width).commit;
    if (ensure_smem(reinterpret_cast<const void *>(k), smem) != cudaSuccess) return CV_ERR_LAUNCH;
    if (launch_pdl(k, dim3((a->dim + bc - 1) / bc, a->n_seq), threads, smem, stream, p) != cudaSuccess)
        return CV_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
}

int check_prefill(const cv_prefill_args *a) {
    if (!a) return CV_ERR_NULL_ARGS;
    if (a->dtype != CV_F32 && a->dtype != CV_BF16) return CV_ERR_DTYPE;
    if (a->width < 2 || a->width > 4) return CV_ERR_WIDTH;
    if (a->n_seq < 0 || a->n_seq > 65535 || a->dim < 1 || a->n_slots < 1 || a->state_cols < a->width - 1 ||
        a->total_tokens < 0 || a->max_seqlen < 0)
        return CV_ERR_SHAPE;
    if (a->qk_channels < 0 || a->qk_channels > a->dim) return CV_ERR_HEAD_DIM;
    if (a->qk_channels > 0 && (!pow2(a->head_dim) || a->head_dim < 8 || a->head_dim > 256 ||
                               a->qk_channels % a->head_dim != 0))
        return CV_ERR_HEAD_DIM;
    if (a->x_tok_stride < 0 || a->out_tok_stride < 0 || a->state_slot_stride < 0 || a->state_ch_stride < 0)
        return CV_ERR_STRIDE;
    if (a->dim > 1 && a->state_ch_stride < a->state_cols) return CV_ERR_STRIDE;
    if (a->n_seq > 0 && (!a->cu_seqlens || !a->conv_state || !a->weight)) return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0 && a->total_tokens > 0 && (!a->x || !a->out)) return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0 && a->out && (a->out == a->x || a->out == a->conv_state || a->out == a->weight))
        return CV_ERR_ALIAS;
    return CV_OK;
}

int launch_prefill(const cv_prefill_args *a, cudaStream_t stream) {
    const int esize = a->dtype == CV_BF16 ? 2 : 4;
    cvk::PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.x = a->x;
    p.x_tok = a->x_tok_stride;
    p.out = a->out;
    p.out_tok = a->out_tok_stride;
    p.cu_seqlens = a->cu_seqlens;
    p.state = a->conv_state;
    p.st_slot = a->state_slot_stride;
    p.st_ch = a->state_ch_stride;
    p.cache_idx = a->cache_idx;
    p.has_init = a->has_initial_state;
    p.weight = a->weight;
    p.bias = a->bias;
    p.err = a->err;
    p.n_slots = a->n_slots;
    p.total_tokens = a->total_tokens;
    p.max_seqlen = a->max_seqlen;
    p.dim = a->dim;
    p.qk_channels = a->qk_channels;
    p.head_dim = a->qk_channels > 0 ? a->head_dim : 8;
    p.eps = a->l2_eps;
    const int cpt = (a->qk_channels > 0 && a->head_dim / 4 > 32) ? 8 : 4;
    // vector rows need the whole run of a thread 16-byte aligned (8 for 4 bf16 channels)
    p.x_vec = a->dim % 8 == 0 && aligned16(a->x) && stride16(a->x_tok_stride, esize);
    p.out_vec = a->dim % 8 == 0 && aligned16(a->out) && stride16(a->out_tok_stride, esize);
    int threads = 128;
    while (threads > 32 && cpt * (threads / 2) >= a->dim) threads /= 2;
    while (a->qk_channels > 0 && cpt * threads < a->head_dim) threads *= 2;
    const long long bc = (long long)cpt * threads;
    const long long nblk = (a->dim + bc - 1) / bc;
    // the longest chunk (fewest halo re-reads) that still gives every SM several blocks, at most 128
    // tokens: more, shorter blocks leave a shorter tail (measured, 8 prompts of 1.5k-5.8k tokens at
    // dim 10240: 262.5 us with 128-token chunks, 271 with 256, 268 with 96, 274 with 64)
    int chunk = kPrefillMaxChunk;
    while (chunk > kPrefillMinChunk &&
           nblk * a->n_seq * ((a->max_seqlen + chunk - 1) / chunk) < 8LL * device_limits().sms)
        chunk /= 2;
    p.chunk = chunk;
    const long long chunks = a->max_seqlen > 0 ? (a->max_seqlen + chunk - 1) / chunk : 1;
    if (chunks > 65535) return CV_ERR_SHAPE;
    const dim3 grid((unsigned)((a->dim + bc - 1) / bc), (unsigned)chunks, (unsigned)a->n_seq);
    auto k = kernel_set(a->dtype, a->width).prefill[cpt == 8 ? 1 : 0];
    // aligned rows: a shared-memory ring of kPrefillRing batches of 8 rows per thread
    const int smem = p.x_vec ? kPrefillRing * 8 * threads * cpt * esize : 0;
    if (ensure_smem(reinterpret_cast<const void *>(k), smem) != cudaSuccess) return CV_ERR_LAUNCH;
    if (launch_pdl(k, grid, threads, smem, stream, p) != cudaSuccess) return CV_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int cv_conv_prefill(const cv_prefill_args *args, void *stream) {
    const int rc = check_prefill(args);
    if (rc != CV_OK) return rc;
    if (args->n_seq == 0) return CV_OK;
    return launch_prefill(args, reinterpret_cast<cudaStream_t>(stream));
}

int cv_verify_plan(const cv_verify_args *args, cv_launch_plan *plan) {
    if (!plan) return CV_ERR_NULL_POINTER;
    return plan_verify(args, plan);
}

int cv_conv_verify(const cv_verify_args *args, void *stream) {
    cv_launch_plan pl;
    const int rc = plan_verify(args, &pl);
    if (rc != CV_OK) return rc;
    if (args->n_seq == 0) return CV_OK;
    return launch_verify(args, pl, reinterpret_cast<cudaStream_t>(stream));
}

int cv_conv_commit(const cv_commit_args *args, void *stream) {
    const int rc = check_commit(args);
    if (rc != CV_OK) return rc;
    if (args->n_seq == 0) return CV_OK;
    return launch_commit(args, reinterpret_cast<cudaStream_t>(stream));
}

const char *cv_status_string(int status) {
    switch (status) {
        case CV_OK: return "ok";
        case CV_ERR_NULL_ARGS: return "argument struct pointer is NULL";
        case CV_ERR_NULL_POINTER: return "a required buffer pointer is NULL";
        case CV_ERR_SHAPE: return "invalid shape (n_seq, dim, n_slots or state_cols)";
        case CV_ERR_TOKENS: return "T outside 1..CV_MAX_T";
        case CV_ERR_WIDTH: return "conv width outside 2..4";
        case CV_ERR_DTYPE: return "unknown dtype";
        case CV_ERR_HEAD_DIM: return "invalid head_dim / qk_channels";
        case CV_ERR_LAYOUT:
            return "unknown window layout, dedup step stride != column stride, or history layout passed to commit";
        case CV_ERR_STRIDE: return "negative stride or overlapping state rows";
        case CV_ERR_ALIAS: return "an output buffer has the base address of an input or of the other output";
        case CV_ERR_LAUNCH: return "CUDA launch failed";
        case CV_ERR_SMEM: return "tile does not fit in shared memory";
        default: return "unknown status";
    }
}

int cv_abi_version(void) { return CV_ABI_VERSION; }

}  // extern "C"
