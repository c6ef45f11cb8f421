// C ABI of the verify/commit library: argument validation, launch planning and dispatch to the
// kernels in cv_kernels.cuh.  Every check runs on the host before anything is launched; the
// function reports a negative status and launches nothing when a check fails.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "convverify.h"
#include "cv_kernels.cuh"

namespace {

constexpr int kMaxThreads = 256;
constexpr int kMinThreads = 32;
constexpr int kSmemBudget = 96 * 1024;   // per-block tile budget; keeps >= 2 blocks per SM
constexpr int kCommitThreads = 256;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride16(long long stride_elems, int esize) { return ((stride_elems * esize) & 15) == 0; }
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

// Validates verify arguments; on success fills the launch plan.
int plan_verify(const cv_verify_args *a, cv_launch_plan *pl) {
    if (!a) return CV_ERR_NULL_ARGS;
    if (a->dtype != CV_F32 && a->dtype != CV_BF16) return CV_ERR_DTYPE;
    if (a->width < 2 || a->width > 4) return CV_ERR_WIDTH;
    if (a->T < 1 || a->T > CV_MAX_T) return CV_ERR_TOKENS;
    if (a->n_seq < 0 || a->n_seq > 65535 || a->dim < 1 || a->n_slots < 1 || a->state_cols < a->width - 1)
        return CV_ERR_SHAPE;
    if (a->window_layout != CV_WINDOW_DENSE && a->window_layout != CV_WINDOW_DEDUP) return CV_ERR_LAYOUT;
    if (a->window_layout == CV_WINDOW_DEDUP && a->win_step_stride != a->win_col_stride) return CV_ERR_LAYOUT;
    if (a->qk_channels < 0 || a->qk_channels > a->dim) return CV_ERR_HEAD_DIM;
    if (a->qk_channels > 0 && (!pow2(a->head_dim) || a->head_dim < 8 || a->head_dim > 256 ||
                               a->qk_channels % a->head_dim != 0))
        return CV_ERR_HEAD_DIM;
    if (a->x_seq_stride < 0 || a->x_tok_stride < 0 || a->out_seq_stride < 0 || a->out_tok_stride < 0 ||
        a->state_slot_stride < 0 || a->state_ch_stride < 0 || a->win_seq_stride < 0 || a->win_step_stride < 0 ||
        a->win_ch_stride < 0 || a->win_col_stride < 0)
        return CV_ERR_STRIDE;
    if (a->dim > 1 && a->state_ch_stride < a->state_cols) return CV_ERR_STRIDE;
    if (a->n_seq > 0 && (!a->x || !a->out || !a->conv_state || !a->weight || !a->window)) return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0) {
        const void *outs[2] = {a->out, a->window};
        const void *ins[3] = {a->x, a->conv_state, a->weight};
        for (const void *o : outs)
            for (const void *i : ins)
                if (o == i) return CV_ERR_ALIAS;
        if (a->out == a->window) return CV_ERR_ALIAS;
    }

    const int esize = a->dtype == CV_BF16 ? 2 : 4;
    const int rows = a->T + a->width - 1;
    const int pad = 16 / esize;  // one 16-byte vector of padding per tile row
    const int min_threads = (a->qk_channels > 0 && a->head_dim / 8 > kMinThreads) ? a->head_dim / 8 : kMinThreads;
    int threads = 128;
    // small channel counts: do not launch threads that own no channel
    while (threads > min_threads && 8 * (threads / 2) >= a->dim) threads /= 2;
    // the block's channel count must hold whole L2 groups
    while (a->qk_channels > 0 && 8 * threads < a->head_dim) threads *= 2;
    long long smem = (long long)rows * (8 * threads + pad) * esize;
    while (smem > kSmemBudget && threads > min_threads && 8 * (threads / 2) >= (a->qk_channels > 0 ? a->head_dim : 8)) {
        threads /= 2;
        smem = (long long)rows * (8 * threads + pad) * esize;
    }
    if (smem > 227 * 1024 || threads > kMaxThreads) return CV_ERR_SMEM;
    const int bc = 8 * threads;
    pl->grid_x = (a->dim + bc - 1) / bc;
    pl->grid_y = a->n_seq;
    pl->threads = threads;
    pl->smem_bytes = (int)smem;
    pl->channels_per_block = bc;
    pl->reserved0 = 0;
    return CV_OK;
}

// Opt a kernel into more than 48 KB of dynamic shared memory, once per device.
template <typename K>
cudaError_t ensure_smem(K kernel, int bytes, std::atomic<unsigned long long> &done) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

template <typename B, int W>
int launch_verify(const cv_verify_args *a, const cv_launch_plan &pl, cudaStream_t stream) {
    static std::atomic<unsigned long long> smem_done{0};
    const int esize = (int)sizeof(B);
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
    p.cache_idx = a->cache_idx;
    p.state_off = a->state_off;
    p.weight = a->weight;
    p.bias = a->bias;
    p.win = a->window;
    p.dedup = a->window_layout == CV_WINDOW_DEDUP;
    p.w_seq = a->win_seq_stride;
    p.w_step = p.dedup ? a->win_col_stride : a->win_step_stride;
    p.w_ch = a->win_ch_stride;
    p.w_col = a->win_col_stride;
    p.err = a->err;
    p.n_seq = a->n_seq;
    p.T = a->T;
    p.dim = a->dim;
    p.n_slots = a->n_slots;
    p.state_cols = a->state_cols;
    p.qk_channels = a->qk_channels;
    p.head_dim = a->qk_channels > 0 ? a->head_dim : 8;
    p.pitch = pl.channels_per_block + 16 / esize;
    p.eps = a->l2_eps;
    p.x_vec = aligned16(a->x) && stride16(a->x_seq_stride, esize) && stride16(a->x_tok_stride, esize);
    p.out_vec = aligned16(a->out) && stride16(a->out_seq_stride, esize) && stride16(a->out_tok_stride, esize);
    p.st_vec = aligned16(a->conv_state) && stride16(a->state_slot_stride, esize) && a->state_ch_stride == W - 1;
    p.w_vec = aligned16(a->weight);
    p.b_vec = a->bias ? aligned16(a->bias) : 0;

    auto kernel = cvk::verify_kernel<B, W>;
    if (ensure_smem(kernel, pl.smem_bytes, smem_done) != cudaSuccess) return CV_ERR_LAUNCH;
    kernel<<<dim3(pl.grid_x, pl.grid_y), pl.threads, pl.smem_bytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
}

template <typename B>
int dispatch_verify(const cv_verify_args *a, const cv_launch_plan &pl, cudaStream_t st) {
    switch (a->width) {
        case 2: return launch_verify<B, 2>(a, pl, st);
        case 3: return launch_verify<B, 3>(a, pl, st);
        default: return launch_verify<B, 4>(a, pl, st);
    }
}

int check_commit(const cv_commit_args *a) {
    if (!a) return CV_ERR_NULL_ARGS;
    if (a->dtype != CV_F32 && a->dtype != CV_BF16) return CV_ERR_DTYPE;
    if (a->width < 2 || a->width > 4) return CV_ERR_WIDTH;
    if (a->T < 1 || a->T > CV_MAX_T) return CV_ERR_TOKENS;
    if (a->n_seq < 0 || a->n_seq > 65535 || a->dim < 1 || a->n_slots < 1 || a->state_cols < a->width - 1)
        return CV_ERR_SHAPE;
    if (a->window_layout != CV_WINDOW_DENSE && a->window_layout != CV_WINDOW_DEDUP) return CV_ERR_LAYOUT;
    if (a->window_layout == CV_WINDOW_DEDUP && a->win_step_stride != a->win_col_stride) return CV_ERR_LAYOUT;
    if (a->state_slot_stride < 0 || a->state_ch_stride < 0 || a->win_seq_stride < 0 || a->win_step_stride < 0 ||
        a->win_ch_stride < 0 || a->win_col_stride < 0)
        return CV_ERR_STRIDE;
    if (a->dim > 1 && a->state_ch_stride < a->state_cols) return CV_ERR_STRIDE;
    if (a->n_seq > 0 && (!a->conv_state || !a->window || !a->accept_len)) return CV_ERR_NULL_POINTER;
    if (a->n_seq > 0 && a->conv_state == a->window) return CV_ERR_ALIAS;
    return CV_OK;
}

template <typename B, int W>
int launch_commit(const cv_commit_args *a, cudaStream_t stream) {
    const int esize = (int)sizeof(B);
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
    p.n_seq = a->n_seq;
    p.T = a->T;
    p.dim = a->dim;
    p.n_slots = a->n_slots;
    p.st_vec = aligned16(a->conv_state) && stride16(a->state_slot_stride, esize) && a->state_ch_stride == W - 1;
    const long long elems = (long long)a->dim * (W - 1);
    const long long per_block = (long long)kCommitThreads * (p.st_vec ? 16 / esize : 1);
    long long gx = (elems + per_block - 1) / per_block;
    if (gx > 1024) gx = 1024;
    cvk::commit_kernel<B, W><<<dim3((unsigned)gx, a->n_seq), kCommitThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? CV_OK : CV_ERR_LAUNCH;
}

template <typename B>
int dispatch_commit(const cv_commit_args *a, cudaStream_t st) {
    switch (a->width) {
        case 2: return launch_commit<B, 2>(a, st);
        case 3: return launch_commit<B, 3>(a, st);
        default: return launch_commit<B, 4>(a, st);
    }
}

}  // namespace

extern "C" {

int cv_verify_plan(const cv_verify_args *args, cv_launch_plan *plan) {
    if (!plan) return CV_ERR_NULL_POINTER;
    return plan_verify(args, plan);
}

int cv_conv_verify(const cv_verify_args *args, void *stream) {
    cv_launch_plan pl;
    const int rc = plan_verify(args, &pl);
    if (rc != CV_OK) return rc;
    if (args->n_seq == 0) return CV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return args->dtype == CV_BF16 ? dispatch_verify<uint16_t>(args, pl, st) : dispatch_verify<uint32_t>(args, pl, st);
}

int cv_conv_commit(const cv_commit_args *args, void *stream) {
    const int rc = check_commit(args);
    if (rc != CV_OK) return rc;
    if (args->n_seq == 0) return CV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return args->dtype == CV_BF16 ? dispatch_commit<uint16_t>(args, st) : dispatch_commit<uint32_t>(args, st);
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
        case CV_ERR_LAYOUT: return "unknown window layout, or dedup step stride != column stride";
        case CV_ERR_STRIDE: return "negative stride or overlapping state rows";
        case CV_ERR_ALIAS: return "an output buffer has the base address of an input or of the other output";
        case CV_ERR_LAUNCH: return "CUDA launch failed";
        case CV_ERR_SMEM: return "tile does not fit in shared memory";
        default: return "unknown status";
    }
}

int cv_abi_version(void) { return CV_ABI_VERSION; }

}  // extern "C"
