// Tree verify: the T draft tokens of a sequence form a tree instead of a chain.
//
// sglang PR #46184 ("Scope"): tree verify keeps dense windows and per-token stores.  Token t has a
// parent p(t) in [-1, t) (-1: the committed window); its conv sees the parent's window followed
// by x_t, and its snapshot is window(t) = [window(p)[1 .. W-2], x_t].  A chain (p(t) = t-1) gives
// the plain verify.  The state is left on window(T-1); the commit then restores the accepted
// path's last node (accept_len = its index + 1), as for a chain.
//
// One block per (block of 8*threads channels, sequence); a thread owns 8 consecutive channels and
// walks the tokens in index order, so a parent is always done before its children.  The parent's
// window is the committed window (registers) or the window this thread kept for the parent: in
// shared memory (laid out [token][column][channel of 8][thread], so a warp's accesses are
// consecutive) when the block's T windows fit, else read back from the dense window buffer with
// plain loads, which see the thread's own earlier stores.  x, out and packed snapshot runs move
// as 16-byte vectors when aligned.  Conv (conv_chain), SiLU, the L2 groups (sum_squares and the
// xor-shuffle tree over head_dim/8 lanes) and the rounding are those of the general kernel, so a
// chain gives its results bit for bit.
#pragma once

#include "cv_device.cuh"

namespace cvk {

constexpr int kSeqBadTree = 32;  // err bit: a draft token's parent is outside [-1, t)

template <typename B, int W>
__global__ void __launch_bounds__(128) verify_tree(const __grid_constant__ VerifyParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int T = p.T;
    const int *par = p.parent + (long long)s * T;

    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int off = p.state_off ? __ldg(p.state_off + s) : 0;
    int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
    if (slot >= 0)
        for (int t = 0; t < T; ++t) {
            const int q = __ldg(par + t);
            if (q < -1 || q >= t) status |= kSeqBadTree;
        }
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;  // (block-uniform)

    const int c = (blockIdx.x * blockDim.x + tid) * 8;  // first channel of this thread
    const int my = max(0, min(8, p.dim - c));

    // committed window, taps, bias
    B w0[R][8];
    B *srow = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch + off;
    float wt[8][W], bs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
        for (int k = 0; k < R; ++k) w0[k][e] = e < my ? srow[(long long)e * p.st_ch + k] : (B)0;
#pragma unroll
        for (int j = 0; j < W; ++j) wt[e][j] = e < my ? widen<B>(reinterpret_cast<const B *>(p.weight)[(long long)(c + e) * W + j]) : 0.0f;
        bs[e] = (p.bias && e < my) ? widen<B>(reinterpret_cast<const B *>(p.bias)[c + e]) : 0.0f;
    }

    const bool l2_block = (int)(blockIdx.x * blockDim.x * 8) < p.qk_channels;  // block-uniform
    const bool l2_mine = c < p.qk_channels;
    const int lanes = p.head_dim >> 3;
    const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c;
    B *ob = reinterpret_cast<B *>(p.out) + (long long)s * p.out_seq + c;
    B *wb = reinterpret_cast<B *>(p.win) + (long long)s * p.w_seq + (long long)c * p.w_ch;
    // token windows kept in shared memory when they fit (p.pitch != 0): element (t, k, e) of thread
    // tid at ((t*R + k)*8 + e)*NT + tid
    extern __shared__ __align__(16) unsigned char smem_raw[];
    B *kept = reinterpret_cast<B *>(smem_raw);
    const int NT = blockDim.x;
    const bool in_smem = p.pitch != 0;
    if (in_smem && (long long)T * R * 8 * NT * (long long)sizeof(B) > (long long)dynamic_smem_bytes()) return;
    const bool full = my == 8;
    // packed dense snapshots: a thread's 8 channels x R columns of one token are one 16-byte-aligned run
    const bool win_vec = full && p.st_vec;
    constexpr int NV = (int)sizeof(B) / 2;  // 16-byte vectors per 8 elements

    B last[R][8];  // window of the newest token (the state after the loop)
    for (int t = 0; t < T; ++t) {
        const int q = __ldg(par + t);
        // the parent's window: committed window, or kept by this thread for the parent
        B pw[R][8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int k = 0; k < R; ++k) {
                if (q < 0)
                    pw[k][e] = w0[k][e];
                else if (in_smem)
                    pw[k][e] = kept[((q * R + k) * 8 + e) * NT + tid];
                else
                    pw[k][e] = e < my ? wb[(long long)q * p.w_step + (long long)e * p.w_ch + (long long)k * p.w_col] : (B)0;
            }
        B xrow[8];
        if (full && p.x_vec) {
            union { uint4 v[NV]; B b[8]; } u;
#pragma unroll
            for (int i = 0; i < NV; ++i) u.v[i] = *reinterpret_cast<const uint4 *>(xs + (long long)t * p.x_tok + i * (8 / NV));
#pragma unroll
            for (int e = 0; e < 8; ++e) xrow[e] = u.b[e];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xrow[e] = e < my ? xs[(long long)t * p.x_tok + e] : (B)0;
        }
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const B xr = xrow[e];
            float in[W];
#pragma unroll
            for (int k = 0; k < R; ++k) in[k] = widen<B>(pw[k][e]);
            in[R] = widen<B>(xr);
            y[e] = silu(conv_chain<B, W>(bs[e], wt[e], in));
            // window(t) = [window(parent)[1 .. W-2], x_t]
#pragma unroll
            for (int k = 0; k + 1 < R; ++k) last[k][e] = pw[k + 1][e];
            last[R - 1][e] = xr;
            if (in_smem)
#pragma unroll
                for (int k = 0; k < R; ++k) kept[((t * R + k) * 8 + e) * NT + tid] = last[k][e];
        }
        // snapshot t (raw bits)
        if (win_vec) {
            union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) u.b[e * R + k] = last[k][e];
#pragma unroll
            for (int i = 0; i < R * NV; ++i)
                reinterpret_cast<uint4 *>(wb + (long long)t * p.w_step)[i] = u.v[i];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < my)
#pragma unroll
                    for (int k = 0; k < R; ++k)
                        wb[(long long)t * p.w_step + (long long)e * p.w_ch + (long long)k * p.w_col] = last[k][e];
        }
        if (l2_block) {
            float ss = sum_squares<8>(y);
            for (int o = lanes >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (l2_mine) {
                const float r = rsqrtf(ss + p.eps);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] *= r;
            }
        }
        if (full && p.out_vec) {
            union { uint4 v[NV]; B b[8]; } u;
#pragma unroll
            for (int e = 0; e < 8; ++e) u.b[e] = narrow<B>(y[e]);
#pragma unroll
            for (int i = 0; i < NV; ++i) reinterpret_cast<uint4 *>(ob + (long long)t * p.out_tok)[i] = u.v[i];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < my) ob[(long long)t * p.out_tok + e] = narrow<B>(y[e]);
        }
    }
    // the state is left on the window of token T-1
    B *sdst = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (e < my)
#pragma unroll
            for (int k = 0; k < R; ++k) sdst[(long long)e * p.st_ch + k] = last[k][e];
}

}  // namespace cvk
