// Tree verify: the T draft tokens of a sequence form a tree instead of a chain.
//
// sglang PR #46184 ("Scope"): tree verify keeps dense windows and per-token stores.  Token t has a
// parent p(t) in [-1, t) (-1: the committed window); its conv sees the parent's window followed
// by x_t, and its snapshot is window(t) = [window(p)[1 .. W-2], x_t].  A chain (p(t) = t-1) gives
// the plain verify.  The state is left on window(T-1); the commit then restores the accepted
// path's last node (accept_len = its index + 1), as for a chain.
//
// Unrolling that recursion: the W inputs of token t are the last W values along its ancestor path
// [committed window, ..., x_{p(p(t))}, x_{p(t)}, x_t].  So once a block holds the committed
// window and the x rows of its channels, its tokens are independent of one another.  One block per
// (block of kTreeChannels channels, sequence) stages, together, the committed window (rows
// 0..W-2), the T x rows (rows W-1..W+T-2, by asynchronous 16-byte copies when aligned) and the
// parents in shared memory, laid out [row][channel].  Then warp w takes tokens w, w + warps, ...
// (the host launches one warp per block: more resident blocks hide more of each block's fixed
// chain of round trips than more warps per block do):
// each lane owns 8 consecutive channels, the warp walks the token's parents (warp-uniform) to its
// W input rows and reads them as 16-byte runs.  Conv (conv_chain), SiLU (the fast form, the exact
// one for a token whose channels reach below -80), the L2 groups (sum_squares and the xor-shuffle
// tree over head_dim/8 lanes) and the rounding are those of the chain kernels, so a chain gives
// their results bit for bit; snapshots and the state are the staged raw bits.
#pragma once

#include "cv_device.cuh"

namespace cvk {

constexpr int kSeqBadTree = 32;  // err bit: a draft token's parent is outside [-1, t)

template <typename B, int W>
__global__ void __launch_bounds__(128) verify_tree(const __grid_constant__ VerifyParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int CB = kTreeChannels;
    constexpr int ES = (int)sizeof(B);
    constexpr int NV = ES / 2;  // 16-byte vectors per 8 elements
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = NT >> 5;
    const int T = p.T;
    const int *par = p.parent + (long long)s * T;

    // shared memory: the stage [R + T][CB] of B, then the T parents
    extern __shared__ __align__(16) unsigned char smem_raw[];
    B *stage = reinterpret_cast<B *>(smem_raw);
    int *spar = reinterpret_cast<int *>(stage + (long long)(R + T) * CB);
    if ((long long)(R + T) * CB * ES + 4LL * T > (long long)dynamic_smem_bytes()) return;

    // this lane's 8 channels: taps and bias, loaded while the cache slot is looked up
    const int c0 = blockIdx.x * CB;
    const int nch = min(CB, p.dim - c0);
    const int cl = lane * 8;
    const int c = c0 + cl;
    const int my = max(0, min(8, nch - cl));
    const bool full = my == 8;
    // taps kept packed (raw words, [8 channels][W]) and widened where used
    uint32_t wr[4 * W * NV];
    float bs[8];
    if (full && p.w_vec) {
#pragma unroll
        for (int i = 0; i < W * NV; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const B *>(p.weight) + (long long)c * W) + i);
            wr[4 * i] = v.x, wr[4 * i + 1] = v.y, wr[4 * i + 2] = v.z, wr[4 * i + 3] = v.w;
        }
    } else {
        const B *wg = reinterpret_cast<const B *>(p.weight) + (long long)c * W;
#pragma unroll
        for (int i = 0; i < 4 * W * NV; ++i) {
            if constexpr (ES == 2) {
                const uint32_t lo = 2 * i < my * W ? wg[2 * i] : 0u, hi = 2 * i + 1 < my * W ? wg[2 * i + 1] : 0u;
                wr[i] = pack_halves(lo, hi);
            } else {
                wr[i] = i < my * W ? wg[i] : 0u;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) bs[e] = (p.bias && e < my) ? widen<B>(reinterpret_cast<const B *>(p.bias)[c + e]) : 0.0f;

    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int off = p.state_off ? __ldg(p.state_off + s) : 0;
    int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
    int bad = 0;
    for (int t = tid; t < T; t += NT) {
        const int q = __ldg(par + t);
        if (q < -1 || q >= t) bad = 1;
        spar[t] = q;
    }
    if (__syncthreads_or(bad) && slot >= 0) status |= kSeqBadTree;
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;  // (block-uniform)

    // x rows -> stage rows R .. R+T-1
    const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c0;
    if (p.x_vec && nch == CB) {
        constexpr int CH = 16 / ES;  // elements per copy
        for (int i = tid; i < T * (CB / CH); i += NT) {
            const int t = i / (CB / CH), m = (i - t * (CB / CH)) * CH;
            cp_async16(stage + (long long)(R + t) * CB + m, xs + (long long)t * p.x_tok + m);
        }
    } else {
        for (int i = tid; i < T * CB; i += NT) {
            const int t = i / CB, ch = i - t * CB;
            stage[(long long)(R + t) * CB + ch] = ch < nch ? xs[(long long)t * p.x_tok + ch] : (B)0;
        }
    }
    // committed window -> stage rows 0 .. R-1
    const B *srow = reinterpret_cast<const B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * p.st_ch + off;
    for (int i = tid; i < R * CB; i += NT) {
        const int ch = i / R, k = i - ch * R;  // consecutive threads read consecutive elements of packed rows
        stage[k * CB + ch] = ch < nch ? srow[(long long)ch * p.st_ch + k] : (B)0;
    }
    cp_async_wait_all();
    __syncthreads();

    // the W input rows of token t: row R+t, then each ancestor's row, then the committed window's
    // columns from the newest back (a code < 0 names committed column R + code)
    auto input_rows = [&](int t, int *rows) {
        int code = t;
#pragma unroll
        for (int j = W - 1; j >= 0; --j) {
            rows[j] = R + code;
            if (j > 0) code = code >= 0 ? spar[code] : code - 1;
        }
    };
    auto load8 = [&](int r, B *v) {
        union { uint4 q[NV]; B b[8]; } u;
#pragma unroll
        for (int i = 0; i < NV; ++i) u.q[i] = reinterpret_cast<const uint4 *>(stage + (long long)r * CB + cl)[i];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = u.b[e];
    };

    const bool l2_mine = c < p.qk_channels;
    const bool l2_warp = c0 < p.qk_channels;  // (warp-uniform: every lane joins the shuffles)
    const int lanes = p.head_dim >> 3;
    B *ob = reinterpret_cast<B *>(p.out) + (long long)s * p.out_seq + c;
    B *wb = reinterpret_cast<B *>(p.win) + (long long)s * p.w_seq + (long long)c * p.w_ch;
    // packed dense snapshots: a lane's 8 channels x R columns of one token are one 16-byte-aligned run
    const bool win_vec = full && p.st_vec;

    for (int t = warp; t < T; t += nwarps) {
        int rows[W];
        input_rows(t, rows);
        B in[W][8];
#pragma unroll
        for (int j = 0; j < W; ++j) load8(rows[j], in[j]);
        float acc[8], y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v[W], wt[W];
#pragma unroll
            for (int j = 0; j < W; ++j) {
                v[j] = widen<B>(in[j][e]);
                wt[j] = elem_f<B>(wr, e * W + j);
            }
            acc[e] = conv_chain<B, W>(bs[e], wt, v);
        }
        silu_run<8>(acc, y);  // (one range check for the token's 8 channels)
        // snapshot t = window(t): the last R inputs (raw bits)
        if (win_vec) {
            union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) u.b[e * R + k] = in[k + 1][e];
#pragma unroll
            for (int i = 0; i < R * NV; ++i) reinterpret_cast<uint4 *>(wb + (long long)t * p.w_step)[i] = u.v[i];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < my)
#pragma unroll
                    for (int k = 0; k < R; ++k)
                        wb[(long long)t * p.w_step + (long long)e * p.w_ch + (long long)k * p.w_col] = in[k + 1][e];
        }
        if (l2_warp) {
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
        // the state is left on the window of token T-1 (its last R inputs); the rows were all read
        // before the barrier above, so no other warp still needs the state
        if (t == T - 1) {
            B *sdst = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
            if (full && p.st_packed) {
                union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int k = 0; k < R; ++k) u.b[e * R + k] = in[k + 1][e];
#pragma unroll
                for (int i = 0; i < R * NV; ++i) reinterpret_cast<uint4 *>(sdst)[i] = u.v[i];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < my)
#pragma unroll
                        for (int k = 0; k < R; ++k) sdst[(long long)e * p.st_ch + k] = in[k + 1][e];
            }
        }
    }
}

}  // namespace cvk
