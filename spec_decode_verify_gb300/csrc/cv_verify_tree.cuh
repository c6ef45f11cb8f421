// Tree verify: the T draft tokens of a sequence form a tree instead of a chain.
//
// sglang PR #46184 ("Scope"): tree verify keeps dense windows and per-token stores.  Token t has a
// parent p(t) in [-1, t) (-1: the committed window); its conv sees the parent's window followed
// by x_t, and its snapshot is window(t) = [window(p)[1 .. W-2], x_t].  A chain (p(t) = t-1) gives
// the plain verify.  The state is left on window(T-1); the commit then restores the accepted
// path's last node (accept_len = its index + 1), as for a chain.
//
// Unrolling that recursion: the W inputs of token t are the last W values along its ancestor path
// [committed window, ..., x_{p(p(t))}, x_{p(t)}, x_t].  So once the committed window and the x
// rows of a block of channels are at hand, the tokens are independent of one another.
//
// A unit is (sequence, block of kTreeChannels channels).  Persistent blocks walk the units
// u = blockIdx.x, blockIdx.x + gridDim.x, ... (the grid is a multiple of the channel-block count
// when it can be, so a block keeps one channel block and loads its taps once).  Each unit's T x
// rows, its committed windows (a packed [channels][W-1] run, rearranged into rows once it lands)
// and its parents are copied into a shared-memory unit buffer by asynchronous copies.  With two
// buffers (p.pitch == 2) the copies of the next unit are started before the current one is
// computed, and the cache slot is read two units ahead, so a block's round trips overlap its own
// arithmetic and stores; with one buffer (p.pitch == 1, long drafts whose two buffers would not
// fit) the next unit's copies start after the current one.  The staged layout is [row][channel]:
// rows 0..W-2 the committed window, rows W-1..W+T-2 the x rows.  For each token the warp walks the
// parents (warp-uniform) to its W input rows and reads them as 16-byte runs; each lane owns 8
// consecutive channels, and warp w of the block takes tokens w, w + warps, ....  Conv
// (conv_chain), SiLU (the fast form; the exact one for each value below -80, see silu_run),
// the L2 groups (sum_squares and the xor-shuffle tree over head_dim/8 lanes) and the rounding are
// those of the chain kernels, so a chain gives their results bit for bit; snapshots and the state
// are the staged raw bits.  Units whose buffers do not allow 16-byte
// copies (strided x, unpacked or wider state rows, the ragged last channel block) are staged with
// plain loads instead.
#pragma once

#include "cv_device.cuh"

namespace cvk {

constexpr int kSeqBadTree = 32;  // err bit: a draft token's parent is outside [-1, t)

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

// Bytes of one unit buffer: the stage [(W-1+T)][kTreeChannels], the packed committed-window run
// [kTreeChannels][W-1] as copied, the T parents (rounded up to 16 bytes).
__host__ __device__ constexpr long long tree_buffer_bytes(int T, int W, int esize) {
    return (long long)(W - 1 + T) * kTreeChannels * esize + (long long)kTreeChannels * (W - 1) * esize +
           (4LL * T + 15) / 16 * 16;
}

template <typename B, int W>
__global__ void __launch_bounds__(128, 4) verify_tree(const __grid_constant__ VerifyParams p) {
    // Before waiting for the previous grid: L2 prefetch hints for the x rows and committed window of
    // the block's first unit (the slot read through L2 only, to form a hint's address inside the
    // state buffer); all data is read after the wait.  (Hints for two units per block -- two thirds
    // of the launch's input with 10 blocks per SM -- made the launch slower: 32.1 against 27.7 us.)
    if (threadIdx.x == 0) {
        const int es = (int)sizeof(B), nb = (p.dim + kTreeChannels - 1) / kTreeChannels;
        {
            const long long u = (long long)blockIdx.x;
            const int sq = (int)(u / nb), cb0 = (int)(u - (long long)sq * nb) * kTreeChannels;
            const int n = min(kTreeChannels, p.dim - cb0);
            if (sq < p.n_seq)
                prefetch_runs_l2(reinterpret_cast<const B *>(p.x) + (long long)sq * p.x_seq + cb0, p.x_tok * es, p.T,
                                 (long long)n * es);
            const int sl = sq >= p.n_seq ? -1 : p.cache_idx ? __ldcg(p.cache_idx + sq) : sq;
            if (sl >= 0 && sl < p.n_slots && p.st_packed)
                prefetch_runs_l2(reinterpret_cast<const B *>(p.state) + (long long)sl * p.st_slot + (long long)cb0 * (W - 1),
                                 0, 1, (long long)n * (W - 1) * es);
        }
    }
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int CB = kTreeChannels;
    constexpr int ES = (int)sizeof(B);
    constexpr int NV = ES / 2;   // 16-byte vectors per 8 elements
    constexpr int CH = 16 / ES;  // elements per 16-byte copy
    const int tid = threadIdx.x, NT = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nw = NT >> 5;
    const int T = p.T;
    const int nbuf = p.pitch;
    const int nblk = (p.dim + CB - 1) / CB;
    const int n_units = p.n_seq * nblk;
    const int iters = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    const long long buf = tree_buffer_bytes(T, W, ES);
    if (NT % 32 != 0 || (nbuf != 1 && nbuf != 2) || nbuf * buf > (long long)dynamic_smem_bytes())
        return;  // launch mismatch
    auto stage_of = [&](int b) { return reinterpret_cast<B *>(smem_raw + b * buf); };
    auto packed_of = [&](int b) { return stage_of(b) + (long long)(R + T) * CB; };
    auto parents_of = [&](int b) { return reinterpret_cast<int *>(packed_of(b) + CB * R); };
    auto unit_of = [&](int k, int &s, int &cb) {
        const int u = (int)blockIdx.x + k * (int)gridDim.x;
        s = u / nblk;
        cb = u - s * nblk;
    };
    auto load_index = [&](int k, int &slot, int &off) {
        if (k >= iters) return;
        int s, cb;
        unit_of(k, s, cb);
        slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
        off = p.state_off ? __ldg(p.state_off + s) : 0;
    };
    // start the loads of unit k into buffer b, then one commit group (possibly empty)
    auto issue = [&](int k, int b, int slot, int off) {
        int s, cb;
        unit_of(k, s, cb);
        const int c0 = cb * CB;
        const int nch = min(CB, p.dim - c0);
        B *stage = stage_of(b);
        if (slot >= 0) {  // parents (validated with the unit; read even when the slot is out of range)
            const int *par = p.parent + (long long)s * T;
            int *sp = parents_of(b);
            for (int t = tid; t < T; t += NT) cp_async4(sp + t, par + t);
        }
        if (slot >= 0 && seq_status(slot, off, p.n_slots, p.state_cols, R) == 0) {
            const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c0;
            if (p.x_vec && nch == CB) {
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
            const B *srow = reinterpret_cast<const B *>(p.state) + (long long)slot * p.st_slot +
                            (long long)c0 * p.st_ch + off;
            if (p.st_packed && nch == CB) {
                B *pk = packed_of(b);
                for (int i = tid; i < CB * R / CH; i += NT) cp_async16(pk + i * CH, srow + i * CH);
            } else {
                for (int i = tid; i < R * CB; i += NT) {
                    const int ch = i / R, kk = i - ch * R;  // consecutive threads, consecutive elements
                    stage[kk * CB + ch] = ch < nch ? srow[(long long)ch * p.st_ch + kk] : (B)0;
                }
            }
        }
        cp_async_commit();
    };

    // indices of the current unit and of the next one
    int slot_k = -1, off_k = 0, slot_n = -1, off_n = 0;
    load_index(0, slot_k, off_k);
    load_index(1, slot_n, off_n);
    if (iters > 0) issue(0, 0, slot_k, off_k);

    const int cl = lane * 8;
    const int lanes = p.head_dim >> 3;
    uint32_t wr[4 * W * NV];  // taps of this lane's channels, packed raw words [8][W]
    float bs[8];
    int wcb = -1;
    for (int k = 0; k < iters; ++k) {
        const int b = nbuf == 2 ? (k & 1) : 0;
        if (nbuf == 2) {  // the next unit's copies go out before this unit is computed
            if (k + 1 < iters)
                issue(k + 1, b ^ 1, slot_n, off_n);
            else
                cp_async_commit();
        }
        int slot_nn = -1, off_nn = 0;
        load_index(k + 2, slot_nn, off_nn);

        int s, cb;
        unit_of(k, s, cb);
        const int c0 = cb * CB;
        const int nch = min(CB, p.dim - c0);
        const int c = c0 + cl;
        const int my = max(0, min(8, nch - cl));
        const bool full = my == 8;
        if (cb != wcb) {  // once per block when the grid is a multiple of the channel-block count
            wcb = cb;
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
        }

        // this unit's copies have landed (with two buffers, the next unit's may still be in flight)
        if (nbuf == 2)
            asm volatile("cp.async.wait_group 1;\n" ::: "memory");
        else
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        __syncthreads();  // every thread's copies and plain stores of this unit are visible
        const int slot = slot_k, off = off_k;
        B *stage = stage_of(b);
        const int *spar = parents_of(b);
        int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
        bool bad = false;
        for (int t = tid; t < T && slot >= 0; t += NT) {
            const int q = spar[t];
            bad |= q < -1 || q >= t;
        }
        if (__syncthreads_or(bad) && slot >= 0) status |= kSeqBadTree;
        if (p.err && cb == 0 && tid == 0) p.err[s] = status;
        if (slot >= 0 && status == 0) {  // (block-uniform)
            if (p.st_packed && nch == CB && warp == 0) {
                // the packed run [channel][W-1] -> stage rows 0 .. W-2 (this lane's 8 channels)
                union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
                for (int i = 0; i < R * NV; ++i) u.v[i] = reinterpret_cast<const uint4 *>(packed_of(b) + cl * R)[i];
#pragma unroll
                for (int kk = 0; kk < R; ++kk) {
                    union { uint4 q[NV]; B b[8]; } r;
#pragma unroll
                    for (int e = 0; e < 8; ++e) r.b[e] = u.b[e * R + kk];
#pragma unroll
                    for (int i = 0; i < NV; ++i) reinterpret_cast<uint4 *>(stage + kk * CB + cl)[i] = r.q[i];
                }
            }
            __syncthreads();

            // the W input rows of token t: row R+t, then each ancestor's row, then the committed
            // window's columns from the newest back (a code < 0 names committed column R + code)
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
            B *ob = reinterpret_cast<B *>(p.out) + (long long)s * p.out_seq + c;
            B *wb = reinterpret_cast<B *>(p.win) + (long long)s * p.w_seq + (long long)c * p.w_ch;
            // packed dense snapshots: a lane's 8 channels x R columns of one token are one 16-byte-aligned run
            const bool win_vec = full && p.st_vec;

            for (int t = warp; t < T; t += nw) {
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
                silu_run<8>(acc, y);  // (one range check for the token's 8 channels, exact form per value)
                // snapshot t = window(t): the last R inputs (raw bits)
                if (win_vec) {
                    union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
#pragma unroll
                        for (int kk = 0; kk < R; ++kk) u.b[e * R + kk] = in[kk + 1][e];
#pragma unroll
                    for (int i = 0; i < R * NV; ++i) reinterpret_cast<uint4 *>(wb + (long long)t * p.w_step)[i] = u.v[i];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e < my)
#pragma unroll
                            for (int kk = 0; kk < R; ++kk)
                                wb[(long long)t * p.w_step + (long long)e * p.w_ch + (long long)kk * p.w_col] = in[kk + 1][e];
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
                // the state is left on the window of token T-1 (its last R inputs); every read of
                // the state row happened when the unit was staged
                if (t == T - 1) {
                    B *sdst = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
                    if (full && p.st_packed) {
                        union { uint4 v[R * NV]; B b[8 * R]; } u;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
#pragma unroll
                            for (int kk = 0; kk < R; ++kk) u.b[e * R + kk] = in[kk + 1][e];
#pragma unroll
                        for (int i = 0; i < R * NV; ++i) reinterpret_cast<uint4 *>(sdst)[i] = u.v[i];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (e < my)
#pragma unroll
                                for (int kk = 0; kk < R; ++kk) sdst[(long long)e * p.st_ch + kk] = in[kk + 1][e];
                    }
                }
            }
        }
        __syncthreads();  // every thread is done with buffer b before it is refilled
        if (nbuf == 1 && k + 1 < iters) issue(k + 1, 0, slot_n, off_n);
        slot_k = slot_n, off_k = off_n;
        slot_n = slot_nn, off_n = off_nn;
    }
}

}  // namespace cvk
