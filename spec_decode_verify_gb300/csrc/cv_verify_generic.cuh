// Verify kernel for any strides and layouts (the general path).
//
// Used when the fast path's preconditions do not hold: unaligned or odd-strided x / out, a
// channel count that is not a multiple of 8, transposed or permuted snapshot layouts, a
// deduplicated row longer than the fast path keeps in registers, or history-row state rows wider
// than the row (or T above the static range).  One block per (channel block,
// sequence); the block's inputs are staged once in a token-major shared-memory tile
//     tile[j][c] = full_c[j],  j in [0, W-1+T)   (rows 0..W-2: committed window, then x_0..x_{T-1})
// and every snapshot layout and the committed window are written from that tile in destination
// order (channel-major runs, channel-stride-1 runs, or element by element).  The arithmetic is the
// same as the fast path's: fp32, bias first, taps in order (conv_chain), SiLU, L2
// over the head_dim group as an xor-shuffle over head_dim/8 lanes.  Packed ragged drafts (p.cu_draft):
// the sequence's T_s rows start at row cu[s] of x and out, and everything runs over T_s tokens
// (snapshot steps and deduplicated columns past them stay untouched; T_s = 0 writes only the state).
#pragma once

#include <type_traits>

#include "cv_device.cuh"

namespace cvk {

// Eight consecutive elements as 16-byte words: one uint4 for bf16, two for fp32.
template <typename B> struct Oct {
    static constexpr int NV = (int)sizeof(B) / 2;  // uint4 vectors per 8 elements
    uint4 v[NV];
    __device__ __forceinline__ B get(int e) const {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(v);
        if (sizeof(B) == 2) return (B)((w[e >> 1] >> ((e & 1) * 16)) & 0xffffu);
        return (B)w[e];
    }
    __device__ __forceinline__ void set(int e, B b) {
        uint32_t *w = reinterpret_cast<uint32_t *>(v);
        if (sizeof(B) == 2) {
            const int sh = (e & 1) * 16;
            w[e >> 1] = (w[e >> 1] & ~(0xffffu << sh)) | ((uint32_t)b << sh);
        } else {
            w[e] = (uint32_t)b;
        }
    }
};

template <typename B> __device__ __forceinline__ void load_oct(Oct<B> &o, const B *p) {
#pragma unroll
    for (int i = 0; i < Oct<B>::NV; ++i) o.v[i] = *reinterpret_cast<const uint4 *>(p + i * (16 / sizeof(B)));
}
template <typename B> __device__ __forceinline__ void load_oct_nc(Oct<B> &o, const B *p) {
#pragma unroll
    for (int i = 0; i < Oct<B>::NV; ++i) o.v[i] = __ldg(reinterpret_cast<const uint4 *>(p + i * (16 / sizeof(B))));
}
template <typename B> __device__ __forceinline__ void store_oct(B *p, const Oct<B> &o) {
#pragma unroll
    for (int i = 0; i < Oct<B>::NV; ++i) *reinterpret_cast<uint4 *>(p + i * (16 / sizeof(B))) = o.v[i];
}

// Write one view of the tile: element (c, q) for c < nch, q < ncol is tile[(jofs+q)*pitch + c] and
// goes to dst[c*ch_stride + q*col_stride].  Three shapes: channel-major contiguous (the dedup row
// and the dense per-token chunks: one coalesced run of nch*ncol elements), channel-stride-1 (a
// transposed row: one contiguous run of channels per column), and anything else element by element.
// Tile element -> destination element: the same bits when the types agree; otherwise (a tile of
// fp32 bits written to bf16) the upper half when the element was widened from the state (its raw
// bits come back, NaN payloads included), else round to nearest even, any NaN to the quiet NaN
// 0x7fc0.
template <typename BD, typename TT>
__device__ __forceinline__ BD from_tile(TT v, bool widened) {
    if constexpr (sizeof(BD) == sizeof(TT)) {
        return (BD)v;
    } else {
        const uint32_t u = (uint32_t)v;
        if (widened) return (BD)(u >> 16);
        if ((u & 0x7fffffffu) > 0x7f800000u) return (BD)0x7fc0u;
        return (BD)__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(u)));
    }
}
// Source element -> tile element: the same bits, or bf16 widened exactly to fp32 bits.
template <typename TT, typename BS>
__device__ __forceinline__ TT to_tile(BS v) {
    if constexpr (sizeof(TT) == sizeof(BS))
        return (TT)v;
    else
        return (TT)((uint32_t)v << 16);
}

// (converting writes: tile rows below state_rows hold the committed window, widened from the
// state's own type)
template <typename B, typename BD = B>
__device__ __forceinline__ void write_view(const B *__restrict__ tile, int pitch, int jofs, int ncol, BD *dst,
                                           long long ch_stride, long long col_stride, int nch, int state_rows = 0) {
    constexpr int CH = 16 / (int)sizeof(B);
    if constexpr (!std::is_same_v<B, BD>) {
        // converting writes: element by element in destination order
        const int n = nch * ncol;
        if (col_stride == 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int c = i / ncol, q = i - c * ncol;
                dst[c * ch_stride + q] = from_tile<BD>(tile[(jofs + q) * pitch + c], jofs + q < state_rows);
            }
        } else {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int q = i / nch, c = i - q * nch;
                dst[c * ch_stride + q * col_stride] = from_tile<BD>(tile[(jofs + q) * pitch + c], jofs + q < state_rows);
            }
        }
        return;
    } else {
    const int tid = threadIdx.x, NT = blockDim.x;
    const int n = nch * ncol;
    const bool aligned = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0);
    if (ch_stride == ncol && col_stride == 1 && aligned) {
        const int nchunks = (n + CH - 1) / CH;
        for (int m = tid; m < nchunks; m += NT) {
            const int pos = m * CH;
            int c = pos / ncol;
            int q = pos - c * ncol;
            uint32_t wv[4];
            B *vb = reinterpret_cast<B *>(wv);
#pragma unroll
            for (int e = 0; e < CH; ++e) {
                vb[e] = (pos + e < n) ? tile[(jofs + q) * pitch + c] : (B)0;
                if (++q == ncol) {
                    q = 0;
                    ++c;
                }
            }
            if (pos + CH <= n) {
                *reinterpret_cast<uint4 *>(dst + pos) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            } else {
                for (int e = 0; pos + e < n; ++e) dst[pos + e] = vb[e];
            }
        }
    } else if (ch_stride == 1 && aligned && ((col_stride * (long long)sizeof(B)) & 15) == 0) {
        const int nv = nch / CH;
        for (int i = tid; i < ncol * nv; i += NT) {
            const int q = i / nv, m = i - q * nv;
            *reinterpret_cast<uint4 *>(dst + q * col_stride + m * CH) =
                *reinterpret_cast<const uint4 *>(tile + (jofs + q) * pitch + m * CH);
        }
        const int rem = nch - nv * CH;
        for (int i = tid; i < ncol * rem; i += NT) {
            const int q = i / rem, c = nv * CH + (i - q * rem);
            dst[q * col_stride + c] = tile[(jofs + q) * pitch + c];
        }
    } else {
        for (int i = tid; i < n; i += NT) {
            const int q = i / nch, c = i - q * nch;
            dst[c * ch_stride + q * col_stride] = tile[(jofs + q) * pitch + c];
        }
    }
    }
}

// ---------------------------------------------------------------- verify
// BX: x, out, taps and bias; BS: state and snapshots.  When they differ (mixed dtypes) the tile
// holds fp32 bits: inputs are widened into it and snapshots are converted out of it.
template <typename BX, int W, typename BS = BX>
__global__ void __launch_bounds__(256) verify_generic(const __grid_constant__ VerifyParams p) {
    using B = BX;
    constexpr bool MIXED = !std::is_same_v<BX, BS>;
    using TT = std::conditional_t<MIXED, uint32_t, BX>;  // tile element
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;  // committed window columns
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TT *tile = reinterpret_cast<TT *>(smem_raw);

    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int BC = 8 * blockDim.x;
    const int c0 = blockIdx.x * BC;
    const int T = p.T, pitch = p.pitch;

    const int slot = p.cache_idx ? p.cache_idx[s] : s;
    const int off = p.state_off ? p.state_off[s] : 0;
    int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
    int Ts = T, row0 = 0;  // draft tokens of this sequence and (packed drafts) its first row
    if (p.cu_draft && slot >= 0) status |= draft_span(p.cu_draft, s, T, p.total_tokens, Ts, row0);
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;  // padded or rejected: touch nothing (uniform per block)
    if ((long long)(T + R) * pitch * (long long)sizeof(TT) > (long long)dynamic_smem_bytes()) return;  // launch mismatch

    const int nch = min(BC, p.dim - c0);
    const int cl = tid * 8;  // first block-local channel of this thread
    const int my = max(0, min(8, nch - cl));
    const bool full8 = (my == 8);

    // (1) x_0..x_{T-1} -> tile rows R..R+T-1 (asynchronous 16-byte copies, no registers)
    const B *xs = reinterpret_cast<const B *>(p.x) + (p.cu_draft ? (long long)row0 * p.x_tok : (long long)s * p.x_seq) + c0;
    if (MIXED) {
        for (int i = tid; i < Ts * nch; i += blockDim.x) {
            const int t = i / nch, c = i - t * nch;
            tile[(R + t) * pitch + c] = to_tile<TT>(xs[t * p.x_tok + c]);
        }
    } else if (p.x_vec) {
        if (full8) {
            for (int t = 0; t < Ts; ++t) {
#pragma unroll
                for (int i = 0; i < Oct<B>::NV; ++i)
                    cp_async16(tile + (R + t) * pitch + cl + i * (16 / sizeof(B)), xs + t * p.x_tok + cl + i * (16 / sizeof(B)));
            }
        } else {
            for (int t = 0; t < Ts; ++t)
                for (int e = 0; e < my; ++e) tile[(R + t) * pitch + cl + e] = to_tile<TT>(xs[t * p.x_tok + cl + e]);
        }
    } else {
        for (int i = tid; i < Ts * nch; i += blockDim.x) {
            const int t = i / nch, c = i - t * nch;
            tile[(R + t) * pitch + c] = to_tile<TT>(xs[t * p.x_tok + c]);
        }
    }

    // (2) committed window of this thread's channels -> registers and tile rows 0..R-1
    float win[R][8];
    {
        BS raw[R][8];
        BS *sp = reinterpret_cast<BS *>(p.state) + (long long)slot * p.st_slot + (long long)(c0 + cl) * p.st_ch +
                 (long long)off * p.st_col;
        if (full8 && p.st_vec && off == 0) {
            // 8 channels x R columns are contiguous: R 16-byte vectors (2R for fp32)
            Oct<BS> o[R];
#pragma unroll
            for (int k = 0; k < R; ++k) load_oct(o[k], sp + k * 8);
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const int lin = e * R + k;
                    raw[k][e] = o[lin / 8].get(lin % 8);
                }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) raw[k][e] = (e < my) ? sp[e * p.st_ch + k * p.st_col] : (BS)0;
        }
#pragma unroll
        for (int k = 0; k < R; ++k) {
            if (full8 && !MIXED) {
                Oct<TT> o;
#pragma unroll
                for (int e = 0; e < 8; ++e) o.set(e, (TT)raw[k][e]);
                store_oct(tile + k * pitch + cl, o);
            } else {
                for (int e = 0; e < my; ++e) tile[k * pitch + cl + e] = to_tile<TT>(raw[k][e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) win[k][e] = widen<BS>(raw[k][e]);
        }
    }

    // (3) taps and bias of this thread's channels
    float wt[8][W];
    float bs[8];
    {
        const B *wp = reinterpret_cast<const B *>(p.weight) + (long long)(c0 + cl) * W;
        if (full8 && p.w_vec) {
            Oct<B> o[W];
#pragma unroll
            for (int i = 0; i < W; ++i) load_oct_nc(o[i], wp + i * 8);
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int j = 0; j < W; ++j) {
                    const int lin = e * W + j;
                    wt[e][j] = widen<B>(o[lin / 8].get(lin % 8));
                }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int j = 0; j < W; ++j) wt[e][j] = (e < my) ? widen<B>(wp[e * W + j]) : 0.0f;
        }
        const B *bp = reinterpret_cast<const B *>(p.bias);
        if (bp && full8 && p.b_vec) {
            Oct<B> o;
            load_oct_nc(o, bp + c0 + cl);
#pragma unroll
            for (int e = 0; e < 8; ++e) bs[e] = widen<B>(o.get(e));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) bs[e] = (bp && e < my) ? widen<B>(bp[c0 + cl + e]) : 0.0f;
        }
    }

    if (p.x_vec) cp_async_wait_all();
    __syncthreads();

    // (4) snapshots and committed window, written from the tile in destination order
    if (p.recomp) {
        // recompute rollback: outputs only; the state keeps the pre-verify window
    } else if (p.hist) {
        // history-row state: the snapshot row [full[1 .. W-2], x_0 .. x_{T-1}] replaces columns
        // [0, T+W-2) of the state row (every thread read its committed window before the barrier)
        // (no draft token, no snapshot: a packed sequence with T_s = 0 writes nothing here)
        BS *sb = reinterpret_cast<BS *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * p.st_ch;
        if (Ts > 0) write_view<TT, BS>(tile, pitch, 1, Ts + R - 1, sb, p.st_ch, p.st_col, nch, R);
    } else {
        BS *wb = reinterpret_cast<BS *>(p.win) + (long long)s * p.w_seq;
        if (p.dedup) {
            if (Ts > 0)
                write_view<TT, BS>(tile, pitch, 1, Ts + R - 1, wb + (long long)c0 * p.w_ch, p.w_ch, p.w_col, nch, R);
        } else {
            for (int t = 0; t < Ts; ++t)
                write_view<TT, BS>(tile, pitch, t + 1, R, wb + t * p.w_step + (long long)c0 * p.w_ch, p.w_ch, p.w_col,
                                   nch, R);
        }
        BS *sb = reinterpret_cast<BS *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * p.st_ch;
        write_view<TT, BS>(tile, pitch, Ts, R, sb, p.st_ch, 1, nch, R);
    }

    // (5) conv + SiLU (+ L2 over the head_dim group) for every token, outputs stored as vectors
    const bool has_bias = (p.bias != nullptr);
    const bool l2_block = (c0 < p.qk_channels);       // block-uniform
    const bool l2_mine = (c0 + cl) < p.qk_channels;   // whole 8-channel group is q|k or V
    const int lanes = p.head_dim >> 3;                // 1..32 threads per group
    B *ob = reinterpret_cast<B *>(p.out) + (p.cu_draft ? (long long)row0 * p.out_tok : (long long)s * p.out_seq) + c0 + cl;
    for (int t = 0; t < Ts; ++t) {
        float xv[8];
        if (full8) {
            Oct<TT> o;
            load_oct(o, tile + (R + t) * pitch + cl);
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = widen<TT>(o.get(e));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = (e < my) ? widen<TT>(tile[(R + t) * pitch + cl + e]) : 0.0f;
        }
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            // the same chain as conv_chain: bias, then the taps in order
            float in[W];
#pragma unroll
            for (int j = 0; j < R; ++j) in[j] = win[j][e];
            in[R] = xv[e];
            // (mixed dtypes: fp32 state values make the products inexact, so each one is rounded)
            const float acc = conv_chain<std::conditional_t<MIXED, uint32_t, B>, W>(has_bias ? bs[e] : 0.0f, wt[e], in);
            y[e] = silu(acc);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
#pragma unroll
            for (int j = 0; j + 1 < R; ++j) win[j][e] = win[j + 1][e];
            win[R - 1][e] = xv[e];
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
        B *op = ob + t * p.out_tok;
        if (full8 && p.out_vec) {
            Oct<B> o;
#pragma unroll
            for (int e = 0; e < 8; ++e) o.set(e, narrow<B>(y[e]));
            store_oct(op, o);
        } else {
            for (int e = 0; e < my; ++e) op[e] = narrow<B>(y[e]);
        }
    }
}

}  // namespace cvk
