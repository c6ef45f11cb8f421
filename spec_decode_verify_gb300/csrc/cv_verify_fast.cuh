// Verify kernel for the packed layouts (the fast path).
//
// Launch: grid (ceil(dim / (8*threads)), n_seq), one block per (channel block, sequence) as in the
// Atlas batched verify (fn gdn_verify_fused_conv_kn_batched, grid (ceil(d_inner/256), n_seq)).
// Each thread owns 8 consecutive channels, so x, out, state and weights move as 16-byte vectors and
// every warp access is 512 contiguous bytes.  Per block:
//   1. loads: the committed window, all T draft inputs (T independent 16-byte loads in flight per
//      thread), taps and bias -- straight into registers;
//   2. everything that depends on the inputs only is written first, so its registers die early and
//      its stores overlap the arithmetic:
//        - deduplicated row (sglang PR #46184: step t's window is columns t..t+W-2 of
//          [state[1..W-2], x_0..x_{T-1}]): each thread assembles its 8 channels x (T+W-2) columns
//          in registers by a static permutation and stages them in shared memory; ONE bulk copy
//          (TMA, cp.async.bulk) then writes the block's channels*(T+W-2) contiguous elements,
//          instead of W-1 scattered stores per token;
//        - dense snapshots: W-1 16-byte vectors per thread and token;
//        - committed window (= snapshot T-1) -> state columns [0, W-1), staged and bulk-copied
//          when the state rows are packed;
//   3. conv (fp32, bias first, taps in order, each product rounded before its add), SiLU, and for
//      q|k channels the L2 normalisation over the head_dim group as an xor-shuffle over
//      head_dim/8 lanes (glm5next_kda mod.rs: conv1d + SiLU -> L2(q,k only), eps inside the
//      root); one rounding to the output type; 16-byte stores.
// T is a template parameter for T <= 16 (bf16) / 8 (fp32), which unrolls the token loop and makes
// the row permutation static; TS = 0 runs any T with a dense window in unrolled chunks of 4.
// Preconditions (checked on the host): dim % 8 == 0; x, out, weight, bias, window 16-byte aligned
// with 16-byte-multiple strides; window packed (dense [.., T, dim, W-1] or dedup [.., dim, T+W-2]
// with unit column stride); TS = 0 only with the dense layout.
#pragma once

#include "cv_device.cuh"

namespace cvk {

template <typename B, int W, int TS>
__global__ void __launch_bounds__(128, (TS > 8 || sizeof(B) == 4) ? 2 : 4)
    verify_fast(const __grid_constant__ VerifyParams p) {
    constexpr int R = W - 1;                    // committed window columns
    constexpr int TC = TS > 0 ? TS : 4;         // tokens held in registers at a time
    constexpr int ES = (int)sizeof(B);          // element bytes
    constexpr int EW = 4 / ES;                  // elements per 32-bit word
    constexpr int NW = 8 / EW;                  // words per 8 elements
    constexpr int NV = NW / 4;                  // 16-byte vectors per 8 elements
    constexpr int VE = 16 / ES;                 // elements per 16-byte vector
    extern __shared__ __align__(128) unsigned char smem[];

    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int BC = 8 * blockDim.x;
    const int c0 = blockIdx.x * BC;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int off = p.state_off ? __ldg(p.state_off + s) : 0;
    const int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;  // padded or rejected: nothing is written (block-uniform)

    const int nch = min(BC, p.dim - c0);  // a multiple of 8 on this path
    const int cl = tid * 8;
    const bool act = cl < nch;
    const int c = c0 + cl;
    const int T = TS > 0 ? TS : p.T;
    const bool dense = !p.dedup;

    // ---- 1. loads.  fw[e][j] = input j of channel e widened to fp32 (j < R: committed window).
    float fw[8][R + TC];
    uint32_t xr[TC][NW];  // raw inputs of the current chunk
    B *const st_row = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
    const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c;
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int k = 0; k < R; ++k) fw[e][k] = 0.0f;
    if (act) {
        if (p.st_vec) {  // packed [dim][R] rows (then the offset is 0): R*NV vectors
            uint32_t sw[R * NW];
#pragma unroll
            for (int v = 0; v < R * NV; ++v) {
                const uint4 q = ld16(st_row + v * VE);
                sw[4 * v] = q.x, sw[4 * v + 1] = q.y, sw[4 * v + 2] = q.z, sw[4 * v + 3] = q.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = elem_f<B>(sw, e * R + k);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = widen<B>(st_row[e * p.st_ch + off + k]);
        }
    }

    auto load_chunk = [&](int t0) {
#pragma unroll
        for (int u = 0; u < TC; ++u) {
#pragma unroll
            for (int i = 0; i < NW; ++i) xr[u][i] = 0u;
            if (act && (TS > 0 || t0 + u < T)) {
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const uint4 q = ld16(xs + (long long)(t0 + u) * p.x_tok + v * VE);
                    xr[u][4 * v] = q.x, xr[u][4 * v + 1] = q.y, xr[u][4 * v + 2] = q.z, xr[u][4 * v + 3] = q.w;
                }
            }
        }
    };
    load_chunk(0);

    float wt[8][W];
    float bs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        bs[e] = 0.0f;
#pragma unroll
        for (int j = 0; j < W; ++j) wt[e][j] = 0.0f;
    }
    if (act) {
        const B *wp = reinterpret_cast<const B *>(p.weight) + (long long)c * W;
        uint32_t ww[W * NW];
#pragma unroll
        for (int v = 0; v < W * NV; ++v) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(wp + v * VE));
            ww[4 * v] = q.x, ww[4 * v + 1] = q.y, ww[4 * v + 2] = q.z, ww[4 * v + 3] = q.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int j = 0; j < W; ++j) wt[e][j] = elem_f<B>(ww, e * W + j);
        if (p.bias) {
            uint32_t bw[NW];
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const uint4 q = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const B *>(p.bias) + c + v * VE));
                bw[4 * v] = q.x, bw[4 * v + 1] = q.y, bw[4 * v + 2] = q.z, bw[4 * v + 3] = q.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) bs[e] = elem_f<B>(bw, e);
        }
    }

    B *wseq = reinterpret_cast<B *>(p.win) + (long long)s * p.w_seq;
    B *os = reinterpret_cast<B *>(p.out) + (long long)s * p.out_seq + c;
    const bool l2_block = c0 < p.qk_channels;  // block-uniform
    const bool l2_mine = c < p.qk_channels;    // the thread's 8 channels are all q|k or all V
    const int lanes = p.head_dim >> 3;         // threads per L2 group (1..32)

    // Raw bits of input j of channel e within the current chunk: j < R is the carried window,
    // j >= R is x of chunk token j - R.
    auto raw_in = [&](int e, int j) -> uint32_t { return j < R ? raw_of<B>(fw[e][j]) : elem_raw<B>(xr[j - R], e); };
    // Words of the [8][R] channel-major run holding inputs j0 .. j0+R-1 of the thread's channels.
    auto window_words = [&](int j0, uint32_t *w) {
#pragma unroll
        for (int i = 0; i < R * NW; ++i) {
            if (ES == 2) {
                const int a = 2 * i, b = 2 * i + 1;
                w[i] = pack_halves(raw_in(a / R, j0 + a % R), raw_in(b / R, j0 + b % R));
            } else {
                w[i] = raw_in(i / R, j0 + i % R);
            }
        }
    };
    auto write_snapshot = [&](int t, int j0) {  // dense snapshot t = inputs j0 .. j0+R-1 of the chunk
        uint32_t w[R * NW];
        window_words(j0, w);
        B *dp = wseq + (long long)t * p.w_step + (long long)c * R;
#pragma unroll
        for (int v = 0; v < R * NV; ++v) st16(dp + v * VE, make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]));
    };
    auto compute_token = [&](int t, int u) {
#pragma unroll
        for (int e = 0; e < 8; ++e) fw[e][R + u] = elem_f<B>(xr[u], e);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = bs[e];
#pragma unroll
            for (int j = 0; j < W; ++j) acc = __fadd_rn(acc, __fmul_rn(wt[e][j], fw[e][u + j]));
            y[e] = silu(acc);
        }
        if (l2_block) {
            float ss = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(y[e], y[e], ss);
            for (int o = lanes >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (l2_mine) {
                const float r = rsqrtf(ss + p.eps);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] *= r;
            }
        }
        if (act) {
            uint32_t ow[NW];
            if (ES == 2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
                    ow[i] = *reinterpret_cast<uint32_t *>(&h);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) ow[i] = __float_as_uint(y[i]);
            }
#pragma unroll
            for (int v = 0; v < NV; ++v)
                st16(os + (long long)t * p.out_tok + v * VE, make_uint4(ow[4 * v], ow[4 * v + 1], ow[4 * v + 2], ow[4 * v + 3]));
        }
    };

    bool bulk = false;
    if constexpr (TS > 0) {
        constexpr int Q = TS + R - 1;  // dedup row columns
        // ---- 2. input-only outputs
        unsigned char *st_img = dense ? smem : smem + (size_t)BC * Q * ES;
        if (act) {
            if (!dense) {
                unsigned char *my = smem + (size_t)tid * Q * NV * 16;
#pragma unroll
                for (int v = 0; v < Q * NV; ++v) {
                    uint32_t wv[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        uint32_t bits[2] = {0u, 0u};
#pragma unroll
                        for (int z = 0; z < EW; ++z) {
                            const int idx = (4 * v + h) * EW + z;  // element (e, q) of the thread's image
                            bits[z] = raw_in(idx / Q, idx % Q + 1);
                        }
                        wv[h] = (ES == 2) ? pack_halves(bits[0], bits[1]) : bits[0];
                    }
                    st16(my + v * 16, make_uint4(wv[0], wv[1], wv[2], wv[3]));
                }
            } else {
#pragma unroll
                for (int t = 0; t < TS; ++t) write_snapshot(t, t + 1);
            }
            uint32_t fin[R * NW];
            window_words(TS, fin);
            if (p.st_vec) {
                unsigned char *my = st_img + (size_t)tid * R * NV * 16;
#pragma unroll
                for (int v = 0; v < R * NV; ++v) st16(my + v * 16, make_uint4(fin[4 * v], fin[4 * v + 1], fin[4 * v + 2], fin[4 * v + 3]));
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int k = 0; k < R; ++k) st_row[e * p.st_ch + k] = (B)elem_raw<B>(fin, e * R + k);
            }
        }
        bulk = !dense || p.st_vec;
        if (bulk) {
            fence_smem_to_async();
            __syncthreads();
            if (tid == 0) {
                if (!dense) bulk_store(wseq + (long long)c0 * Q, smem, (unsigned)(nch * Q * ES));
                if (p.st_vec)
                    bulk_store(reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * R, st_img,
                               (unsigned)(nch * R * ES));
                asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            }
        }
        // ---- 3. arithmetic
#pragma unroll
        for (int u = 0; u < TS; ++u) compute_token(u, u);
    } else {
        // chunked: any T, dense window
        uint32_t fin[R * NW];
#pragma unroll
        for (int i = 0; i < R * NW; ++i) fin[i] = 0u;
        for (int t0 = 0; t0 < T; t0 += TC) {
            if (t0 > 0) load_chunk(t0);
#pragma unroll
            for (int u = 0; u < TC; ++u) {
                if (t0 + u < T) {
                    if (act) write_snapshot(t0 + u, u + 1);
                    if (t0 + u == T - 1) window_words(u + 1, fin);
                }
            }
#pragma unroll
            for (int u = 0; u < TC; ++u)
                if (t0 + u < T) compute_token(t0 + u, u);
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = fw[e][TC + k];
        }
        if (act) {
            if (p.st_vec) {
                unsigned char *my = smem + (size_t)tid * R * NV * 16;
#pragma unroll
                for (int v = 0; v < R * NV; ++v) st16(my + v * 16, make_uint4(fin[4 * v], fin[4 * v + 1], fin[4 * v + 2], fin[4 * v + 3]));
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int k = 0; k < R; ++k) st_row[e * p.st_ch + k] = (B)elem_raw<B>(fin, e * R + k);
            }
        }
        bulk = p.st_vec;
        if (bulk) {
            fence_smem_to_async();
            __syncthreads();
            if (tid == 0) {
                bulk_store(reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * R, smem,
                           (unsigned)(nch * R * ES));
                asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            }
        }
    }
    // the issuing thread keeps the block's shared memory alive until the bulk copies have read it
    if (bulk && tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

}  // namespace cvk
