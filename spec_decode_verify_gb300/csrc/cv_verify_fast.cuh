// Verify kernel for the packed layouts (the fast path).
//
// Launch: grid (ceil(dim / (CPT*threads)), n_seq), one block per (channel block, sequence) as in
// the Atlas batched verify (fn gdn_verify_fused_conv_kn_batched, grid (ceil(d_inner/256), n_seq)).
// Each thread owns CPT consecutive channels (4 or 8), so x, out, state and weights move as 8- or
// 16-byte vectors and every warp access is contiguous.  Per block:
//   1. loads: the committed window, all T draft inputs (T independent vector loads in flight per
//      thread), taps and bias -- straight into registers;
//   2. everything that depends on the inputs only is written first, so its registers die early and
//      its stores overlap the arithmetic:
//        - deduplicated row (sglang PR #46184: the W-1 columns from column t of
//          [state[1..W-2], x_0..x_{T-1}] form the window of step t): each thread assembles its CPT channels x (T+W-2)
//          columns in registers by a static permutation and stages them in shared memory; ONE bulk
//          copy (TMA, cp.async.bulk) then writes the block's channels*(T+W-2) contiguous elements,
//          instead of W-1 scattered stores per token;
//        - dense snapshots: the thread's CPT x (W-1) run per token as vector stores;
//        - committed window (= snapshot T-1) -> state columns [0, W-1), staged and bulk-copied
//          when the state rows are packed.  Rows wider than the window (read at a state offset),
//          when packed, are staged whole in shared memory (cp.async, 16-byte pieces) at the start
//          and leave whole by one bulk copy with the window in their first W-1 columns (the other
//          columns go back with their own bits): one contiguous run per block instead of 2-byte
//          loads and stores at the row pitch;
//   3. conv (fp32, bias first, taps in order, see conv_chain), SiLU, and for
//      q|k channels the L2 normalisation over the head_dim group as an xor-shuffle over
//      head_dim/CPT lanes (glm5next_kda mod.rs: SiLU after the conv, then L2 on q and k alone,
//      eps inside the root); one rounding to the output type; vector stores.
// T is a template parameter for T <= 17 (bf16) / 8 (fp32), which unrolls the token loop and makes
// the row permutation static; TS = 0 runs any T with a dense window in unrolled chunks of 4, and
// may split the tokens among blockDim.y thread groups (small batches, where one group per block
// would leave the SMs with too few warps): group g takes tokens [g*TH, min(T, (g+1)*TH)), TH =
// ceil(T / groups), starting from the W-1 x rows before them (group 0: the committed window); the
// group holding token T-1 writes the committed window.  Each warp stays within one group, so the
// L2 shuffles see one token's channels.
// Preconditions (checked on the host): dim % 8 == 0; x, out, weight, bias, window 16-byte aligned
// with 16-byte-multiple strides; window packed (dense [.., T, dim, W-1] or dedup [.., dim, T+W-2]
// with unit column stride); TS = 0 only with the dense layout; head_dim / CPT <= 32.
#pragma once

#include <type_traits>

#include "cv_device.cuh"

namespace cvk {

// Alignment (8 or 16 bytes) of a per-thread chunk of `bytes` bytes whose start is a multiple of it.
__host__ __device__ constexpr int chunk_align(int bytes) { return bytes % 16 == 0 ? 16 : 8; }

template <typename B, int W, int TS, int CPT>
__global__ void __launch_bounds__(256) verify_fast(const __grid_constant__ VerifyParams p) {
    // Before waiting for the previous grid: L2 prefetch hints for the block's x rows and state run.
    // The cache slot is read through L2 only and only to form a hint's address (inside the state
    // buffer); all data is read after the wait.
    if (threadIdx.x == 0 && threadIdx.y == 0) {
        const int bc = CPT * (int)blockDim.x, cb0 = (int)blockIdx.x * bc, sq = (int)blockIdx.y;
        const int n = min(bc, p.dim - cb0), es = (int)sizeof(B);
        prefetch_runs_l2(reinterpret_cast<const B *>(p.x) + (long long)sq * p.x_seq + cb0, p.x_tok * es,
                         TS > 0 ? TS : p.T, (long long)n * es);
        const int sl = p.cache_idx ? __ldcg(p.cache_idx + sq) : sq;
        if (sl >= 0 && sl < p.n_slots && (p.st_vec || p.st_rows))
            prefetch_runs_l2(reinterpret_cast<const B *>(p.state) + (long long)sl * p.st_slot + (long long)cb0 * p.state_cols,
                             0, 1, (long long)n * p.state_cols * es);
    }
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;                  // committed window columns
    constexpr int TC = TS > 0 ? TS : 4;       // tokens held in registers at a time
    constexpr int ES = (int)sizeof(B);        // element bytes
    constexpr int EW = 4 / ES;                // elements per 32-bit word
    constexpr int NW = CPT / EW;              // words per thread vector (CPT elements)
    constexpr int VX = chunk_align(CPT * ES);      // x / out / bias vectors
    constexpr int VS = chunk_align(CPT * R * ES);  // committed window run
    constexpr int VW = chunk_align(CPT * W * ES);  // taps
    extern __shared__ __align__(128) unsigned char smem[];

    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const bool lead = threadIdx.x == 0 && threadIdx.y == 0;  // issues the block's bulk copies
    const int BC = CPT * blockDim.x;
    const int c0 = blockIdx.x * BC;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int off = p.state_off ? __ldg(p.state_off + s) : 0;
    const int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
    if (p.err && blockIdx.x == 0 && lead) p.err[s] = status;
    if (slot < 0 || status) return;  // padded or rejected: nothing is written (block-uniform)

    const int nch = min(BC, p.dim - c0);  // a multiple of 8 on this path
    const int cl = tid * CPT;
    const bool act = cl < nch;
    const int c = c0 + cl;
    const int T = TS > 0 ? TS : p.T;
    const bool dense = !p.dedup;
    // token groups (TS = 0 only): this thread's group takes tokens [tb, te)
    const int G = TS > 0 ? 1 : (int)blockDim.y, g = TS > 0 ? 0 : (int)threadIdx.y;
    const int TH = (T + G - 1) / G;
    const int tb = min(T, g * TH), te = min(T, tb + TH);
    const bool last_group = tb < te && te == T;  // holds token T-1: writes the committed window
    // shared memory: [dedup image: BC x (TS+W-2)] then the state part: the committed-window image
    // (BC x (W-1)) or, for staged wide rows, the rows themselves (BC x state_cols)
    const bool rows = p.st_rows;  // block-uniform
    const int SC = p.state_cols;
    const long long img_bytes = (TS > 0 && !dense) ? (long long)BC * (TS + R - 1) * ES : 0;
    if (img_bytes + (long long)BC * (rows ? SC : R) * ES > (long long)dynamic_smem_bytes()) return;  // launch mismatch
    unsigned char *st_img = smem + img_bytes;
    B *const st_blk = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * SC;
    if (rows && g == 0) {
        // the block's [nch][SC] rows: contiguous, 16-byte aligned, a multiple of 16 bytes (host-checked)
        const int nbytes = nch * SC * ES;
        for (int o = tid * 16; o < nbytes; o += (int)blockDim.x * 16)
            cp_async16(st_img + o, reinterpret_cast<const unsigned char *>(st_blk) + o);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    }

    // ---- 1. loads.  fw[e][j] = input j of channel e widened to fp32 (j < R: committed window).
    float fw[CPT][R + TC];
    uint32_t xr[TC][NW];  // raw inputs of the current chunk
    B *const st_row = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
    const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c;
#pragma unroll
    for (int e = 0; e < CPT; ++e)
#pragma unroll
        for (int k = 0; k < R; ++k) fw[e][k] = 0.0f;
    if (act && g > 0) {
        // a later token group starts from the W-1 x rows before its first token (tb >= W-1, host)
#pragma unroll
        for (int k = 0; k < R; ++k) {
            uint32_t hw[NW];
            ldv<VX, NW>(hw, xs + (long long)(tb - R + k) * p.x_tok);
#pragma unroll
            for (int e = 0; e < CPT; ++e) fw[e][k] = elem_f<B>(hw, e);
        }
    } else if (act && !rows) {
        if (p.st_vec) {  // packed [dim][R] rows (then the offset is 0)
            uint32_t sw[R * NW];
            ldv<VS, R * NW>(sw, st_row);
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = elem_f<B>(sw, e * R + k);
        } else {
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = widen<B>(st_row[e * p.st_ch + off + k]);
        }
    }

    auto load_chunk = [&](int t0) {
#pragma unroll
        for (int u = 0; u < TC; ++u) {
#pragma unroll
            for (int i = 0; i < NW; ++i) xr[u][i] = 0u;
            if (act && (TS > 0 || t0 + u < te)) ldv<VX, NW>(xr[u], xs + (long long)(t0 + u) * p.x_tok);
        }
    };
    load_chunk(tb);

    float wt[CPT][W];
    float bs[CPT];
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
        bs[e] = 0.0f;
#pragma unroll
        for (int j = 0; j < W; ++j) wt[e][j] = 0.0f;
    }
    if (act) {
        uint32_t ww[W * NW];
        ldv<VW, W * NW>(ww, reinterpret_cast<const B *>(p.weight) + (long long)c * W);
#pragma unroll
        for (int e = 0; e < CPT; ++e)
#pragma unroll
            for (int j = 0; j < W; ++j) wt[e][j] = elem_f<B>(ww, e * W + j);
        if (p.bias) {
            uint32_t bw[NW];
            ldv<VX, NW>(bw, reinterpret_cast<const B *>(p.bias) + c);
#pragma unroll
            for (int e = 0; e < CPT; ++e) bs[e] = elem_f<B>(bw, e);
        }
    }
    const B *const srow_img = reinterpret_cast<const B *>(st_img) + (size_t)cl * SC;  // staged rows
    if (rows) {
        cp_async_wait_all();
        __syncthreads();
        if (act && g == 0) {
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = widen<B>(srow_img[e * SC + off + k]);
        }
        // (the last group writes the new window over the rows' first columns later)
        if (G > 1) __syncthreads();
    }

    B *wseq = reinterpret_cast<B *>(p.win) + (long long)s * p.w_seq;
    B *os = reinterpret_cast<B *>(p.out) + (long long)s * p.out_seq + c;
    const bool l2_block = c0 < p.qk_channels;  // block-uniform
    const bool l2_mine = c < p.qk_channels;    // the thread's channels are all q|k or all V
    const int lanes = p.head_dim / CPT;        // threads per L2 group (1..32)

    // Raw bits of input j of channel e within the current chunk: j < R is the carried window,
    // j >= R is x of chunk token j - R.
    auto raw_in = [&](int e, int j) -> uint32_t { return j < R ? raw_of<B>(fw[e][j]) : elem_raw<B>(xr[j - R], e); };
    // Words of the [CPT][R] channel-major run holding inputs j0 .. j0+R-1 of the thread's channels.
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
        stv<VS, R * NW>(wseq + (long long)t * p.w_step + (long long)c * R, w);
    };
    // conv + SiLU of chunk token u into y[u] (fw[e][R+u] <- x_u first)
    auto conv_token = [&](int u, float *yu) {
#pragma unroll
        for (int e = 0; e < CPT; ++e) fw[e][R + u] = elem_f<B>(xr[u], e);
        float acc[CPT];
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
            acc[e] = conv_chain<B, W>(bs[e], wt[e], &fw[e][u]);
        }
        silu_run<CPT>(acc, yu);
    };
    // L2 of NT tokens at once: the NT xor-shuffle trees are independent, so they overlap
    auto l2_tokens = [&](auto &y, auto nt_tag) {
        constexpr int NTOK = decltype(nt_tag)::value;
        if (!l2_block) return;
        float ss[NTOK];
#pragma unroll
        for (int u = 0; u < NTOK; ++u) ss[u] = sum_squares<CPT>(y[u]);
        // same association as 8 channels per thread: with 4 per thread the neighbour lane holds the
        // other half of the 8-channel run, so it is added first
        if (CPT == 4 && lanes > 1) {
#pragma unroll
            for (int u = 0; u < NTOK; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], 1);
        }
        for (int o = lanes >> 1; o >= (CPT == 4 ? 2 : 1); o >>= 1) {
#pragma unroll
            for (int u = 0; u < NTOK; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
        }
        if (l2_mine) {
#pragma unroll
            for (int u = 0; u < NTOK; ++u) {
                const float r = rsqrtf(ss[u] + p.eps);
#pragma unroll
                for (int e = 0; e < CPT; ++e) y[u][e] *= r;
            }
        }
    };
    auto store_token = [&](int t, const float *yu) {
        if (!act) return;
        uint32_t ow[NW];
        if (ES == 2) {
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                __nv_bfloat162 h = __floats2bfloat162_rn(yu[2 * i], yu[2 * i + 1]);
                ow[i] = *reinterpret_cast<uint32_t *>(&h);
            }
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i) ow[i] = __float_as_uint(yu[i]);
        }
        stv<VX, NW>(os + (long long)t * p.out_tok, ow);
    };
    auto stage_state = [&](const uint32_t *fin) {
        if (p.st_vec) {
            stv<VS, R * NW>(st_img + (size_t)tid * CPT * R * ES, fin);
        } else if (rows) {
            // into the staged rows, in place: this thread's own channels, read above
            B *const rr = reinterpret_cast<B *>(st_img) + (size_t)cl * SC;
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) rr[e * SC + k] = (B)elem_raw<B>(fin, e * R + k);
        } else {
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) st_row[e * p.st_ch + k] = (B)elem_raw<B>(fin, e * R + k);
        }
    };

    bool bulk = false;
    if constexpr (TS > 0) {
        constexpr int Q = TS + R - 1;  // dedup row columns
        constexpr int VI = chunk_align(CPT * Q * ES);
        // ---- 2. input-only outputs
        if (act) {
            if (!dense) {
                uint32_t img[Q * NW];  // the thread's CPT x Q image, channel-major
#pragma unroll
                for (int word = 0; word < Q * NW; ++word) {
                    uint32_t bits[2] = {0u, 0u};
#pragma unroll
                    for (int z = 0; z < EW; ++z) {
                        const int idx = word * EW + z;  // element (e, q) of the thread's image
                        bits[z] = raw_in(idx / Q, idx % Q + 1);
                    }
                    img[word] = (ES == 2) ? pack_halves(bits[0], bits[1]) : bits[0];
                }
                stv<VI, Q * NW>(smem + (size_t)tid * CPT * Q * ES, img);
            } else {
#pragma unroll
                for (int t = 0; t < TS; ++t) write_snapshot(t, t + 1);
            }
            uint32_t fin[R * NW];
            window_words(TS, fin);
            stage_state(fin);
        }
        bulk = !dense || p.st_vec || rows;
        if (bulk) {
            fence_smem_to_async();
            __syncthreads();
            if (lead) {
                if (!dense) bulk_store(wseq + (long long)c0 * Q, smem, (unsigned)(nch * Q * ES));
                if (p.st_vec || rows) bulk_store(st_blk, st_img, (unsigned)(nch * SC * ES));
                asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            }
        }
        // ---- 3. arithmetic
        float y[TS][CPT];
#pragma unroll
        for (int u = 0; u < TS; ++u) conv_token(u, y[u]);
        l2_tokens(y, std::integral_constant<int, TS>{});
#pragma unroll
        for (int u = 0; u < TS; ++u) store_token(u, y[u]);
    } else {
        // chunked: any T, dense window; this group's tokens [tb, te)
        uint32_t fin[R * NW];
#pragma unroll
        for (int i = 0; i < R * NW; ++i) fin[i] = 0u;
        for (int t0 = tb; t0 < te; t0 += TC) {
            if (t0 > tb) load_chunk(t0);
#pragma unroll
            for (int u = 0; u < TC; ++u) {
                if (t0 + u < te) {
                    if (act) write_snapshot(t0 + u, u + 1);
                    if (t0 + u == T - 1) window_words(u + 1, fin);
                }
            }
            float y[TC][CPT];
#pragma unroll
            for (int u = 0; u < TC; ++u)
                if (t0 + u < te) conv_token(u, y[u]);
            l2_tokens(y, std::integral_constant<int, TC>{});
#pragma unroll
            for (int u = 0; u < TC; ++u)
                if (t0 + u < te) store_token(t0 + u, y[u]);
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int k = 0; k < R; ++k) fw[e][k] = fw[e][TC + k];
        }
        if (act && last_group) stage_state(fin);
        bulk = p.st_vec || rows;
        if (bulk) {
            fence_smem_to_async();
            __syncthreads();
            if (lead) {
                bulk_store(st_blk, st_img, (unsigned)(nch * SC * ES));
                asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            }
        }
    }
    // the issuing thread keeps the block's shared memory alive until the bulk copies have read it
    if (bulk && lead) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

}  // namespace cvk
