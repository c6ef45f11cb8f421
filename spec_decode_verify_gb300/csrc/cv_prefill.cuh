// Prefill conv over packed variable-length sequences.
//
// glm5next_kda mod.rs (the layer's prefill path): the causal depthwise conv with SiLU over every
// prompt token, then the L2 normalisation of the q|k channels per head_dim group.  Here the
// normalisation is fused and applied to the fp32 SiLU values before the single rounding, exactly
// as the verify kernels do (the same conv chain, SiLU, sum order and shuffle tree), so a prompt
// gives bit for bit the outputs a verify over the same tokens gives.
//
// The conv needs only the W-1 inputs before each token, so the work is a stencil in time: block
// (channel block, chunk, sequence) covers a chunk of tokens of one sequence (the host picks its
// length, 32..128) for CPT*threads channels.  Its halo is the sequence's initial window (the cached state, or zeros without one)
// for the first chunk and the W-1 x rows before the chunk otherwise (a chunk is at least W-1
// tokens long).  Each thread keeps its channels' window in registers and walks the chunk 8 tokens
// at a time.  With aligned rows it stages its own pieces of the next x rows in a shared-memory ring
// by cp.async, 3 batches ahead, while this batch's conv + SiLU, batched L2 shuffle trees, rounding
// and stores run (otherwise the next batch's rows are loaded into registers).  The launch bounds
// hold a thread to 128 registers (4 blocks, 16 warps per SM), which beat more registers with fewer
// warps, fewer registers with more warps, smaller batches with more warps, and a bulk-copy ring of
// staged rows when timed; ring depths of 2 / 3 / 4 batches measured 262.1 / 262.9 / 260.8 us on
// 30,822 tokens at dim 10240, against 267.1 with registers only.  The first chunk's block also writes the
// final window -- the last W-1 entries of [initial window, x] -- into the state: it is the only
// block that reads the initial window, so no other block races with that write.
#pragma once

#include "cv_device.cuh"

namespace cvk {

constexpr int kPrefillBatch = 8;  // tokens per batch; the next batch's rows load during this one
constexpr int kPrefillRing = 4;   // batches of x rows staged in shared memory: 3 in flight, 1 in use

// cp.async of BYTES (8 or 16) into shared memory, zero-filled past src_bytes (0: nothing is read)
template <int BYTES>
__device__ __forceinline__ void prefill_cp_async(void *dst, const void *src, unsigned src_bytes) {
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(smem_u32(dst)), "l"(src), "n"(BYTES),
                     "r"(src_bytes)
                     : "memory");
}

template <typename B, int W, int CPT>
__global__ void __launch_bounds__(128, CPT == 4 ? 4 : 2) prefill_conv(const __grid_constant__ PrefillParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int EW = 4 / ES;
    constexpr int NW = CPT / EW;
    constexpr int VX = (CPT * ES) % 16 == 0 ? 16 : 8;
    constexpr int U = kPrefillBatch;

    const int s = blockIdx.z;
    const int chunk = blockIdx.y;
    const int tid = threadIdx.x;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int b = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
    int status = 0;
    if (slot >= 0) {
        if (slot >= p.n_slots) status |= 1;
        if (b < 0 || e < b || e > p.total_tokens || e - b > p.max_seqlen) status |= kSeqBadSpan;
    }
    if (p.err && chunk == 0 && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;
    const int L = e - b;
    const int CH = p.chunk;  // tokens per block: a multiple of the batch, at least W-1 (host)
    const int t0 = chunk * CH;
    if (t0 >= L && chunk > 0) return;
    const int t1 = min(L, t0 + CH);

    const int c = (blockIdx.x * blockDim.x + tid) * CPT;  // first channel of this thread
    const int my = max(0, min(CPT, p.dim - c));            // its channels (0 past the end)
    const bool full = my == CPT;
    const bool has_init = p.has_init ? __ldg(p.has_init + s) != 0 : true;

    const B *xq = reinterpret_cast<const B *>(p.x) + c;
    B *oq = reinterpret_cast<B *>(p.out) + c;
    B *srow = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;

    // element j of the thread's run of CPT channels in row `row` of x (0 past the end)
    auto load_x = [&](uint32_t *w, long long row) {
        const B *src = xq + row * p.x_tok;
        if (full && p.x_vec) {
            ldv<VX, NW>(w, src);
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i) w[i] = 0u;
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                if (j < my) w[j / EW] |= (uint32_t)src[j] << (ES == 2 ? 16 * (j % EW) : 0);
        }
    };

    // taps and bias
    float wt[CPT][W], bs[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        bs[j] = (p.bias && j < my) ? widen<B>(reinterpret_cast<const B *>(p.bias)[c + j]) : 0.0f;
#pragma unroll
        for (int k = 0; k < W; ++k) wt[j][k] = j < my ? widen<B>(reinterpret_cast<const B *>(p.weight)[(long long)(c + j) * W + k]) : 0.0f;
    }

    // the window before token t0: initial window (first chunk) or the W-1 x rows before it
    float win[CPT][R];
    B init_raw[CPT][R];
    if (chunk == 0) {
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int k = 0; k < R; ++k) {
                init_raw[j][k] = (has_init && j < my) ? srow[(long long)j * p.st_ch + k] : (B)0;
                win[j][k] = widen<B>(init_raw[j][k]);
            }
    } else {
#pragma unroll
        for (int k = 0; k < R; ++k) {
            uint32_t w[NW];
            load_x(w, (long long)b + t0 - R + k);
#pragma unroll
            for (int j = 0; j < CPT; ++j) win[j][k] = elem_f<B>(w, j);
        }
    }

    const bool l2_block = (int)(blockIdx.x * blockDim.x * CPT) < p.qk_channels;  // block-uniform
    const bool l2_mine = c < p.qk_channels;
    constexpr int LOG_CPT = CPT == 4 ? 2 : 3;
    const int lanes = p.head_dim >> LOG_CPT;
    // rows of the batch starting at token tb (zeros past the chunk)
    auto load_batch = [&](uint32_t (*xr)[NW], int tb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u < t1) {
                load_x(xr[u], (long long)b + tb + u);
            } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) xr[u][i] = 0u;
            }
        }
    };
    // channels in pairs (paired fp32 lanes: the same operations per lane, half the instructions)
    constexpr int P = CPT / 2;
    f2 win2[P][R], wt2[P][W], bs2[P];
#pragma unroll
    for (int q = 0; q < P; ++q) {
        bs2[q] = f2_pack(bs[2 * q], bs[2 * q + 1]);
#pragma unroll
        for (int k = 0; k < W; ++k) wt2[q][k] = f2_pack(wt[2 * q][k], wt[2 * q + 1][k]);
#pragma unroll
        for (int k = 0; k < R; ++k) win2[q][k] = f2_pack(win[2 * q][k], win[2 * q + 1][k]);
    }
    // conv + SiLU + L2 + stores of the batch of rows xr starting at token tb
    auto run_batch = [&](const uint32_t (*xr)[NW], int tb) {
        float y[U][CPT];
        f2 acc2[U][P];
        float lo = 0.0f;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int q = 0; q < P; ++q) {
                f2 in[W];
#pragma unroll
                for (int k = 0; k < R; ++k) in[k] = win2[q][k];
                in[R] = f2_pack(elem_f<B>(xr[u], 2 * q), elem_f<B>(xr[u], 2 * q + 1));
                acc2[u][q] = conv_chain2<B, W>(bs2[q], wt2[q], in);
#pragma unroll
                for (int k = 0; k + 1 < R; ++k) win2[q][k] = win2[q][k + 1];
                win2[q][R - 1] = in[R];
                float a0, a1;
                f2_unpack(acc2[u][q], a0, a1);
                lo = fminf(lo, fminf(a0, a1));
                f2_unpack(silu_fast2(acc2[u][q]), y[u][2 * q], y[u][2 * q + 1]);
            }
        if (lo < -80.0f) {
            // only the values below -80 take the exact form (the same bits as silu())
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    float a0, a1;
                    f2_unpack(acc2[u][q], a0, a1);
                    if (a0 < -80.0f) y[u][2 * q] = silu_exact(a0);
                    if (a1 < -80.0f) y[u][2 * q + 1] = silu_exact(a1);
                }
        }
        if (l2_block) {
            float ss[U];
#pragma unroll
            for (int u = 0; u < U; ++u) ss[u] = sum_squares<CPT>(y[u]);
            if (CPT == 4 && lanes > 1) {
#pragma unroll
                for (int u = 0; u < U; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], 1);
            }
            for (int o = lanes >> 1; o >= (CPT == 4 ? 2 : 1); o >>= 1) {
#pragma unroll
                for (int u = 0; u < U; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
            }
            if (l2_mine) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float r = rsqrtf(ss[u] + p.eps);
                    const f2 r2 = f2_pack(r, r);
#pragma unroll
                    for (int q = 0; q < P; ++q)
                        f2_unpack(f2_mul(f2_pack(y[u][2 * q], y[u][2 * q + 1]), r2), y[u][2 * q], y[u][2 * q + 1]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tb + u >= t1 || my == 0) continue;
            B *dst = oq + ((long long)b + tb + u) * p.out_tok;
            if (full && p.out_vec) {
                uint32_t ow[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    if (ES == 2) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(y[u][2 * i], y[u][(2 * i + 1) % CPT]);
                        ow[i] = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        ow[i] = __float_as_uint(y[u][i]);
                    }
                }
                stv<VX, NW>(dst, ow);
            } else {
#pragma unroll
                for (int j = 0; j < CPT; ++j)
                    if (j < my) dst[j] = narrow<B>(y[u][j]);
            }
        }
    };

    extern __shared__ __align__(16) unsigned char ring[];
    const int NT = blockDim.x;
    constexpr int RB = CPT * ES;  // bytes of a thread's piece of one x row: 8, 16 or 32
    if (p.x_vec && dynamic_smem_bytes() >= (unsigned)(kPrefillRing * U * NT * RB)) {
        // aligned rows: each thread stages its own RB-byte pieces of the next batches in shared
        // memory by cp.async ([batch][row][thread] cells, conflict-free), kPrefillRing - 1 batches
        // ahead, so no register holds data in flight.  With x_vec a thread has all CPT channels or
        // none (dim % 8 == 0); one with none, and rows past the chunk, get zeros and read nothing
        // (their source address is the row base, inside the buffer).
        constexpr int D = kPrefillRing;
        auto cell = [&](int slot, int u) { return ring + ((size_t)(slot * U + u) * NT + tid) * RB; };
        auto issue = [&](int k, int nb) {
            if (k < nb) {
                const int tb = t0 + k * U;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const bool ok = my > 0 && tb + u < t1;
                    const B *src = ok ? xq + ((long long)b + tb + u) * p.x_tok : reinterpret_cast<const B *>(p.x);
                    if constexpr (RB == 8) {
                        prefill_cp_async<8>(cell(k % D, u), src, ok ? 8u : 0u);
                    } else {
#pragma unroll
                        for (int h = 0; h < RB / 16; ++h)
                            prefill_cp_async<16>(cell(k % D, u) + 16 * h, reinterpret_cast<const unsigned char *>(src) + (ok ? 16 * h : 0),
                                                 ok ? 16u : 0u);
                    }
                }
            }
            asm volatile("cp.async.commit_group;\n" ::: "memory");  // (an empty group past the end)
        };
        const int nb = (t1 - t0 + U - 1) / U;
#pragma unroll
        for (int k = 0; k < D - 1; ++k) issue(k, nb);
        for (int k = 0; k < nb; ++k) {
            issue(k + D - 1, nb);  // into the cell batch k - 1 was read from
            asm volatile("cp.async.wait_group %0;\n" ::"n"(D - 1) : "memory");  // batch k has landed
            uint32_t xr[U][NW];
#pragma unroll
            for (int u = 0; u < U; ++u) ldv<VX, NW>(xr[u], cell(k % D, u));
            run_batch(xr, t0 + k * U);
        }
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    } else {
        uint32_t xn[U][NW];  // the next batch, in flight while this one is computed
        if (t0 < t1) load_batch(xn, t0);
        for (int tb = t0; tb < t1; tb += U) {
            uint32_t xr[U][NW];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < NW; ++i) xr[u][i] = xn[u][i];
            if (tb + U < t1) load_batch(xn, tb + U);
            run_batch(xr, tb);
        }
    }

    // the final window, written by the block that read the initial one (raw bit copies)
    if (chunk == 0 && my > 0) {
        B fin[CPT][R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int j = L + k;  // index into [initial window, x]
            if (j < R) {
#pragma unroll
                for (int q = 0; q < CPT; ++q) {
                    B v = init_raw[q][0];
#pragma unroll
                    for (int r = 1; r < R; ++r) v = j == r ? init_raw[q][r] : v;
                    fin[q][k] = v;
                }
            } else {
                const B *src = xq + ((long long)b + j - R) * p.x_tok;
#pragma unroll
                for (int q = 0; q < CPT; ++q) fin[q][k] = q < my ? src[q] : (B)0;
            }
        }
#pragma unroll
        for (int q = 0; q < CPT; ++q)
            if (q < my)
#pragma unroll
                for (int k = 0; k < R; ++k) srow[(long long)q * p.st_ch + k] = fin[q][k];
    }
}

}  // namespace cvk
