// Commit kernel: restore the conv state of the accepted prefix from the verify's snapshots.
//
// sglang PR #46184 ("Motivation"): the intermediate window lets the conv state of the accepted
// prefix be restored after verify; glm5next_kda mod.rs decode_k: snapshot t is the state after row
// t, which a partial accept rewinds to.  The accept count a = accept_len[s] is read on the device,
// so no host round trip sits between the accept decision and the restore; the state becomes
// snapshot a-1.
//
// One block per (block of 8*threads channels, sequence).  Three shapes:
//   mode 1, dense snapshots packed [.., dim, W-1] and state rows packed [dim][W-1]: the snapshot's
//     channel block is one contiguous run, copied with 16-byte vectors;
//   mode 2, deduplicated rows packed [.., dim, T+W-2] and packed state: the block's rows (one
//     contiguous run) are staged in shared memory with 16-byte asynchronous copies, and the state
//     run [c][k] = row[c][a-1+k] is gathered from there and written with 16-byte coalesced stores;
//   mode 0, anything else: element by element.
#pragma once

#include "cv_device.cuh"

namespace cvk {

template <typename B, int W>
__global__ void __launch_bounds__(128) commit_kernel(const __grid_constant__ CommitParams p) {
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int VE = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];

    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int status = 0;
    if (slot >= 0) {
        if (slot >= p.n_slots) status |= 1;
        if (a < 1 || a > p.T) status |= 4;
    }
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status) return;

    const int BC = 8 * NT;
    const int c0 = blockIdx.x * BC;
    const int nch = min(BC, p.dim - c0);
    B *dst = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot;

    if (p.mode == 1) {
        const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_step +
                       (long long)c0 * R;
        B *d = dst + (long long)c0 * R;
        const int nv = nch * R / VE;
        for (int i = tid; i < nv; i += NT) st16(d + i * VE, ld16(src + i * VE));
    } else if (p.mode == 2) {
        const int Q = p.T + R - 1;
        const B *rows = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)c0 * Q;
        B *sm = reinterpret_cast<B *>(smem);
        const int nv = nch * Q / VE;
        for (int i = tid; i < nv; i += NT) cp_async16(sm + i * VE, rows + i * VE);
        cp_async_wait_all();
        __syncthreads();
        B *d = dst + (long long)c0 * R;
        const int nd = nch * R / VE;
        const int col0 = a - 1;
        for (int m = tid; m < nd; m += NT) {
            uint32_t wv[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t bits[2];
#pragma unroll
                for (int z = 0; z < 4 / ES; ++z) {
                    const int pos = m * VE + h * (4 / ES) + z;
                    const int cc = pos / R, k = pos - cc * R;
                    bits[z] = (uint32_t)sm[cc * Q + col0 + k];
                }
                wv[h] = (ES == 2) ? pack_halves(bits[0], bits[1]) : bits[0];
            }
            st16(d + m * VE, make_uint4(wv[0], wv[1], wv[2], wv[3]));
        }
    } else {
        const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_step;
        for (int i = tid; i < nch * R; i += NT) {
            const int cc = c0 + i / R, k = i % R;
            dst[(long long)cc * p.st_ch + k] = src[(long long)cc * p.w_ch + (long long)k * p.w_col];
        }
    }
}

}  // namespace cvk
