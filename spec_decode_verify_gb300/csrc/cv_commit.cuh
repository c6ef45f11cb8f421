// Commit kernel: restore the conv state of the accepted prefix from the verify's snapshots.
//
// sglang PR #46184 ("Motivation"): the intermediate window is kept so the state can be rolled
// back to the accepted prefix once verify is done; glm5next_kda mod.rs decode_k: snapshot t is the state after row
// t, which a partial accept rewinds to.  The accept count a = accept_len[s] is read on the device,
// so no host round trip sits between the accept decision and the restore; the state becomes
// snapshot a-1.
//
// commit_kernel: one block per (block of 8*threads channels, sequence), two instances:
//   PACKED (mode 1), dense snapshots packed [.., dim, W-1] and state rows packed [dim][W-1]: the
//     snapshot's channel block is one contiguous run, copied with 16-byte vectors;
//   otherwise (mode 0), anything else: element by element.
// They are separate kernels so that the element path's registers do not cut the packed path's
// residency.
// commit_wide (below) handles packed dense snapshots with packed state rows wider than the window,
// commit_rows packed deduplicated rows with packed state rows, commit_cols the same
// rows laid out transposed (column-major), and commit_recompute the recompute rollback (no
// snapshots: the state is rebuilt from its kept window and the verify's inputs).
#pragma once

#include <type_traits>

#include "cv_device.cuh"

namespace cvk {

constexpr unsigned kCommitWaitPolls = 1u << 20;  // mbarrier polls before a block gives up

// Status of sequence s for a commit: 1 = slot out of range, 16 = invalid packed draft span, 4 =
// accept count a outside 1..T_s.  Sets ts to the sequence's draft count (T, or its packed span's
// length) and row0 to its first packed row.  A sequence with ts = 0 has nothing to commit.
__device__ __forceinline__ int commit_status(const CommitParams &p, int s, int slot, int a, int &ts, int &row0) {
    ts = p.T;
    row0 = 0;
    if (slot < 0) return 0;
    int st = slot >= p.n_slots ? 1 : 0;
    if (p.cu_draft) st |= draft_span(p.cu_draft, s, p.T, p.total_tokens, ts, row0);
    if (!(st & kSeqBadSpan) && ts > 0 && (a < 1 || a > ts)) st |= 4;
    return st;
}

template <typename B, int W, bool PACKED>
__global__ void __launch_bounds__(128) commit_kernel(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int VE = 16 / ES;

    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status || ts == 0) return;

    const int BC = 8 * NT;
    const int c0 = blockIdx.x * BC;
    const int nch = min(BC, p.dim - c0);
    B *dst = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot;

    // A block covers at most 8*NT channels.  A thread issues its loads before its stores (the
    // compiler cannot move a load above a store that may alias it): the packed path's whole share
    // at once, so its data costs one round trip; the element path's in rounds of 8 elements (one
    // round of 16 measured slower in the verify + commit step, 13.5 us against 12.95 for 64
    // sequences x 8 tokens x 6144 channels, width 3, state rows of 9 columns, although the commit
    // alone took 4.3 us against 4.8).
    if constexpr (PACKED) {
        const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_step +
                       (long long)c0 * R;
        B *d = dst + (long long)c0 * R;
        const int nv = nch * R / VE;
        constexpr int UV = 8 * R / VE;  // 16-byte vectors per thread
        uint4 v[UV];
#pragma unroll
        for (int u = 0; u < UV; ++u)
            if (tid + u * NT < nv) v[u] = ld16(src + (tid + u * NT) * VE);
#pragma unroll
        for (int u = 0; u < UV; ++u)
            if (tid + u * NT < nv) st16(d + (tid + u * NT) * VE, v[u]);
    } else {
        // element by element, consecutive threads on consecutive elements
        constexpr int U = 8;
        const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_step;
        const int n = nch * R;
        for (int i0 = tid; i0 < n; i0 += U * NT) {
            B v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * NT;
                const int cc = c0 + i / R, k = i % R;
                if (i < n) v[u] = src[(long long)cc * p.w_ch + (long long)k * p.w_col];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * NT;
                const int cc = c0 + i / R, k = i % R;
                if (i < n) dst[(long long)cc * p.st_ch + k] = v[u];
            }
        }
    }
}

// Commit of packed dense snapshots into packed state rows wider than the window (mode 5): the rows
// [dim][S] per slot with S > W-1, the layout whose window the verify reads at a state offset
// ([kda-mod] binding).  One block per (8*threads channels, sequence).  The block's rows are one
// contiguous run: they are copied into shared memory by 16-byte cp.async copies while each thread
// loads its 16-byte pieces of snapshot a-1 (one contiguous run as well); the new window then goes
// over the rows' first W-1 columns in shared memory, and the rows go back whole as coalesced 16-byte
// stores.  So every access is a 16-byte vector, every store fills whole sectors, the data costs one
// round trip, and the other columns are written back with their own bits.
template <typename B, int W>
__global__ void __launch_bounds__(128) commit_wide(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int VE = 16 / ES;
    constexpr int UV = 8 * R / VE;  // 16-byte snapshot vectors per thread
    using U = std::conditional_t<ES == 2, unsigned short, unsigned>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && tid == 0) p.err[s] = status;
    if (slot < 0 || status || ts == 0) return;

    const int c0 = blockIdx.x * 8 * NT;
    const int nch = min(8 * NT, p.dim - c0);  // a multiple of 8 (dim % 8 == 0 on this path)
    const int S = (int)p.st_ch;               // the row width (host: st_ch == state_cols)
    const int nbytes = nch * S * ES;          // a multiple of 16
    unsigned char *rows =
        reinterpret_cast<unsigned char *>(reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * S);
    for (int o = tid * 16; o < nbytes; o += NT * 16) cp_async16(smem + o, rows + o);
    const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_step +
                   (long long)c0 * R;
    const int nv = nch * R / VE;
    union {
        uint4 v[UV];
        U e[UV * VE];
    } sn;
#pragma unroll
    for (int u = 0; u < UV; ++u)
        if (tid + u * NT < nv) sn.v[u] = ld16(src + (tid + u * NT) * VE);
    cp_async_wait_all();
    __syncthreads();
    U *img = reinterpret_cast<U *>(smem);
#pragma unroll
    for (int u = 0; u < UV; ++u) {
        if (tid + u * NT < nv) {
            const int i0 = (tid + u * NT) * VE;  // element of the snapshot run: channel i / R, column i % R
#pragma unroll
            for (int z = 0; z < VE; ++z) img[((i0 + z) / R) * S + (i0 + z) % R] = sn.e[u * VE + z];
        }
    }
    __syncthreads();
    for (int o = tid * 16; o < nbytes; o += NT * 16)
        st16(rows + o, *reinterpret_cast<const uint4 *>(smem + o));
}

// Commit of packed deduplicated rows into packed state rows (mode 2): one block per (block of
// 8*threads channels, sequence), a single wave of small blocks.  The row address does not depend
// on the cache slot, so thread 0 starts the bulk copy (TMA, cp.async.bulk) of the block's rows --
// one contiguous run of channels*(T+W-2) elements -- before anything else, and the slot and the
// accept count are read while it is in flight; no dependent load precedes the data.  (Right after
// the verify the rows are in L2: reading them whole in parallel with the indices beats reading the
// slot first and then only the needed columns; the rows of padded sequences are read too.)  The
// state run [c][k] = row[c][a-1+k] is then gathered from shared memory and written with 16-byte
// coalesced stores.  A padded or rejected sequence still waits for its copy (the shared memory must
// outlive it) and writes nothing.  The wait is bounded (p.wait_polls polls, 0 = the default,
// negative = none): a timeout sets CV_SEQ_TIMEOUT in err, and the copy is then drained with the
// default limit before the block leaves.  Every err bit is ORed in; the library clears err before
// the launch.
template <typename B, int W>
__global__ void __launch_bounds__(64) commit_rows(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int VE = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int s = blockIdx.y;
    const int BC = 8 * blockDim.x;
    const int c0 = blockIdx.x * BC;
    const int nch = min(BC, p.dim - c0);
    const int Q = p.T + R - 1;
    const long long row_bytes = ((long long)BC * Q * ES + 127) / 128 * 128;
    uint64_t *const bar = reinterpret_cast<uint64_t *>(smem + row_bytes);
    if (row_bytes + 8 > (long long)dynamic_smem_bytes()) return;  // launch mismatch
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
        mbar_arrive_expect_tx(bar, (unsigned)(nch * Q * ES));
        bulk_load(smem, reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)c0 * Q,
                  (unsigned)(nch * Q * ES), bar);
    }
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && tid == 0 && status) atomicOr(p.err + s, status);
    __syncthreads();  // the barrier's initialisation is visible to every waiting thread
    const unsigned polls = p.wait_polls == 0 ? kCommitWaitPolls : p.wait_polls < 0 ? 0u : (unsigned)p.wait_polls;
    const bool ok = mbar_wait_bounded(bar, 0u, polls);
    if (__syncthreads_or(!ok)) {  // every thread agrees before anyone leaves
        if (tid == 0) {
            if (p.err && slot >= 0) atomicOr(p.err + s, kSeqTimeout);
            mbar_wait_bounded(bar, 0u, kCommitWaitPolls);  // drain the copy (bounded)
        }
        return;
    }
    if (slot < 0 || status || ts == 0) return;
    const B *sm = reinterpret_cast<const B *>(smem);
    B *d = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * R;
    const int col0 = a - 1;
    const int nd = nch * R / VE;
    for (int m = tid; m < nd; m += blockDim.x) {
        uint32_t wv[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint32_t bits[2] = {0u, 0u};
#pragma unroll
            for (int z = 0; z < 4 / ES; ++z) {
                const int pos = m * VE + h * (4 / ES) + z;
                const int cc = pos / R, kk = pos - cc * R;
                bits[z] = (uint32_t)sm[cc * Q + col0 + kk];
            }
            wv[h] = (ES == 2) ? pack_halves(bits[0], bits[1]) : bits[0];
        }
        st16(d + m * VE, make_uint4(wv[0], wv[1], wv[2], wv[3]));
    }
}

// Commit of packed deduplicated rows laid out transposed -- the window row of sequence s stored
// column by column, [n_seq][T+W-2][dim] seen as [n_seq][dim][T+W-2] with a channel stride of 1
// (sglang PR #46184, "Modifications", test coverage: MambaPool's axis-0 window layout seen
// transposed) -- into packed state rows (mode 4).  Snapshot a-1 is columns a-1 .. a+W-3, each a
// contiguous run of channels, so a thread of 8 channels reads exactly its W-1 16-byte pieces (after
// the slot and the accept count that locate them) and writes its [8][W-1] state run as 16-byte
// stores: the commit moves its algorithmic bytes and nothing else.
template <typename B, int W>
__global__ void __launch_bounds__(128) commit_cols(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int NV = 8 * ES / 16;  // 16-byte vectors per column piece of 8 channels
    using U = std::conditional_t<ES == 2, unsigned short, unsigned>;
    const int s = blockIdx.y;
    const int c = 8 * (blockIdx.x * blockDim.x + threadIdx.x);
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && threadIdx.x == 0) p.err[s] = status;
    if (c >= p.dim || slot < 0 || status || ts == 0) return;
    union {
        uint4 v[NV];
        U e[8];
    } col[R];
    const B *src = reinterpret_cast<const B *>(p.win) + (long long)s * p.w_seq + (long long)(a - 1) * p.w_col + c;
#pragma unroll
    for (int k = 0; k < R; ++k)
#pragma unroll
        for (int i = 0; i < NV; ++i) col[k].v[i] = __ldg(reinterpret_cast<const uint4 *>(src + (long long)k * p.w_col) + i);
    union {
        uint4 v[R * NV];
        U e[8 * R];
    } run;
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int k = 0; k < R; ++k) run.e[e * R + k] = col[k].e[e];
    uint4 *d = reinterpret_cast<uint4 *>(reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * R);
#pragma unroll
    for (int i = 0; i < R * NV; ++i) d[i] = run.v[i];
}

// Recompute rollback (memra-engine Engine doc, ssm_conv_ring_rebuild_dc: the conv state is rebuilt
// from the window kept from before the verify and the verify's inputs, with the accept count read
// on the device).  One thread per channel: with full = [state[0 .. W-2], x_0 .. x_{T-1}], the new
// window is full[a .. a+W-2] -- state columns while a+k < W-1, x rows a+k-(W-1) after -- loaded
// first and stored after, so the in-place rewrite of the row is safe.  Across a warp the state
// elements are one contiguous run (packed rows) and each x row is contiguous, so every access is
// coalesced; the accesses are 2- or 4-byte, enough since at most 3 x 2 elements move per channel.
template <typename B, int W>
__global__ void __launch_bounds__(128) commit_recompute(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    const int s = blockIdx.y;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && threadIdx.x == 0) p.err[s] = status;
    if (slot < 0 || status || ts == 0) return;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= p.dim) return;
    B *row = reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot + (long long)c * p.st_ch;
    const B *xs = reinterpret_cast<const B *>(p.x) + (p.cu_draft ? (long long)row0 * p.x_tok : (long long)s * p.x_seq) + c;
    B v[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const int j = a + k;  // position in full
        v[k] = j < R ? row[j] : xs[(long long)(j - R) * p.x_tok];
    }
#pragma unroll
    for (int k = 0; k < R; ++k) row[k] = v[k];
}

// The same rebuild for packed state rows and 16-byte aligned x rows: 8 channels per thread, so a
// thread moves its window run and each needed x row as 16-byte vectors and one block covers
// 8*threads channels -- the whole batch fits in one wave, each thread making one round trip for
// the indices and one for the data.  The accept count is a runtime value, so each new column k
// takes, per channel, either old column a+k (picked by selects among the W-1 old columns) or
// element e of the x row a+k-(W-1) (loaded whole when some column needs it).
template <typename B, int W>
__global__ void __launch_bounds__(128) commit_recompute_vec(const __grid_constant__ CommitParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int R = W - 1;
    constexpr int ES = (int)sizeof(B);
    constexpr int NXV = 8 * ES / 16;      // 16-byte vectors per x row of 8 channels
    constexpr int NSV = 8 * R * ES / 16;  // 16-byte vectors per window run of 8 channels
    using U = std::conditional_t<ES == 2, unsigned short, unsigned>;
    const int s = blockIdx.y;
    const int slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
    const int a = __ldg(p.accept_len + s);
    int ts, row0;
    const int status = commit_status(p, s, slot, a, ts, row0);
    if (p.err && blockIdx.x == 0 && threadIdx.x == 0) p.err[s] = status;
    if (slot < 0 || status || ts == 0) return;
    const int c = 8 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (c >= p.dim) return;  // dim % 8 == 0 on this path
    uint4 *run = reinterpret_cast<uint4 *>(reinterpret_cast<B *>(p.state) + (long long)slot * p.st_slot +
                                           (long long)c * R);
    const B *xs = reinterpret_cast<const B *>(p.x) + (p.cu_draft ? (long long)row0 * p.x_tok : (long long)s * p.x_seq) + c;
    union {
        uint4 v[NSV];
        U e[8 * R];
    } old, neu;
    union {
        uint4 v[NXV];
        U e[8];
    } xr[R];
#pragma unroll
    for (int i = 0; i < NSV; ++i) old.v[i] = run[i];
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const int j = a + k;
        if (j >= R) {
#pragma unroll
            for (int i = 0; i < NXV; ++i)
                xr[k].v[i] = __ldg(reinterpret_cast<const uint4 *>(xs + (long long)(j - R) * p.x_tok) + i);
        } else {
#pragma unroll
            for (int i = 0; i < NXV; ++i) xr[k].v[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int j = a + k;
            U o = old.e[e * R];
#pragma unroll
            for (int q = 1; q < R; ++q) o = j == q ? old.e[e * R + q] : o;
            neu.e[e * R + k] = j < R ? o : xr[k].e[e];
        }
#pragma unroll
    for (int i = 0; i < NSV; ++i) run[i] = neu.v[i];
}

}  // namespace cvk
