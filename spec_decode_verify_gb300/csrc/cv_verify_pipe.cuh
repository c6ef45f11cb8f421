// Persistent, bulk-copy-pipelined verify kernel: the main path for packed buffers with T <= 17.
//
// A unit of work is one block of CPT*threads channels of one sequence (the block of the Atlas
// batched verify, fn gdn_verify_fused_conv_kn_batched).  A persistent block walks the units
// u = blockIdx.x, blockIdx.x + gridDim.x, ...; when the grid is a multiple of the channel-block
// count every unit of a block has the same channels, so the taps and bias are loaded once.  One
// thread issues each unit's loads as bulk copies (TMA, cp.async.bulk) into one of two
// shared-memory stages -- the T x rows and the committed windows -- completing on that stage's
// mbarrier, two units ahead.  So the reads of later units overlap the arithmetic and the stores of
// the current one on every SM, instead of all blocks loading, then computing, then storing in
// lock-step.  The staged images are double-buffered too, so one block barrier per unit suffices.
// Per unit each thread moves its CPT channels from the stage to registers, writes what depends on
// the inputs only (the deduplicated row of sglang PR #46184 -- the window of step t is the W-1
// columns from column t of [state[1..W-2], x_0..x_{T-1}] -- as one staged image written by one
// bulk copy;
// dense snapshots as vector stores; the committed window, staged and bulk-copied into the packed
// state rows) and computes the outputs: fp32 conv with bias first and the taps in order
// (conv_chain), SiLU, the L2 normalisation of the q|k groups over head_dim/CPT lanes with the T
// shuffle trees interleaved (glm5next_kda mod.rs), one rounding, vector stores.
// Every mbarrier wait is bounded: a block that waits too long for a unit's copies sets
// CV_SEQ_TIMEOUT in err (when given) for that unit's sequence and for the sequence of every later
// unit it owns (none of which it will run), drains its copies in flight (with the full default
// limit, so nothing lands in shared memory after the block has left) and returns.  The limit of
// that first wait per unit is p.wait_polls (0: the default; negative: no poll at all, a wait
// that gives up at once).  Every err bit is ORed in; the library zeroes err before the launch.
// Deduplicated rows laid out transposed ([n_seq][T+W-2][dim] seen as [n_seq][dim][T+W-2], channel
// stride 1: sglang PR #46184, "Modifications", test coverage: MambaPool's axis-0 window layout seen
// transposed): the image is staged column by column, [T+W-2][channels], and leaves as one bulk copy
// per column, each a contiguous run of the block's channels.
// History-row state (no window buffer): the stage holds each channel's whole [T+W-2] state row,
// the committed window is taken from columns [off, off+W-1) of it, and the row image is stored
// back over the state row instead of into a window buffer; there is no separate committed-window
// image.  Column-major history rows (the state row stored column by column, channel stride 1): the
// stage holds only the W-1 columns at the offset, one bulk copy each, and the row image is staged
// column by column like a transposed dedup row and stored as one bulk copy per column, so the
// commit-free step moves exactly the bytes the method reads and writes.  Recompute rollback: outputs only; nothing is staged for storing and no bulk store runs.
// State rows wider than the window (read at a state offset) are staged whole too; each thread
// copies its channels' staged rows into the state image with the committed window over their first
// W-1 columns, and the image leaves whole by one bulk copy (the other columns go back with their
// own bits): one contiguous run per unit instead of element stores at the row pitch.
// Mixed dtypes (S, the type of the state and the snapshots, differs from B, the type of x, out, taps
// and bias): the stages and the images hold each part in its own type; state columns keep their
// bits, x elements enter them widened exactly (bf16 -> fp32) or rounded to the nearest bf16, and
// the conv takes every input at its own precision with each product rounded (fp32 state values
// make the products inexact).
// Packed ragged drafts (VL; sglang PR #46184, "Related upstream work": target verify on packed ragged
// tokens, the tile store covering the packed rows): sequence s owns rows [cu[s], cu[s+1]) of x and
// out, T_s <= p.T of them, cut into chunks of at most TS tokens (TS = p.T when p.T <= 8, else 8):
// a unit is (sequence, chunk, channel block), so a draft of any length runs with the registers of
// an 8-token unit.  Chunk c holds tokens [8c, 8c + n); its first W-1 inputs are the committed
// window (c = 0) or the 3 x rows before it (the halo, staged after the chunk's rows), and it writes
// its outputs, its dense snapshot steps and its columns of the snapshot row: a full row leaves as
// one bulk copy, a transposed row as one bulk copy per column, anything shorter is copied out of
// the staged image by the block element by element (columns past T_s+W-2 are never written).  The
// committed window full[T_s .. T_s+W-2] is written by chunk 0 alone -- from its own rows, or from
// the last W-1 rows of the draft, which it stages as a tail -- so no other block's chunk writes a
// state row that chunk 0 reads.  Units of long and short chunks differ in cost, so the list of
// units is ordered by tokens per chunk, most first (list_chunks, identical in every block):
// consecutive units of the round-robin walk then cost about the same.
// Preconditions (checked on the host): those of the fast path, packed 16-byte-aligned state rows
// (state_ch_stride == state_cols; exactly T+W-2 columns for the history layout), T <= 17 (bf16) /
// 8 (fp32), head_dim / CPT <= 32.
#pragma once

#include <type_traits>

#include "cv_device.cuh"

namespace cvk {

constexpr unsigned kWaitPolls = 1u << 20;  // mbarrier polls before a block gives up

// Bytes of one stage for a block of bc channels (x rows, windows, taps, bias), each part 128-aligned.
__host__ __device__ constexpr long long pipe_part(long long b) { return (b + 127) / 128 * 128; }

template <typename B, int W, int TS, int CPT, typename S = B, bool VL = false>
__global__ void __launch_bounds__(128, (CPT == 4 && TS <= 8) ? 4 : 2) verify_pipe(const __grid_constant__ VerifyParams p) {
    // (griddepcontrol.wait comes after the L2 prefetch hints below: nothing before it reads data)
    static_assert(TS > 0, "the pipelined kernel needs a compile-time T");
    static_assert(!VL || std::is_same_v<B, S>, "packed ragged drafts use one dtype");
    // (taps and bias are read from global memory, so W*CPT*ES need only be 8-byte aligned)
    constexpr int R = W - 1;
    constexpr int Q = TS + R - 1;  // dedup row columns
    constexpr bool MIXED = !std::is_same_v<B, S>;
    constexpr int ES = (int)sizeof(B);   // x, out, taps, bias
    constexpr int ESS = (int)sizeof(S);  // state, snapshots
    constexpr int EW = 4 / ES;
    constexpr int NW = CPT / EW;          // words of CPT x elements
    constexpr int NWS = CPT * ESS / 4;    // words of CPT state elements
    constexpr int VX = pipe_align(CPT * ES);
    constexpr int VS = pipe_align(CPT * R * ESS);
    constexpr int VW = pipe_align(CPT * W * ES);
    constexpr int VI = pipe_align(CPT * Q * ESS);
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int BC = CPT * blockDim.x;
    const int nblk = (p.dim + BC - 1) / BC;
    const bool hist = p.hist != 0;        // history-row state: no window buffer
    const bool recomp = p.recomp != 0;    // recompute rollback: outputs only
    const bool dense = !p.dedup && !hist;  // dense window (or none): no row image
    const bool dedup_t = p.dedup_t != 0;     // dedup rows stored column by column
    const bool has_bias = p.bias != nullptr;
    // state columns staged per channel: the committed windows of packed [dim][W-1] rows, or whole
    // rows when they are wider (history rows, or rows read at a state offset)
    const int SC = p.state_cols;
    const bool hist_t = hist && p.st_col != 1;  // column-major history rows: W-1 columns staged
    const int SCS = hist_t ? R : SC;            // state columns per staged channel (or staged columns)
    const bool whole_rows = !hist_t && SC != R;
    const bool wide = whole_rows && !hist;  // wider rows, not history: staged whole, stored whole
    // Each thread stores its committed-window run straight to the packed state rows (coalesced
    // vectors) instead of through a shared-memory image and a bulk copy: with mixed dtypes, so that
    // the larger fp32 images leave room for a third block per SM (measured, bf16 x with fp32 state
    // and rows, 128 x 8 x 10240: 23.1 us against 24.2 with two blocks per SM; storing the dedup rows
    // from registers too, for four blocks per SM, took 27.5 us), and with packed drafts (ragged
    // step 31.9 against 32.0 us).  Only where the kernel's type parameters decide it: as a runtime
    // choice (for transposed rows, where it measured 19.18 against 19.46 us) the extra branch cost
    // the row-major rows 0.1 us.
    const bool direct_state = (MIXED || VL) && !wide && !hist && !recomp;

    // packed drafts longer than a chunk: W-1 more staged x rows per unit (a halo or a tail)
    const bool chunked = VL && p.T > TS;
    const int XR = TS + (chunked ? R : 0);
    const int Qrow = p.T + R - 1;  // columns of the snapshot row in global memory (Q: of the staged image)

    // shared memory: stage 0, stage 1 (x rows + committed windows, or whole history rows), image
    // buffers 0 and 1 (dedup row image + committed-window image -- whole rows when they are wider
    // -- or the history row image alone),
    // 2 mbarriers and the unit information (kPipeInfoBytes), then (when compacting) the sort or warp
    // counts (AUX ints) and the list of active sequences (of chunks, for packed drafts)
    const long long xb = pipe_part((long long)XR * BC * ES);
    const long long stage_bytes = xb + pipe_part((long long)SCS * BC * ESS);
    const long long rb = dense ? 0 : pipe_part((long long)Q * BC * ESS);
    const long long img_bytes =
        recomp ? 0 : rb + ((hist || direct_state) ? 0 : pipe_part((long long)(wide ? SC : R) * BC * ESS));
    unsigned char *const img0 = smem + 2 * stage_bytes;
    uint64_t *const bar = reinterpret_cast<uint64_t *>(img0 + 2 * img_bytes);
    // [0, 2): slots, [2, 4): state offsets, [4, 6): draft counts, [6, 8): first rows (packed drafts)
    volatile int *const info = reinterpret_cast<volatile int *>(bar + 2);
    constexpr int AUX = pipe_aux_ints(VL, TS);
    int *const wcount = reinterpret_cast<int *>(smem + 2 * stage_bytes + 2 * img_bytes + kPipeInfoBytes);
    int *const act = wcount + AUX;
    const bool compact = p.compact != 0;
    const long long list_len = VL ? (long long)p.n_seq * ((p.T + TS - 1) / TS) : p.n_seq;
    // (whole batches: each listed sequence's cache slot and state offset, read while listing)
    int *const act_slot = act + list_len;
    int *const act_off = act_slot + list_len;
    if (2 * stage_bytes + 2 * img_bytes + kPipeInfoBytes + (compact ? 4LL * AUX + (VL ? 4 : 12) * list_len : 0) >
        (long long)dynamic_smem_bytes())
        return;  // launch mismatch

    // Before waiting for the previous grid: L2 prefetch hints for the x rows and state rows of the
    // block's first unit, taking unit u as sequence u / nblk (as if no sequence were padded).  The
    // cache slot is read through L2 only (never cached in L1), and only to form a hint's address,
    // which stays inside the state buffer; all data is read after the wait, so a hint that is stale
    // or misses costs only its bandwidth.  (Measured on the 128 x 8 x 10240 step: hints for the
    // first unit 19.9 us per verify + commit, two units 20.2, three 20.9.)
    if (!VL && tid == 0) {
        for (int k = 0; k < 1; ++k) {
            const long long u = (long long)blockIdx.x + (long long)k * gridDim.x;
            if (u >= (long long)p.n_seq * nblk) break;
            const int s = (int)(u / nblk), c0 = (int)(u - (long long)s * nblk) * BC;
            const int nch = min(BC, p.dim - c0);
            const B *xs = reinterpret_cast<const B *>(p.x) + (long long)s * p.x_seq + c0;
            for (int t = 0; t < TS; ++t) bulk_prefetch_l2(xs + (long long)t * p.x_tok, (unsigned)(nch * ES));
            const int slot = p.cache_idx ? __ldcg(p.cache_idx + s) : s;
            if (slot >= 0 && slot < p.n_slots && !hist_t)
                bulk_prefetch_l2(reinterpret_cast<const S *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * SC,
                                 (unsigned)(nch * SC * ESS));
        }
    }
    grid_dep_wait();
    grid_dep_launch();

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init_fence();
    }
    __syncthreads();

    // Units walk the active sequences only: the block lists the sequences whose cache slot is not
    // negative (ascending; packed drafts: by draft count), so padded sequences cost no unit and every
    // block gets its fair share of real work.  (Padded sequences' err entries stay 0: the library
    // clears err before the launch.)
    int n_act = p.n_seq;
    if (VL && compact) {
        n_act = list_chunks(p, wcount, TS);
    } else if (compact) {
        const int lane = tid & 31, warp = tid >> 5, nwarps = ((int)blockDim.x + 31) >> 5;
        n_act = 0;
        for (int i0 = 0; i0 < p.n_seq; i0 += (int)blockDim.x) {
            const int i = i0 + tid;
            const int sl = i < p.n_seq ? __ldg(p.cache_idx + i) : -1;
            const int of = (i < p.n_seq && p.state_off) ? __ldg(p.state_off + i) : 0;
            const bool a = sl >= 0;
            const unsigned m = __ballot_sync(0xffffffffu, a);
            if (lane == 0) wcount[warp] = __popc(m);
            __syncthreads();
            int before = 0, total = 0;
            for (int w = 0; w < nwarps; ++w) {
                const int cw = wcount[w];
                before += w < warp ? cw : 0;
                total += cw;
            }
            if (a) {
                const int pos = n_act + before + __popc(m & ((1u << lane) - 1u));
                act[pos] = i;
                act_slot[pos] = sl;
                act_off[pos] = of;
            }
            n_act += total;
            __syncthreads();
        }
    }
    // list entry q: (chunk << 16) | sequence (chunk 0 without packed drafts)
    auto seq_at = [&](int q) { return compact ? act[q] : q; };
    const int n_units = n_act * nblk;
    const int iters = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    // thread 0: start the copies of iteration k into stage k & 1 (or only arrive, for padding).  The
    // index data of the next unit (cache slot, state offset, packed row span) is loaded one issue
    // ahead, so no issue waits for a global-memory round trip; the first two units load theirs
    // together at the start and (whole-T batches) send their x copies out before the indices arrive
    // (those x rows do not depend on the slot).
    auto unit_of = [&](int k, int &s, int &c0, int &nch) {
        const int u = (int)blockIdx.x + k * (int)gridDim.x;
        const int q = u / nblk;
        s = seq_at(q) & 0xffff;
        c0 = (u - q * nblk) * BC;
        nch = min(BC, p.dim - c0);
    };
    auto chunk_of = [&](int k) { return VL ? seq_at(((int)blockIdx.x + k * (int)gridDim.x) / nblk) >> 16 : 0; };
    // a unit's index data: cache slot, state offset and (packed drafts) its row span [b, e)
    struct UnitIdx {
        int slot, off, b, e;
    };
    auto load_index = [&](int k, UnitIdx &ix) {
        if (k >= iters) return;
        const int q = ((int)blockIdx.x + k * (int)gridDim.x) / nblk;
        const int s = seq_at(q) & 0xffff;
        if (!VL && compact) {  // (read while listing)
            ix.slot = act_slot[q];
            ix.off = act_off[q];
        } else {
            ix.slot = p.cache_idx ? __ldg(p.cache_idx + s) : s;
            ix.off = p.state_off ? __ldg(p.state_off + s) : 0;
        }
        if constexpr (VL) {
            ix.b = __ldg(p.cu_draft + s);
            ix.e = __ldg(p.cu_draft + s + 1);
        } else {
            ix.b = s;  // (the rows of sequence s start at s * x_seq)
            ix.e = s + TS;
        }
    };
    // the unit's x rows: n rows from row b (packed drafts: the chunk's rows), or the TS rows of
    // sequence s, into stage rows 0 .. n-1
    auto issue_x = [&](int k, int b, int n) {
        const int st = k & 1;
        int s, c0, nch;
        unit_of(k, s, c0, nch);
        mbar_expect_tx(&bar[st], (unsigned)(n * nch * ES));
        const B *xs = reinterpret_cast<const B *>(p.x) + (VL ? (long long)b * p.x_tok : (long long)s * p.x_seq) + c0;
        for (int t = 0; t < n; ++t)
            bulk_load(smem + st * stage_bytes + (long long)t * BC * ES, xs + (long long)t * p.x_tok,
                      (unsigned)(nch * ES), &bar[st]);
    };
    // (packed drafts) W-1 x rows from row b into stage rows TS .. TS+W-2: a later chunk's halo, or
    // chunk 0's tail (the draft's last W-1 rows, which hold the committed window)
    auto issue_extra = [&](int k, int b) {
        const int st = k & 1;
        int s, c0, nch;
        unit_of(k, s, c0, nch);
        mbar_expect_tx(&bar[st], (unsigned)(R * nch * ES));
        const B *xs = reinterpret_cast<const B *>(p.x) + (long long)b * p.x_tok + c0;
        for (int j = 0; j < R; ++j)
            bulk_load(smem + st * stage_bytes + (long long)(TS + j) * BC * ES, xs + (long long)j * p.x_tok,
                      (unsigned)(nch * ES), &bar[st]);
    };
    // the phase cannot complete before the single arrival at its end, so a late expect_tx is safe
    auto issue = [&](int k, const UnitIdx &ix, bool x_sent) {
        const int st = k & 1;
        int s, c0, nch;
        unit_of(k, s, c0, nch);
        const int slot = ix.slot, off = ix.off;
        int status = seq_status(slot, off, p.n_slots, p.state_cols, R);
        int ts = TS;
        const int ch = chunk_of(k);
        if constexpr (VL) {  // (the span was loaded with the indices, one issue ahead)
            ts = ix.e - ix.b;
            if (slot >= 0) status |= span_status(ix.b, ix.e, p.T, p.total_tokens);
        }
        if (p.err && c0 == 0 && ch == 0 && status) atomicOr(p.err + s, status);
        const bool go = slot >= 0 && status == 0;
        info[st] = go ? slot : -1;
        info[2 + st] = off;
        info[4 + st] = (ch << 16) | ts;
        info[6 + st] = ix.b;
        if (go) {
            const int t0 = ch * TS;
            const int n = VL ? min(TS, ts - t0) : TS;
            if (!x_sent) issue_x(k, ix.b + t0, n);
            if (ch > 0) {
                issue_extra(k, ix.b + t0 - R);  // the halo: the W-1 rows before the chunk
            } else {
                if (chunked && ts > TS) issue_extra(k, ix.b + ts - R);  // the tail: the draft's last W-1 rows
                if (hist_t) {
                    // column-major history rows: columns [off, off+W-1), each a run of nch channels,
                    // into stage columns [0, W-1) of BC channels each
                    mbar_expect_tx(&bar[st], (unsigned)(R * nch * ESS));
                    const S *col0 = reinterpret_cast<const S *>(p.state) + (long long)slot * p.st_slot +
                                    (long long)off * p.st_col + c0;
                    for (int kk = 0; kk < R; ++kk)
                        bulk_load(smem + st * stage_bytes + xb + (long long)kk * BC * ESS, col0 + (long long)kk * p.st_col,
                                  (unsigned)(nch * ESS), &bar[st]);
                } else {
                    // packed state rows of SC columns: the committed windows, or whole rows
                    mbar_expect_tx(&bar[st], (unsigned)(SC * nch * ESS));
                    bulk_load(smem + st * stage_bytes + xb,
                              reinterpret_cast<const S *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * SC,
                              (unsigned)(nch * SC * ESS), &bar[st]);
                }
            }
        }
        mbar_arrive(&bar[st]);
    };
    // polls of each unit's first wait for its copies (the drain after a timeout uses kWaitPolls)
    const unsigned first_polls = p.wait_polls == 0 ? kWaitPolls : p.wait_polls < 0 ? 0u : (unsigned)p.wait_polls;
    UnitIdx pf{0, 0, 0, 0};
    if (tid == 0) {
        UnitIdx i0{0, 0, 0, 0}, i1{0, 0, 0, 0};
        load_index(0, i0);
        load_index(1, i1);
        if (!VL) {  // (x rows of a whole-T batch do not depend on the indices: send them first)
            if (iters > 0) issue_x(0, 0, TS);
            if (iters > 1) issue_x(1, 0, TS);
        }
        if (iters > 0) issue(0, i0, !VL);
        if (iters > 1) issue(1, i1, !VL);
        load_index(2, pf);
    }

    const int cl = tid * CPT;
    // products rounded one by one unless they are exact (bf16 times bf16)
    using CB = std::conditional_t<MIXED, uint32_t, B>;
    // unit u = blockIdx.x + k * gridDim.x as (sequence, channel block), stepped without divisions
    const int g_s = (int)gridDim.x / nblk, g_b = (int)gridDim.x - g_s * nblk;
    int q = (int)blockIdx.x / nblk, cb = (int)blockIdx.x - q * nblk;  // q: index into the sequence list
    constexpr int LOG_CPT = CPT == 4 ? 2 : 3;
    const int lanes = p.head_dim >> LOG_CPT;  // threads per L2 group
    // taps and bias of the current channel block, channels in pairs (paired fp32 lanes: the same
    // operations per lane as scalar code, half the instructions)
    constexpr int P = CPT / 2;
    f2 wt2[P][W];
    f2 bs2[P];
    int wcb = -1;
    for (int k = 0; k < iters; ++k) {
        const int st = k & 1;
        const int s = seq_at(q) & 0xffff;  // (a list entry of packed drafts also holds the chunk)
        const unsigned char *stg = smem + st * stage_bytes;
        unsigned char *const img = img0 + (k & 1) * img_bytes;
        unsigned char *const stimg = img + rb;
        const int c0 = cb * BC;
        const int nch = min(BC, p.dim - c0);
        const bool act = cl < nch;
        const int c = c0 + cl;
        if (cb != wcb) {  // once per block when the grid is a multiple of the channel-block count
            wcb = cb;
            float wt[CPT][W], bs[CPT];
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
                if (has_bias) {
                    uint32_t bw[NW];
                    ldv<VX, NW>(bw, reinterpret_cast<const B *>(p.bias) + c);
#pragma unroll
                    for (int e = 0; e < CPT; ++e) bs[e] = elem_f<B>(bw, e);
                }
            }
#pragma unroll
            for (int q = 0; q < P; ++q) {
                bs2[q] = f2_pack(bs[2 * q], bs[2 * q + 1]);
#pragma unroll
                for (int j = 0; j < W; ++j) wt2[q][j] = f2_pack(wt[2 * q][j], wt[2 * q + 1][j]);
            }
        }

        const bool ok = mbar_wait_bounded(&bar[st], (unsigned)((k >> 1) & 1), first_polls);
        const int slot = ok ? info[st] : -1;
        const int off = info[2 + st];
        const bool go = slot >= 0;
        const int Ts = VL ? (info[4 + st] & 0xffff) : TS;   // draft tokens of this unit's sequence
        const int chunk = VL ? (info[4 + st] >> 16) : 0;    // which chunk of them
        const int t0 = chunk * TS;                          // its first token
        const int nt = VL ? max(0, min(TS, Ts - t0)) : TS;  // its token count
        const bool first = chunk == 0;                      // (reads and writes the state)
        const bool tail = chunked && first && Ts > TS;      // (its committed window is in the tail rows)
        const long long row0 = VL ? info[6 + st] : 0;       // the sequence's first packed row

        f2 fw2[P][R + TS];  // inputs widened to fp32, channel pairs: [0, R) committed window, then x
        uint32_t xr[TS][NW];    // raw x rows
        uint32_t sw[R * NWS];   // raw committed window, channel-major [CPT][R]
        if (go && act) {
#pragma unroll
            for (int t = 0; t < TS; ++t) {
                if (!VL || t < nt) {
                    ldv<VX, NW>(xr[t], stg + ((long long)t * BC + cl) * ES);
                } else {
#pragma unroll
                    for (int i = 0; i < NW; ++i) xr[t][i] = 0u;  // (no row: keep stale bits out)
                }
            }
            if (VL && !first) {
                // a later chunk: its first W-1 inputs are the halo rows (the x rows before it)
                uint32_t hr[R][NW];
#pragma unroll
                for (int j = 0; j < R; ++j) ldv<VX, NW>(hr[j], stg + ((long long)(TS + j) * BC + cl) * ES);
#pragma unroll
                for (int i = 0; i < R * NWS; ++i) {
                    if (ESS == 2) {
                        const int a = 2 * i, b2 = 2 * i + 1;  // elements (channel a / R, input a % R)
                        sw[i] = pack_halves(elem_raw<S>(hr[a % R], a / R), elem_raw<S>(hr[b2 % R], b2 / R));
                    } else {
                        sw[i] = hr[i % R][i / R];
                    }
                }
            } else if (hist_t) {
                // staged column kk holds the committed window's column kk of all BC channels
                uint32_t cw[R][NWS];
#pragma unroll
                for (int kk = 0; kk < R; ++kk)
                    ldv<pipe_align(CPT * ESS), NWS>(cw[kk], stg + xb + ((long long)kk * BC + cl) * ESS);
#pragma unroll
                for (int i = 0; i < R * NWS; ++i) {
                    if (ESS == 2) {
                        const int a = 2 * i, b2 = 2 * i + 1;  // elements (channel a / R, column a % R)
                        sw[i] = pack_halves(elem_raw<S>(cw[a % R], a / R), elem_raw<S>(cw[b2 % R], b2 / R));
                    } else {
                        sw[i] = cw[i % R][i / R];
                    }
                }
            } else if (whole_rows) {
                // the committed window sits at columns [off, off+W-1) of each staged row
                using U = std::conditional_t<ESS == 2, unsigned short, unsigned>;
                const U *row = reinterpret_cast<const U *>(stg + xb) + (long long)cl * SC + off;
                U v[CPT * R];
#pragma unroll
                for (int e = 0; e < CPT; ++e)
#pragma unroll
                    for (int kk = 0; kk < R; ++kk) v[e * R + kk] = row[e * SC + kk];
#pragma unroll
                for (int i = 0; i < R * NWS; ++i)
                    sw[i] = ESS == 2 ? ((uint32_t)v[2 * i] | ((uint32_t)v[(2 * i + 1) % (CPT * R)] << 16)) : (uint32_t)v[i];
            } else {
                ldv<VS, R * NWS>(sw, stg + xb + (long long)cl * R * ESS);
            }
#pragma unroll
            for (int e = 0; e < CPT; ++e)
#pragma unroll
                for (int kk = 0; kk < R; ++kk) {
                    if (e % 2 == 0) fw2[e / 2][kk] = f2_pack(elem_f<S>(sw, e * R + kk), elem_f<S>(sw, (e + 1) * R + kk));
                }

            // word and half holding input j of channel e (j < R: committed window, else x_{j-R})
            auto word_of = [&](int e, int j) -> uint32_t { return j < R ? sw[(e * R + j) / EW] : xr[j - R][e / EW]; };
            auto half_of = [&](int e, int j) -> int { return j < R ? (e * R + j) % EW : e % EW; };
            // raw bits of input j of channel e in the state's type (x elements converted)
            auto elem_bits = [&](int e, int j) -> uint32_t {
                if constexpr (MIXED)
                    return j < R ? elem_raw<S>(sw, e * R + j) : convert_bits<B, S>(elem_raw<B>(xr[j - R], e));
                else
                    return ES == 2 ? (word_of(e, j) >> (16 * half_of(e, j))) & 0xffffu : word_of(e, j);
            };
            // word i (state type) of a channel-major run of n columns starting at input j0
            auto run_word = [&](int i, int n, int j0) -> uint32_t {
                if constexpr (MIXED) {
                    if constexpr (ESS == 2) {
                        const int a = 2 * i, b = 2 * i + 1;
                        return pack_halves(elem_bits(a / n, j0 + a % n), elem_bits(b / n, j0 + b % n));
                    }
                    return elem_bits(i / n, j0 + i % n);
                }
                if (ES == 2) {
                    const int a = 2 * i, b = 2 * i + 1;
                    return halves(word_of(a / n, j0 + a % n), half_of(a / n, j0 + a % n), word_of(b / n, j0 + b % n),
                                  half_of(b / n, j0 + b % n));
                }
                return word_of(i / n, j0 + i % n);
            };
            if (recomp) {
                // outputs only: no snapshots, and the state keeps the pre-verify window
            } else if (dedup_t || hist_t) {
                // column q (input q+1) of the thread's CPT channels, in the state's type, at image
                // position [q][cl]
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int j = q + 1;
                    uint32_t w[NWS];
#pragma unroll
                    for (int i = 0; i < NWS; ++i) {
                        if (ESS == 2)
                            w[i] = pack_halves(elem_bits(2 * i, j), elem_bits(2 * i + 1, j));
                        else
                            w[i] = elem_bits(i, j);
                    }
                    stv<pipe_align(CPT * ESS), NWS>(img + ((long long)q * BC + cl) * ESS, w);
                }
            } else if (!dense) {
                uint32_t im[Q * NWS];  // CPT channels x Q columns; column q holds input q+1
#pragma unroll
                for (int i = 0; i < Q * NWS; ++i) im[i] = run_word(i, Q, 1);
                stv<VI, Q * NWS>(img + (long long)tid * CPT * Q * ESS, im);
            } else {
                S *wsq = reinterpret_cast<S *>(p.win) + (long long)s * p.w_seq + (long long)c * R;
#pragma unroll
                for (int t = 0; t < TS; ++t) {
                    if (VL && t >= nt) break;
                    uint32_t w[R * NWS];
#pragma unroll
                    for (int i = 0; i < R * NWS; ++i) w[i] = run_word(i, R, t + 1);
                    stv<VS, R * NWS>(wsq + (long long)(t0 + t) * p.w_step, w);
                }
            }
            // committed window = full[T_s .. T_s+W-2], channel-major [CPT][R] words
            uint32_t fin[R * NWS];
#pragma unroll
            for (int i = 0; i < R * NWS; ++i) fin[i] = 0u;
            if (VL && !first) {
                // a later chunk writes no committed window (chunk 0 does)
            } else if constexpr (VL) {
                // column kk is x row T_s+kk-R when that is >= 0 (read back from the stage: from the
                // chunk's rows, or from the tail rows when the draft is longer than a chunk), else
                // committed-window column T_s+kk (T_s < W-1)
                uint32_t col[R][NW];
#pragma unroll
                for (int kk = 0; kk < R; ++kk) {
                    const int j = Ts + kk;
                    if (tail) {
                        ldv<VX, NW>(col[kk], stg + ((long long)(TS + kk) * BC + cl) * ES);
                    } else if (j >= R) {
                        ldv<VX, NW>(col[kk], stg + ((long long)(j - R) * BC + cl) * ES);
                    } else {
#pragma unroll
                        for (int i = 0; i < NW; ++i) {
                            uint32_t lo = 0u, hi = 0u;
#pragma unroll
                            for (int jj = 0; jj < R; ++jj) {
                                if (jj != j) continue;
                                lo = elem_raw<S>(sw, (EW * i) * R + jj);
                                if (EW == 2) hi = elem_raw<S>(sw, (EW * i + 1) * R + jj);
                            }
                            col[kk][i] = EW == 2 ? pack_halves(lo, hi) : lo;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < R * NWS; ++i) {
                    if (ES == 2) {
                        const int a = 2 * i, b2 = 2 * i + 1;
                        fin[i] = pack_halves(elem_raw<S>(col[a % R], a / R), elem_raw<S>(col[b2 % R], b2 / R));
                    } else {
                        fin[i] = col[i % R][i / R];
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < R * NWS; ++i) fin[i] = run_word(i, R, TS);
            }
            if (wide) {
                // the thread's CPT staged rows (CPT * SC contiguous elements, a whole number of
                // words) into the state image, the committed window over columns [0, W-1).  (Only
                // chunk 0 of a packed draft writes the state.)
                if (!recomp && first) {
                    const int nwords = CPT * SC * ESS / 4;
                    const unsigned *src = reinterpret_cast<const unsigned *>(stg + xb) + (long long)tid * nwords;
                    unsigned *dst = reinterpret_cast<unsigned *>(stimg) + (long long)tid * nwords;
                    for (int i = 0; i < nwords; ++i) dst[i] = src[i];
                    S *const drow = reinterpret_cast<S *>(stimg) + (long long)cl * SC;
#pragma unroll
                    for (int e = 0; e < CPT; ++e)
#pragma unroll
                        for (int kk = 0; kk < R; ++kk) drow[e * SC + kk] = (S)elem_raw<S>(fin, e * R + kk);
                }
            } else if (direct_state) {
                if (first)  // (chunk 0 of a packed draft writes the state)
                    stv<VS, R * NWS>(reinterpret_cast<S *>(p.state) + (long long)slot * p.st_slot + (long long)c * R, fin);
            } else if (!hist && !recomp) {
                stv<VS, R * NWS>(stimg + (long long)tid * CPT * R * ESS, fin);
            }
        }
        fence_smem_to_async();
        // the image buffer written next unit was last read by this unit's predecessor's bulk copy,
        // the only group thread 0 can still have in flight
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
        // one barrier per unit: images complete, stage st moved to registers, and the vote on
        // whether any thread's wait timed out
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                // this unit and every later unit of the block stay (partly) unwritten: flag their
                // sequences (padded ones excepted)
                if (p.err)
                    for (int k2 = k; k2 < iters; ++k2) {
                        int s2, c2, n2;
                        unit_of(k2, s2, c2, n2);
                        if (!p.cache_idx || __ldg(p.cache_idx + s2) >= 0) atomicOr(p.err + s2, kSeqTimeout);
                    }
                // drain the copies still in flight into this block's shared memory (bounded)
                mbar_wait_bounded(&bar[st], (unsigned)((k >> 1) & 1), kWaitPolls);
                if (k + 1 < iters) mbar_wait_bounded(&bar[st ^ 1], (unsigned)(((k + 1) >> 1) & 1), kWaitPolls);
            }
            return;
        }
        // the row image (dedup row, or history row): whole rows leave as one bulk copy.  A packed
        // draft's unit writes columns [qd, qd + cnt) of each channel's row from image columns
        // [qs, qs + cnt): its own inputs only (chunk 0 also the window's columns 1 .. W-2)
        const bool full_row = !VL || (!chunked && Ts == TS);
        const int qs = first ? 0 : R - 1, qd = first ? 0 : t0 + R - 1;
        const int cnt = first ? (nt > 0 ? nt + R - 1 : 0) : nt;
        S *const row_dst = hist ? reinterpret_cast<S *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * Qrow
                                : reinterpret_cast<S *>(p.win) + (long long)s * p.w_seq + (long long)c0 * Qrow;
        if (tid == 0) {
            if (go && !recomp) {
                if (dedup_t || hist_t) {
                    // one bulk copy per column (of the window row, or of the column-major state row)
                    const int ncols = full_row ? Q : cnt;
                    S *const colb = hist_t ? reinterpret_cast<S *>(p.state) + (long long)slot * p.st_slot + c0
                                           : reinterpret_cast<S *>(p.win) + (long long)s * p.w_seq + c0;
                    const long long cstride = hist_t ? p.st_col : p.w_col;
                    for (int q2 = 0; q2 < ncols; ++q2)
                        bulk_store(colb + (long long)(qd + q2) * cstride, img + (long long)(qs + q2) * BC * ESS,
                                   (unsigned)(nch * ESS));
                } else if (!dense && full_row) {
                    bulk_store(row_dst, img, (unsigned)(nch * Q * ESS));
                }
                if (!hist && first && !direct_state)  // (SC == W-1 unless the rows are wide)
                    bulk_store(reinterpret_cast<S *>(p.state) + (long long)slot * p.st_slot + (long long)c0 * SC, stimg,
                               (unsigned)(nch * SC * ESS));
                asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
            }
            if (k + 2 < iters) {
                issue(k + 2, pf, false);
                load_index(k + 3, pf);
            }
        }
        if (VL && go && !recomp && !dense && !dedup_t && !hist_t && !full_row && cnt > 0) {
            if (!chunked) {
                // one chunk, columns [0, T_s+W-2): word w of the staged image holds elements 2w,
                // 2w+1 (bf16) or w (fp32) of the block's [nch][Q] run, Q = the row's width
                const unsigned *iw = reinterpret_cast<const unsigned *>(img);
                unsigned *dw = reinterpret_cast<unsigned *>(row_dst);
                const int nwords = nch * Q * ESS / 4;
                for (int w = tid; w < nwords; w += (int)blockDim.x) {
                    const unsigned v = iw[w];
                    if (ESS == 4) {
                        if (w % Q < cnt) dw[w] = v;
                    } else {
                        const bool lo = (2 * w) % Q < cnt, hi = (2 * w + 1) % Q < cnt;
                        if (lo && hi) {
                            dw[w] = v;
                        } else if (lo) {
                            reinterpret_cast<unsigned short *>(dw)[2 * w] = (unsigned short)(v & 0xffffu);
                        } else if (hi) {
                            reinterpret_cast<unsigned short *>(dw)[2 * w + 1] = (unsigned short)(v >> 16);
                        }
                    }
                }
            } else {
                // a chunk of a longer draft: element by element, channel-major, consecutive threads
                // on consecutive elements; element i = (channel i / cnt, column i % cnt), stepped
                // by the block size without a division per element
                using U = std::conditional_t<ESS == 2, unsigned short, unsigned>;
                const U *ie = reinterpret_cast<const U *>(img);
                U *de = reinterpret_cast<U *>(row_dst);
                const int nthr = (int)blockDim.x;
                const int dcc = nthr / cnt, dq = nthr - dcc * cnt;
                int cc = tid / cnt, q2 = tid - cc * cnt;
                for (int i = tid; i < nch * cnt; i += nthr) {
                    de[(long long)cc * Qrow + qd + q2] = ie[cc * Q + qs + q2];
                    cc += dcc;
                    q2 += dq;
                    if (q2 >= cnt) {
                        q2 -= cnt;
                        ++cc;
                    }
                }
            }
        }
        if (go) {
            const bool l2_block = c0 < p.qk_channels;
            const bool l2_mine = c < p.qk_channels;
            float y[TS][CPT];
            if (act) {
                // conv + SiLU; one range check for the whole unit (see silu_fast)
                float lo = 0.0f;
#pragma unroll
                for (int t = 0; t < TS; ++t) {
#pragma unroll
                    for (int q = 0; q < P; ++q) fw2[q][R + t] = f2_pack(elem_f<B>(xr[t], 2 * q), elem_f<B>(xr[t], 2 * q + 1));
#pragma unroll
                    for (int q = 0; q < P; ++q) {
                        const f2 acc = conv_chain2<CB, W>(bs2[q], wt2[q], &fw2[q][t]);
                        f2_unpack(silu_fast2(acc), y[t][2 * q], y[t][2 * q + 1]);
                        float a0, a1;
                        f2_unpack(acc, a0, a1);
                        lo = fminf(lo, fminf(a0, a1));
                    }
                }
                if (lo < -80.0f) {
                    // only the values below -80 take the exact form (the same bits as silu())
#pragma unroll
                    for (int t = 0; t < TS; ++t)
#pragma unroll
                        for (int q = 0; q < P; ++q) {
                            float a0, a1;
                            f2_unpack(conv_chain2<CB, W>(bs2[q], wt2[q], &fw2[q][t]), a0, a1);
                            if (a0 < -80.0f) y[t][2 * q] = silu_exact(a0);
                            if (a1 < -80.0f) y[t][2 * q + 1] = silu_exact(a1);
                        }
                }
            } else {
#pragma unroll
                for (int t = 0; t < TS; ++t)
#pragma unroll
                    for (int e = 0; e < CPT; ++e) y[t][e] = 0.0f;
            }
            if (l2_block) {
                float ss[TS];
#pragma unroll
                for (int t = 0; t < TS; ++t) ss[t] = sum_squares<CPT>(y[t]);
                if (CPT == 4 && lanes > 1) {
#pragma unroll
                    for (int t = 0; t < TS; ++t) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], 1);
                }
                for (int o = lanes >> 1; o >= (CPT == 4 ? 2 : 1); o >>= 1) {
#pragma unroll
                    for (int t = 0; t < TS; ++t) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
                }
                if (l2_mine) {
#pragma unroll
                    for (int t = 0; t < TS; ++t) {
                        const float r = rsqrtf(ss[t] + p.eps);
                        const f2 r2 = f2_pack(r, r);
#pragma unroll
                        for (int q = 0; q < P; ++q)
                            f2_unpack(f2_mul(f2_pack(y[t][2 * q], y[t][2 * q + 1]), r2), y[t][2 * q], y[t][2 * q + 1]);
                    }
                }
            }
            if (act) {
                B *os = reinterpret_cast<B *>(p.out) + (VL ? (row0 + t0) * p.out_tok : (long long)s * p.out_seq) + c;
#pragma unroll
                for (int t = 0; t < TS; ++t) {
                    if (VL && t >= nt) break;
                    uint32_t ow[NW];
                    if (ES == 2) {
#pragma unroll
                        for (int i = 0; i < NW; ++i) {
                            __nv_bfloat162 h = __floats2bfloat162_rn(y[t][2 * i], y[t][2 * i + 1]);
                            ow[i] = *reinterpret_cast<uint32_t *>(&h);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < NW; ++i) ow[i] = __float_as_uint(y[t][i]);
                    }
                    stv<VX, NW>(os + (long long)t * p.out_tok, ow);
                }
            }
        }
        q += g_s;
        cb += g_b;
        if (cb >= nblk) {
            cb -= nblk;
            ++q;
        }
    }
    // keep the block's shared memory alive until the last bulk copies have read it
    if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

}  // namespace cvk
