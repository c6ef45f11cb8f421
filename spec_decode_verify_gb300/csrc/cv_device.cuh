// Shared device definitions of the verify/commit kernels (sm_103a): launch parameters and the
// element helpers.  B is the raw bit type of one element: uint16_t for bf16, uint32_t for fp32.
// Snapshot and state traffic always moves these raw bits; only the conv arithmetic widens them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cvk {

struct VerifyParams {
    const void *x;
    long long x_seq, x_tok;
    void *out;
    long long out_seq, out_tok;
    void *state;
    long long st_slot, st_ch;
    long long st_col;  // state column stride: 1, or (history rows only) column-major rows with st_ch == 1
    const int *cache_idx;
    const int *state_off;
    const void *weight;
    const void *bias;
    void *win;
    long long w_seq, w_step, w_ch, w_col;  // for the dedup layout w_step already equals w_col
    int *err;
    int n_seq, T, dim, n_slots, state_cols;
    int qk_channels, head_dim, pitch;      // pitch: elements per shared-memory row (generic kernel)
    float eps;
    int dedup;
    int dedup_t;  // dedup rows laid out transposed: channel stride 1, one contiguous run per column
    int hist;     // history-row state: the snapshot row goes into the state row (no window buffer)
    int compact;  // pipelined kernel: walk only the sequences with a cache slot >= 0 (list in shared memory)
    int recomp;   // recompute rollback: outputs only (no snapshots, state not written)
    const int *parent;  // tree verify: [n_seq][T] parent of each draft token, or null (a chain)
    int x_vec, out_vec, st_vec, w_vec, b_vec;  // 16-byte vector access allowed (checked on the host)
    int st_packed;  // tree verify: the committed windows are packed, 16-byte-aligned [dim][W-1] rows
    int st_rows;    // one-pass verify: packed state rows wider than the window, staged whole (16-byte
                    // aligned [dim][state_cols] runs per slot)
    int wait_polls;  // polls of the first bounded wait per unit: 0 = the default, < 0 = none (gives up at once)
    const int *cu_draft;  // packed ragged drafts: [n_seq + 1] row offsets into x and out, or null
    int total_tokens;     // rows of x and out when cu_draft is given
};

// Pipelined verify: shared memory after the stages and images holds 2 mbarriers, then 8 ints of
// unit information (slots, state offsets, draft counts, first rows of the two units in flight),
// then the listing scratch (pipe_aux_ints of them: 4 warp counts, or list_chunks' counts) and the
// list of active sequences (or of chunks).
constexpr int kPipeInfoBytes = 16 + 32;
__host__ __device__ constexpr int pipe_aux_ints(bool varlen, int TS) { return varlen ? 5 * (TS + 2) : 4; }

constexpr int kSeqTimeout = 8;  // err bit: a bounded wait for a bulk copy gave up
__host__ __device__ constexpr int pipe_align(int bytes) { return bytes % 16 == 0 ? 16 : 8; }

// Tree verify: channels per block, 8 per lane of a warp.
constexpr int kTreeChannels = 256;

struct CommitParams {
    void *state;
    long long st_slot, st_ch;
    const int *cache_idx;
    const void *win;
    long long w_seq, w_step, w_ch, w_col;
    const int *accept_len;
    int *err;
    int n_seq, T, dim, n_slots;
    // 0: element by element, 1: packed dense snapshot -> packed state, 2: packed dedup row -> packed
    // state, 3: recompute from x, 4: packed transposed dedup row (channel stride 1) -> packed state
    int mode;
    const void *x;  // mode 3: the verify's input
    long long x_seq, x_tok;
    const int *cu_draft;  // packed ragged drafts of the matching verify, or null (T tokens each)
    int total_tokens;
    int wait_polls;  // polls of the bounded wait for the staged rows: 0 = the default, < 0 = none
};

struct PrefillParams {
    const void *x;
    long long x_tok;
    void *out;
    long long out_tok;
    const int *cu_seqlens;  // [n_seq + 1]
    void *state;
    long long st_slot, st_ch;
    const int *cache_idx;
    const int *has_init;  // [n_seq] or null (every sequence has an initial window)
    const void *weight;
    const void *bias;
    int *err;
    int n_slots, total_tokens, max_seqlen, dim, qk_channels, head_dim;
    float eps;
    int x_vec, out_vec;  // vector access of x / out allowed (checked on the host)
    int chunk;           // tokens per block
};

// Per-sequence status shared by both kernels: 1 = slot out of range, 2 = state offset out of range.
__device__ __forceinline__ int seq_status(int slot, int off, int n_slots, int state_cols, int R) {
    int st = 0;
    if (slot >= 0) {
        if (slot >= n_slots) st |= 1;
        if (off < 0 || off > state_cols - R) st |= 2;
    }
    return st;
}

constexpr int kSeqBadSpan = 16;  // err bit: a packed draft span (or prefill span) is invalid

// Packed ragged drafts (sglang PR #46184, "Related upstream work": target verify on packed ragged
// tokens): sequence s owns rows [cu[s], cu[s+1]) of x and out.  Sets ts = its draft count and row0
// = its first row; returns kSeqBadSpan when the span is reversed, leaves [0, total) or holds more
// than T rows (the sequence is then left untouched).
__device__ __forceinline__ int span_status(int b, int e, int T, int total) {
    return (b < 0 || e < b || e > total || e - b > T) ? kSeqBadSpan : 0;
}
__device__ __forceinline__ int draft_span(const int *cu, int s, int T, int total, int &ts, int &row0) {
    const int b = __ldg(cu + s), e = __ldg(cu + s + 1);
    row0 = b;
    ts = e - b;
    return span_status(b, e, T, total);
}

// The work list of a persistent verify kernel over packed ragged drafts, built identically by every
// block (block-wide: every thread of a block of at most 4 warps calls it).  A sequence with a cache
// slot >= 0 contributes one entry per chunk of at most TS of its T_s draft tokens (one entry when
// T_s = 0 or its span is bad), encoded (chunk << 16) | sequence.  Entries are ordered by the number
// of tokens they hold, most first, so that units of similar cost come together in the round-robin
// walk; ties are ordered by chunk, then sequence.  A stable counting sort: a shared-memory
// histogram of the keys (TS - tokens), its prefix sums, then each entry's place from its key's
// start, the counts of earlier warps in the chunk of sequences and its rank among its warp's lanes
// of the same key (__match_any_sync).  scratch holds pipe_aux_ints(true, TS) ints of counts, then
// the list.  Returns its length.
__device__ __forceinline__ int list_chunks(const VerifyParams &p, int *scratch, int TS) {
    const int NB = TS + 1;             // keys 0 .. TS
    int *const cnt = scratch;          // [NB + 1]: bucket sizes, then each bucket's next position
    int *const wc = scratch + NB + 1;  // [NB][4]: per-warp counts of the current chunk of sequences
    int *const list = scratch + pipe_aux_ints(true, TS);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const int C = (p.T + TS - 1) / TS;  // chunks of the longest draft
    // the key of sequence i's chunk c, or -1 when it has none
    auto key_of = [&](int i, int c) -> int {
        if (i >= p.n_seq || (p.cache_idx && __ldg(p.cache_idx + i) < 0)) return -1;
        int ts, r0;
        if (draft_span(p.cu_draft, i, p.T, p.total_tokens, ts, r0)) return c == 0 ? TS : -1;
        if (c > 0 && c * TS >= ts) return -1;
        return TS - min(TS, ts - c * TS);
    };
    for (int v = tid; v <= NB; v += nt) cnt[v] = 0;
    __syncthreads();
    for (int c = 0; c < C; ++c)
        for (int i0 = 0; i0 < p.n_seq; i0 += nt) {
            const int key = key_of(i0 + tid, c);
            if (key >= 0) atomicAdd(cnt + key, 1);
        }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int v = 0; v < NB; ++v) {
            const int n = cnt[v];
            cnt[v] = run;
            run += n;
        }
        cnt[NB] = run;
    }
    __syncthreads();
    const int n_list = cnt[NB];
    for (int c = 0; c < C; ++c)
        for (int i0 = 0; i0 < p.n_seq; i0 += nt) {
            const int i = i0 + tid;
            const int key = key_of(i, c);
            for (int v = tid; v < 4 * NB; v += nt) wc[v] = 0;
            __syncthreads();
            const unsigned m = __match_any_sync(0xffffffffu, key);
            if (key >= 0 && lane == __ffs(m) - 1) wc[key * 4 + warp] = __popc(m);
            __syncthreads();
            if (key >= 0) {
                int before = 0;
                for (int w = 0; w < warp; ++w) before += wc[key * 4 + w];
                list[cnt[key] + before + __popc(m & ((1u << lane) - 1u))] = (c << 16) | i;
            }
            __syncthreads();
            for (int v = tid; v < NB; v += nt) cnt[v] += wc[v * 4] + wc[v * 4 + 1] + wc[v * 4 + 2] + wc[v * 4 + 3];
            __syncthreads();
        }
    return n_list;
}

template <typename B> __device__ __forceinline__ float widen(B b);
template <> __device__ __forceinline__ float widen<uint16_t>(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
template <> __device__ __forceinline__ float widen<uint32_t>(uint32_t b) { return __uint_as_float(b); }

template <typename B> __device__ __forceinline__ B narrow(float f);
template <> __device__ __forceinline__ uint16_t narrow<uint16_t>(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <> __device__ __forceinline__ uint32_t narrow<uint32_t>(float f) { return __float_as_uint(f); }

// Raw bits of a value that was widened from B (exact: bf16 -> fp32 -> upper half is the identity,
// NaN payloads included, because no arithmetic touched it).
template <typename B> __device__ __forceinline__ uint32_t raw_of(float f) {
    return sizeof(B) == 2 ? (__float_as_uint(f) >> 16) : __float_as_uint(f);
}

// Raw bits of an element of type BX as an element of type BS: the same bits when the types agree,
// bf16 widened exactly to fp32, or fp32 rounded to the nearest bf16 (ties to even; any NaN becomes
// the quiet NaN 0x7fc0).
template <typename BX, typename BS>
__device__ __forceinline__ uint32_t convert_bits(uint32_t v) {
    if constexpr (sizeof(BX) == sizeof(BS)) {
        return v;
    } else if constexpr (sizeof(BX) == 2) {
        return v << 16;
    } else {
        if ((v & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
        return __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v)));
    }
}

// Element i (0..7) of 8 packed elements held as 32-bit words, widened to fp32.
template <typename B> __device__ __forceinline__ float elem_f(const uint32_t *w, int i) {
    if (sizeof(B) == 2) return (i & 1) ? __uint_as_float(w[i >> 1] & 0xffff0000u) : __uint_as_float(w[i >> 1] << 16);
    return __uint_as_float(w[i]);
}

// Raw bits of element i of 8 packed elements.
template <typename B> __device__ __forceinline__ uint32_t elem_raw(const uint32_t *w, int i) {
    if (sizeof(B) == 2) return (w[i >> 1] >> ((i & 1) * 16)) & 0xffffu;
    return w[i];
}

// One word holding half h0 of word a (low half) and half h1 of word b (high half): one byte
// permute with a selector that is a compile-time constant once the callers are unrolled.
__device__ __forceinline__ uint32_t halves(uint32_t a, int h0, uint32_t b, int h1) {
    return __byte_perm(a, b, (2 * h0) | ((2 * h0 + 1) << 4) | ((4 + 2 * h1) << 8) | ((5 + 2 * h1) << 12));
}

// Two raw 16-bit values -> one word (lo in the low half).  For fp32 only lo is used.
__device__ __forceinline__ uint32_t pack_halves(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x5410); }

// Two fp32 lanes in one 64-bit register.  The paired fp32 instructions (fma / mul / add .f32x2,
// sm_100 and later) compute each lane exactly as the scalar instruction does (IEEE fp32, round to
// nearest even) in one issue slot, so paired arithmetic gives the scalar results bit for bit.
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// SiLU(a) = a / (1 + exp(-a)).  silu_fast evaluates exp(-a) = 2^(-a * log2 e) with the
// ex2.approx instruction and the quotient as a * rcp.approx(1 + exp(-a)); relative error a few
// fp32 ulp.  Both instructions flush subnormals, which matters only below a = -87
// (1 + exp(-a) > 2^126): silu_exact is the plain expression, taken for every value below -80 and
// for no other (see silu), so each output's bits depend on its own conv result alone, whichever
// kernel computes it and whatever other values it is computed beside.
__device__ __forceinline__ float silu_fast(float a) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(a * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return a * r;
}
__device__ __forceinline__ float silu_exact(float a) { return a / (1.0f + expf(-a)); }
// silu_fast of two values in paired lanes: the same operations per lane, so the same bits.
__device__ __forceinline__ f2 silu_fast2(f2 a) {
    float t0, t1, e0, e1, r0, r1;
    f2_unpack(f2_mul(a, f2_pack(-1.4426950408889634f, -1.4426950408889634f)), t0, t1);
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
    float s0, s1;
    f2_unpack(f2_add(f2_pack(1.0f, 1.0f), f2_pack(e0, e1)), s0, s1);
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(s0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(s1));
    return f2_mul(a, f2_pack(r0, r1));
}

// SiLU of n values with one range check for the run (a branch realistic inputs never take); in
// that branch only the values below -80 switch to the exact form, so the result equals silu()
// value by value.
template <int N>
__device__ __forceinline__ void silu_run(const float *a, float *y) {
    float lo = a[0];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        y[i] = silu_fast(a[i]);
        lo = fminf(lo, a[i]);
    }
    if (lo < -80.0f) {
#pragma unroll
        for (int i = 0; i < N; ++i) y[i] = a[i] < -80.0f ? silu_exact(a[i]) : y[i];
    }
}
__device__ __forceinline__ float silu(float a) { return a < -80.0f ? silu_exact(a) : silu_fast(a); }

// Programmatic dependent launch (the library launches every kernel with programmatic stream
// serialization).  grid_dep_wait returns once the grids this one depends on in the stream have
// completed and their memory is visible -- immediately when there is no such dependency -- so
// every kernel calls it before its first global-memory access.  grid_dep_launch then lets the
// next grid in the stream be scheduled onto SMs this one frees, so its launch and prologue overlap
// this grid's tail (it still waits for this grid's completion before touching memory).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// One token's conv: the bias (or 0) first, then the W taps in order.  For bf16 elements every
// product of a tap and an input (8 significant bits each) is exact in fp32, so a fused
// multiply-add rounds exactly where the separate multiply and add would: the chain costs one
// instruction per tap and still equals the rounded-product definition bit for bit (a product
// below 2^-126 could round differently, far outside any real input).  For fp32 elements the
// product itself is rounded first, as the definition says.
template <typename B, int W>
__device__ __forceinline__ float conv_chain(float acc, const float *w, const float *in) {
#pragma unroll
    for (int j = 0; j < W; ++j) acc = sizeof(B) == 2 ? fmaf(w[j], in[j], acc) : __fadd_rn(acc, __fmul_rn(w[j], in[j]));
    return acc;
}

// conv_chain for two channels at once (paired lanes), each lane bit for bit the scalar chain.  The
// bf16 chain is paired fused multiply-adds.  The fp32 chain rounds each product before its add, so
// it stays scalar: a paired multiply feeding a paired add may be contracted into a fused one by the
// compiler (measured: the results then differed from the scalar chain), which the scalar .rn forms
// rule out.
template <typename B, int W>
__device__ __forceinline__ f2 conv_chain2(f2 acc, const f2 *w, const f2 *in) {
    if constexpr (sizeof(B) == 2) {
#pragma unroll
        for (int j = 0; j < W; ++j) acc = f2_fma(w[j], in[j], acc);
        return acc;
    } else {
        float a0, a1;
        f2_unpack(acc, a0, a1);
#pragma unroll
        for (int j = 0; j < W; ++j) {
            float w0, w1, x0, x1;
            f2_unpack(w[j], w0, w1);
            f2_unpack(in[j], x0, x1);
            a0 = __fadd_rn(a0, __fmul_rn(w0, x0));
            a1 = __fadd_rn(a1, __fmul_rn(w1, x1));
        }
        return f2_pack(a0, a1);
    }
}

// Sum of squares of a thread's CPT (4 or 8) values in one fixed order: a chain over each run of 4
// channels, then the runs added pairwise.  The xor-shuffle tree over lanes continues the same
// pairwise order, so the group sum is bit-identical whether a thread owns 4 or 8 channels.
template <int CPT>
__device__ __forceinline__ float sum_squares(const float *y) {
    static_assert(CPT == 4 || CPT == 8, "4 or 8 channels per thread");
    float a = y[0] * y[0];
    a = fmaf(y[1], y[1], a);
    a = fmaf(y[2], y[2], a);
    a = fmaf(y[3], y[3], a);
    if constexpr (CPT == 8) {
        float b = y[4] * y[4];
        b = fmaf(y[5], y[5], b);
        b = fmaf(y[6], y[6], b);
        b = fmaf(y[7], y[7], b);
        a = a + b;
    }
    return a;
}

// Vector access of `NWORDS` 32-bit words at an address aligned to VA bytes (8 or 16).
template <int VA, int NWORDS>
__device__ __forceinline__ void ldv(uint32_t *w, const void *p) {
    static_assert(VA == 8 || VA == 16, "vector width");
    if constexpr (VA == 16) {
        static_assert(NWORDS % 4 == 0, "16-byte vectors");
#pragma unroll
        for (int i = 0; i < NWORDS / 4; ++i) {
            const uint4 q = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = q.x, w[4 * i + 1] = q.y, w[4 * i + 2] = q.z, w[4 * i + 3] = q.w;
        }
    } else {
        static_assert(NWORDS % 2 == 0, "8-byte vectors");
#pragma unroll
        for (int i = 0; i < NWORDS / 2; ++i) {
            const uint2 q = reinterpret_cast<const uint2 *>(p)[i];
            w[2 * i] = q.x, w[2 * i + 1] = q.y;
        }
    }
}
template <int VA, int NWORDS>
__device__ __forceinline__ void stv(void *p, const uint32_t *w) {
    if constexpr (VA == 16) {
#pragma unroll
        for (int i = 0; i < NWORDS / 4; ++i)
            reinterpret_cast<uint4 *>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < NWORDS / 2; ++i) reinterpret_cast<uint2 *>(p)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 ld16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

__device__ __forceinline__ unsigned smem_u32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

// Dynamic shared memory the launch provided, in bytes.  Kernels that carve a layout out of it
// compare the two on entry and return without touching anything when the layout does not fit.
__device__ __forceinline__ unsigned dynamic_smem_bytes() {
    unsigned v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

// Shared -> global bulk copy (TMA, no tensor map): both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// ---- mbarrier + bulk (TMA) loads for the pipelined kernel
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
// Arrive once and announce `bytes` of asynchronous transactions that complete the phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Announce `bytes` more asynchronous transactions for the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for the phase with the given parity to complete, giving up after `limit` polls (each poll
// may suspend the thread for a hardware-defined time).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity, unsigned limit) {
    for (unsigned i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Global -> shared bulk copy completing `bytes` transactions on `bar`: 16-byte aligned addresses,
// bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(sdst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// L2 prefetch hint of `bytes` (a multiple of 16) from a 16-byte-aligned global address.
__device__ __forceinline__ void bulk_prefetch_l2(const void *gsrc, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(gsrc), "r"(bytes) : "memory");
}
// L2 prefetch hints for n runs of `bytes` bytes, `stride` bytes apart, from `base`, when every run
// starts on a 16-byte boundary and is a multiple of 16 bytes (else nothing: hints only).
__device__ __forceinline__ void prefetch_runs_l2(const void *base, long long stride, int n, long long bytes) {
    if ((reinterpret_cast<uintptr_t>(base) & 15u) || (stride & 15) || (bytes & 15) || bytes <= 0) return;
    const unsigned char *b = reinterpret_cast<const unsigned char *>(base);
    for (int i = 0; i < n; ++i) bulk_prefetch_l2(b + (long long)i * stride, (unsigned)bytes);
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

}  // namespace cvk
