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
    int x_vec, out_vec, st_vec, w_vec, b_vec;  // 16-byte vector access allowed (checked on the host)
};

struct CommitParams {
    void *state;
    long long st_slot, st_ch;
    const int *cache_idx;
    const void *win;
    long long w_seq, w_step, w_ch, w_col;
    const int *accept_len;
    int *err;
    int n_seq, T, dim, n_slots;
    int mode;  // 0: element by element, 1: packed dense snapshot -> packed state, 2: packed dedup row -> packed state
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

// Two raw 16-bit values -> one word (lo in the low half).  For fp32 only lo is used.
__device__ __forceinline__ uint32_t pack_halves(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x5410); }

// SiLU(a) = a * sigmoid(a), sigmoid through the exp intrinsic and the approximate reciprocal
// instruction (rcp.approx keeps subnormal results, so a very negative a still yields its tiny
// value and a -> -inf gives -0 like a / (1 + exp(-a))).  Relative error a few fp32 ulp.
__device__ __forceinline__ float silu(float a) {
    const float d = 1.0f + __expf(-a);
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return a * r;
}

__device__ __forceinline__ uint4 ld16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

__device__ __forceinline__ unsigned smem_u32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

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

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

}  // namespace cvk
