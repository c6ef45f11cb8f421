// Internal: the kernel tables each instantiation unit provides to the C ABI layer.
#pragma once

#include "cv_device.cuh"

namespace cvk {

using VerifyKernel = void (*)(VerifyParams);
using CommitKernel = void (*)(CommitParams);
using PrefillKernel = void (*)(PrefillParams);

// Largest T compiled with T as a template parameter (fully unrolled token loop, dedup row built
// in registers).  Above it the dense layout runs the chunked kernel and the dedup layout the
// general kernel.
constexpr int kMaxStaticT = 17;
// Largest T of the pipelined kernel compiled for mixed dtypes; above it they take the general kernel.
constexpr int kMaxMixedT = 8;

struct KernelSet {
    // fast[c][T]: c = 0 for 4 channels per thread, 1 for 8; T in 1..max_static_t compiled with T
    // as a constant, [c][0] = chunked, any T, dense layout only
    VerifyKernel fast[2][kMaxStaticT + 1];
    // pipe[c][T]: persistent, bulk-copy pipelined, T in 1..max_static_t (index 0 unused)
    VerifyKernel pipe[2][kMaxStaticT + 1];
    // pipe_mixed[c][T]: the same with the state and the snapshots in the other dtype (bf16 <-> fp32),
    // T in 1..kMaxMixedT
    VerifyKernel pipe_mixed[2][kMaxMixedT + 1];
    int max_static_t;
    VerifyKernel generic;
    VerifyKernel tree;  // draft tokens with parents (dense snapshots)
    VerifyKernel generic_mixed;  // state and snapshots in the other dtype (bf16 <-> fp32)
    CommitKernel commit;         // element by element (mode 0)
    CommitKernel commit_packed;  // packed dense snapshots into packed state rows (mode 1)
    CommitKernel commit_wide;    // packed dense snapshots into packed rows wider than the window (mode 5)
    CommitKernel commit_rows;
    CommitKernel commit_cols;
    CommitKernel commit_recompute;
    CommitKernel commit_recompute_vec;
    // prefill[c]: c = 0 for 4 channels per thread, 1 for 8
    PrefillKernel prefill[2];
};

// The pipelined kernel for packed ragged drafts, pipe[c][T] as in KernelSet (T = the largest draft
// count), compiled in translation units of their own.
struct VarlenSet {
    VerifyKernel pipe[2][kMaxStaticT + 1];
};

const VarlenSet &varlen_bf16_w2();
const VarlenSet &varlen_bf16_w3();
const VarlenSet &varlen_bf16_w4();
const VarlenSet &varlen_f32_w2();
const VarlenSet &varlen_f32_w3();
const VarlenSet &varlen_f32_w4();

const KernelSet &kernels_bf16_w2();
const KernelSet &kernels_bf16_w3();
const KernelSet &kernels_bf16_w4();
const KernelSet &kernels_f32_w2();
const KernelSet &kernels_f32_w3();
const KernelSet &kernels_f32_w4();

}  // namespace cvk
