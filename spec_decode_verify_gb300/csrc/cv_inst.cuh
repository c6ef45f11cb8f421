// Builds the kernel table of one (element type, conv width); included once per instantiation unit
// with CV_INST_B, CV_INST_W, CV_INST_MAXT and CV_INST_NAME defined, and CV_INST_VARLEN defined for
// the units that hold the packed-ragged-draft variants of the pipelined kernel (VarlenSet).
#include <utility>

#ifdef CV_INST_VARLEN
#include "cv_launch.h"
#include "cv_verify_pipe.cuh"

namespace cvk {
namespace {
template <typename B, int W, int... Ts>
VarlenSet make_varlen(std::integer_sequence<int, Ts...>) {
    VarlenSet k{};
    ((k.pipe[0][Ts + 1] = verify_pipe<B, W, Ts + 1, 4, B, true>), ...);
    ((k.pipe[1][Ts + 1] = verify_pipe<B, W, Ts + 1, 8, B, true>), ...);
    return k;
}
}  // namespace

const VarlenSet &CV_INST_NAME() {
    static const VarlenSet k = make_varlen<CV_INST_B, CV_INST_W>(std::make_integer_sequence<int, CV_INST_MAXT>{});
    return k;
}
}  // namespace cvk
#else

#include "cv_commit.cuh"
#include "cv_launch.h"
#include "cv_prefill.cuh"
#include "cv_verify_fast.cuh"
#include "cv_verify_generic.cuh"
#include "cv_verify_pipe.cuh"
#include "cv_verify_tree.cuh"

namespace cvk {
namespace {
// the other dtype of the state and the snapshots (mixed dtypes)
template <typename B>
using OtherT = std::conditional_t<sizeof(B) == 2, uint32_t, uint16_t>;

template <typename B, int W, int... Ms>
void set_mixed(KernelSet &k, std::integer_sequence<int, Ms...>) {
    ((k.pipe_mixed[0][Ms + 1] = verify_pipe<B, W, Ms + 1, 4, OtherT<B>>), ...);
    ((k.pipe_mixed[1][Ms + 1] = verify_pipe<B, W, Ms + 1, 8, OtherT<B>>), ...);
}

template <typename B, int W, int... Ts>
KernelSet make_set(std::integer_sequence<int, Ts...>) {
    KernelSet k{};
    set_mixed<B, W>(k, std::make_integer_sequence<int, (sizeof...(Ts) < kMaxMixedT ? sizeof...(Ts) : kMaxMixedT)>{});
    k.fast[0][0] = verify_fast<B, W, 0, 4>;
    k.fast[1][0] = verify_fast<B, W, 0, 8>;
    ((k.fast[0][Ts + 1] = verify_fast<B, W, Ts + 1, 4>), ...);
    ((k.fast[1][Ts + 1] = verify_fast<B, W, Ts + 1, 8>), ...);
    ((k.pipe[0][Ts + 1] = verify_pipe<B, W, Ts + 1, 4>), ...);
    ((k.pipe[1][Ts + 1] = verify_pipe<B, W, Ts + 1, 8>), ...);
    k.max_static_t = (int)sizeof...(Ts);
    k.generic = verify_generic<B, W>;
    k.tree = verify_tree<B, W>;
    // mixed dtypes: the state and the snapshots in the other dtype
    k.generic_mixed = verify_generic<B, W, OtherT<B>>;
    k.commit = commit_kernel<B, W, false>;
    k.commit_packed = commit_kernel<B, W, true>;
    k.commit_wide = commit_wide<B, W>;
    k.commit_rows = commit_rows<B, W>;
    k.commit_cols = commit_cols<B, W>;
    k.commit_recompute = commit_recompute<B, W>;
    k.commit_recompute_vec = commit_recompute_vec<B, W>;
    k.prefill[0] = prefill_conv<B, W, 4>;
    k.prefill[1] = prefill_conv<B, W, 8>;
    return k;
}
}  // namespace

const KernelSet &CV_INST_NAME() {
    static const KernelSet k = make_set<CV_INST_B, CV_INST_W>(std::make_integer_sequence<int, CV_INST_MAXT>{});
    return k;
}
}  // namespace cvk
#endif  // CV_INST_VARLEN
