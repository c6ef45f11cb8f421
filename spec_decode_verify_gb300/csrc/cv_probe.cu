// Bandwidth probe for the roofline of the verify: how fast HBM moves a given mix of reads and
// writes.  The verify kernel reads about 1 byte for every 1.9 it writes (x and the committed
// windows in; outputs, snapshot rows and the committed windows out), and a plain copy measures the
// 1:1 mix only, so this probe times streams of other ratios with the access shape the verify uses:
// 16-byte vector loads and stores, each warp covering contiguous runs, a grid sized to the SM
// count.  It is measurement infrastructure, built into its own library (libcvprobe.so) and used
// only by bench.py --probe-mix; the verify library does not contain it.
//
// cv_probe_mix(src, dst, n_units, r, w, blocks, threads, sink, stream): src holds r streams and dst
// w streams of n_units 16-byte vectors each; unit i reads vector i of every src stream
// (src[j*n_units + i]) and writes vector i of every dst stream, each a mix of the vectors read (so
// no load is dead).  With r = 0 the unit writes a value made from its index; with
// w = 0 the values read are folded into one vector per thread, written to sink[thread] at the end.
// Units are spread over the grid by a grid-stride loop.  (r, w) must be one of the compiled mixes:
// (1,0) (0,1) (1,1) (2,1) (1,2) (1,3) (2,3) (10,19).  Returns 0, or a CUDA error code.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

template <int R, int W>
__global__ void __launch_bounds__(256, 1) probe_mix(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                 long long n_units, uint4 *__restrict__ sink) {
    uint4 fold = make_uint4(0u, 0u, 0u, 0u);
    const long long stride = (long long)gridDim.x * blockDim.x;
    // consecutive threads take consecutive units, so every warp access is one contiguous 512-byte run
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_units; i += stride) {
        uint4 v[R > 0 ? R : 1];
        uint4 acc = make_uint4((unsigned)i, (unsigned)(i >> 32), 0x9e3779b9u, 0u);
#pragma unroll
        for (int j = 0; j < R; ++j) v[j] = src[j * n_units + i];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            acc.x ^= v[j].x;
            acc.y ^= v[j].y;
            acc.z ^= v[j].z;
            acc.w ^= v[j].w;
        }
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const uint4 a = R > 0 ? v[j % (R > 0 ? R : 1)] : acc;
            dst[j * n_units + i] = make_uint4(a.x ^ acc.y, a.y ^ acc.z, a.z ^ acc.w, a.w ^ (unsigned)j);
        }
        fold.x ^= acc.x;
        fold.y ^= acc.y;
        fold.z ^= acc.z;
        fold.w ^= acc.w;
    }
    if (W == 0) sink[(long long)blockIdx.x * blockDim.x + threadIdx.x] = fold;
}

template <int R, int W>
int launch(const void *src, void *dst, long long n_units, int blocks, int threads, void *sink, cudaStream_t st) {
    probe_mix<R, W><<<blocks, threads, 0, st>>>(reinterpret_cast<const uint4 *>(src), reinterpret_cast<uint4 *>(dst),
                                                n_units, reinterpret_cast<uint4 *>(sink));
    return (int)cudaGetLastError();
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int cv_probe_mix(const void *src, void *dst, long long n_units,
                                                                   int r, int w, int blocks, int threads,
                                                                   void *sink, void *stream) {
    if (blocks < 1 || threads < 32 || threads > 256 || n_units < 0) return (int)cudaErrorInvalidValue;
    if ((r > 0 && !src) || (w > 0 && !dst) || (w == 0 && !sink)) return (int)cudaErrorInvalidValue;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int key = r * 100 + w;
    switch (key) {
        case 100: return launch<1, 0>(src, dst, n_units, blocks, threads, sink, st);
        case 1: return launch<0, 1>(src, dst, n_units, blocks, threads, sink, st);
        case 101: return launch<1, 1>(src, dst, n_units, blocks, threads, sink, st);
        case 201: return launch<2, 1>(src, dst, n_units, blocks, threads, sink, st);
        case 102: return launch<1, 2>(src, dst, n_units, blocks, threads, sink, st);
        case 103: return launch<1, 3>(src, dst, n_units, blocks, threads, sink, st);
        case 203: return launch<2, 3>(src, dst, n_units, blocks, threads, sink, st);
        case 1019: return launch<10, 19>(src, dst, n_units, blocks, threads, sink, st);
        default: return (int)cudaErrorInvalidValue;
    }
}
