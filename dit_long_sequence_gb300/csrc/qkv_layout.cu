// qkv_layout.cu -- bit-exact split of a fused [B, N, 3, H, D] QKV projection
// into three head-major [B, H, N, D] tensors.
//
// "Scaling Video Generation Across NVL72 rack with TensorRT-LLM", "Ulysses
// Parallelism": attention wants the head-sharded layout, and the stacked
// buffer is [B, S, 3, H, D] ("Fused vs. unfused QKV all-to-all").  "CUDA IPC
// Ulysses：在 H100 上重叠 Attention 通信", "Strided Copy Engine scatter": the
// source pitch is taken from the input stride, head and channel contiguous
// within each sequence row.  Here the scatter target is this GPU's own HBM.
//
// Pure data movement, HBM-bound.  A CTA copies kRows consecutive sequence rows
// of one batch entry: 16-byte loads walk each fused row contiguously, and for
// every (t, h) plane the kRows destination rows form one contiguous run of
// kRows * D * 2 bytes.  All loads of a thread are issued before its stores.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dit {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kRows = 4;     // sequence rows per CTA step
constexpr int kUnroll = 4;   // 16-byte vectors in flight per thread

__global__ void __launch_bounds__(kLayoutThreads) qkv_layout_kernel(const LayoutArgs a) {
    const int vec_per_d = a.D / 8;                    // 16-byte vectors per head row
    const int vec_per_row = 3 * a.H * vec_per_d;      // per fused sequence row
    const int64_t groups_per_b = (a.N + kRows - 1) / kRows;
    const int64_t n_groups = groups_per_b * a.B;
    const int items = kRows * vec_per_row;            // vectors per CTA step

    for (int64_t g = blockIdx.x; g < n_groups; g += gridDim.x) {
        const int64_t b = g / groups_per_b;
        const int n0 = static_cast<int>(g - b * groups_per_b) * kRows;
        const uint16_t* src_b = a.qkv + b * a.stride_b;
        for (int base = threadIdx.x; base < items; base += kLayoutThreads * kUnroll) {
            uint4 v[kUnroll];
            const uint16_t* dst[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int it = base + u * kLayoutThreads;
                dst[u] = nullptr;
                if (it < items) {
                    // item -> (plane p = t*H + h, row r, vector c); plane-major so
                    // that consecutive threads write one contiguous run per plane.
                    const int per_plane = kRows * vec_per_d;
                    const int p = it / per_plane;
                    const int rem = it - p * per_plane;
                    const int r = rem / vec_per_d;
                    const int c = rem - r * vec_per_d;
                    const int n = n0 + r;
                    if (n < a.N) {
                        const int t = p / a.H;
                        const int hh = p - t * a.H;
                        const uint16_t* src = src_b + static_cast<int64_t>(n) * a.stride_n +
                                              static_cast<int64_t>(p) * a.D + c * 8;
                        v[u] = __ldcs(reinterpret_cast<const uint4*>(src));
                        dst[u] = a.out[t] + ((b * a.H + hh) * static_cast<int64_t>(a.N) + n) * a.D + c * 8;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (dst[u] != nullptr) __stcs(reinterpret_cast<uint4*>(const_cast<uint16_t*>(dst[u])), v[u]);
        }
    }
}

}  // namespace

cudaError_t launch_qkv_to_head_major(const LayoutArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t n_groups = static_cast<int64_t>((a.N + kRows - 1) / kRows) * a.B;
    int64_t blocks = static_cast<int64_t>(device_sm_count(dev)) * 8;
    if (blocks > n_groups) blocks = n_groups;
    if (blocks < 1) blocks = 1;
    qkv_layout_kernel<<<static_cast<unsigned>(blocks), kLayoutThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dit
