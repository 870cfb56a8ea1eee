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
// Pure data movement, HBM-bound.  One warp copies one run of 32 consecutive
// sequence rows of one (b, t, h) plane: its stores form a single contiguous
// 32 * D * 2-byte range of the destination, its loads 32 strided 2*D-byte
// segments of the source; every lane keeps kUnroll 16-byte loads in flight
// before it stores.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dit {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kRunRows = 32;   // sequence rows per warp unit
constexpr int kUnroll = 8;     // 16-byte vectors in flight per lane

__global__ void __launch_bounds__(kLayoutThreads) qkv_layout_kernel(const LayoutArgs a) {
    const int vec_per_d = a.D / 8;                 // 16-byte vectors per head row
    const int64_t n_runs = (a.N + kRunRows - 1) / kRunRows;
    const int planes = 3 * a.H;
    const int64_t units = static_cast<int64_t>(a.B) * planes * n_runs;
    const int lane = threadIdx.x & 31;
    const int warps_per_block = kLayoutThreads / 32;
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
    const int64_t ws = static_cast<int64_t>(gridDim.x) * warps_per_block;
    const int total = kRunRows * vec_per_d;        // vectors in one run
    for (int64_t u = w0; u < units; u += ws) {
        const int64_t run = u % n_runs;
        const int64_t rest = u / n_runs;
        const int p = static_cast<int>(rest % planes);   // p = t*H + h
        const int64_t b = rest / planes;
        const int t = p / a.H;
        const int hh = p - t * a.H;
        const int n0 = static_cast<int>(run * kRunRows);
        const uint16_t* src = a.qkv + b * a.stride_b + static_cast<int64_t>(p) * a.D;
        uint16_t* plane = t == 0 ? a.out[0] : (t == 1 ? a.out[1] : a.out[2]);
        uint16_t* dst = plane + (b * a.H + hh) * static_cast<int64_t>(a.N) * a.D;
        for (int base = lane; base < total; base += 32 * kUnroll) {
            uint4 v[kUnroll];
            int n[kUnroll], c[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int it = base + k * 32;
                n[k] = n0 + it / vec_per_d;
                c[k] = it - (it / vec_per_d) * vec_per_d;
                if (it < total && n[k] < a.N)
                    v[k] = __ldcs(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(n[k]) * a.stride_n + c[k] * 8));
                else
                    n[k] = -1;
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k)
                if (n[k] >= 0)
                    __stcs(reinterpret_cast<uint4*>(dst + static_cast<int64_t>(n[k]) * a.D + c[k] * 8), v[k]);
        }
    }
}

}  // namespace

cudaError_t launch_qkv_to_head_major(const LayoutArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>(a.B) * 3 * a.H * ((a.N + kRunRows - 1) / kRunRows);
    int64_t blocks = static_cast<int64_t>(device_sm_count(dev)) * 8;
    const int64_t need = (units + kLayoutThreads / 32 - 1) / (kLayoutThreads / 32);
    if (blocks > need) blocks = need;
    if (blocks < 1) blocks = 1;
    qkv_layout_kernel<<<static_cast<unsigned>(blocks), kLayoutThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dit
