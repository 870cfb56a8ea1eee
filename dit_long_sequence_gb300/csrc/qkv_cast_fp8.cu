// qkv_cast_fp8.cu -- one pass over a stacked [B, N, 3, H, D] bf16 QKV buffer
// that writes it as E4M3 in the same stacked layout, each of q, k, v scaled by
// its own per-tensor factor first: "Scaling Video Generation Across NVL72 rack
// with TensorRT-LLM", "Ulysses Parallelism", paragraph "Fused vs. unfused QKV
// all-to-all" (a single FP8 cast over the contiguous stacked buffer instead of
// three casts, whose result goes to the attention kernel without a copy).
//
// HBM-bound: 2 bytes read and 1 byte written per element.  Each thread moves
// 16 elements per chunk (two 16-byte loads, one 16-byte store) and keeps four
// chunks in flight; chunks never straddle q/k/v because H*D is a multiple of
// 16.  Grid: a multiple of the SM count, grid-stride over the chunks.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 cast16(const uint4& a, const uint4& b, float s) {
    uint4 r;
    r.x = pack_e4m3x4(bf16_lo(a.x) * s, bf16_hi(a.x) * s, bf16_lo(a.y) * s, bf16_hi(a.y) * s);
    r.y = pack_e4m3x4(bf16_lo(a.z) * s, bf16_hi(a.z) * s, bf16_lo(a.w) * s, bf16_hi(a.w) * s);
    r.z = pack_e4m3x4(bf16_lo(b.x) * s, bf16_hi(b.x) * s, bf16_lo(b.y) * s, bf16_hi(b.y) * s);
    r.w = pack_e4m3x4(bf16_lo(b.z) * s, bf16_hi(b.z) * s, bf16_lo(b.w) * s, bf16_hi(b.w) * s);
    return r;
}

__global__ void __launch_bounds__(kThreads) qkv_cast_fp8_kernel(const CastArgs a) {
    const uint32_t C = a.chunks_per_row;     // 3*H*D / 16
    const uint32_t hd = a.hd;                // H*D
    const uint64_t total = a.total_chunks;   // B*N*C < 2^32
    const uint64_t step = static_cast<uint64_t>(gridDim.x) * kThreads;
    for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; base < total;
         base += step * kUnroll) {
        uint4 va[kUnroll], vb[kUnroll];
        float sc[kUnroll];
        uint8_t* dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t g = base + u * step;
            dst[u] = nullptr;
            if (g < total) {
                const uint32_t gi = static_cast<uint32_t>(g);
                const uint32_t row = gi / C;
                const uint32_t w = gi - row * C;
                const uint32_t b = row / static_cast<uint32_t>(a.N);
                const uint32_t n = row - b * static_cast<uint32_t>(a.N);
                const uint32_t off = w * 16;
                const uint16_t* src = a.qkv + b * a.stride_b + n * a.stride_n + off;
                va[u] = __ldcs(reinterpret_cast<const uint4*>(src));
                vb[u] = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
                sc[u] = off >= 2 * hd ? a.scale[2] : (off >= hd ? a.scale[1] : a.scale[0]);
                dst[u] = a.out + static_cast<uint64_t>(row) * (16ull * C) + off;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dst[u] != nullptr) __stcs(reinterpret_cast<uint4*>(dst[u]), cast16(va[u], vb[u], sc[u]));
    }
}

}  // namespace

cudaError_t launch_qkv_cast_fp8(const CastArgs& args, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t per_block = static_cast<uint64_t>(kThreads) * kUnroll;
    const uint64_t need = (args.total_chunks + per_block - 1) / per_block;
    const uint64_t cap = static_cast<uint64_t>(device_sm_count(dev)) * 8;
    const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
    qkv_cast_fp8_kernel<<<grid, kThreads, 0, stream>>>(args);
    return cudaGetLastError();
}

}  // namespace dit
