// lse_merge.cu -- exact combine of (O, LSE) partial attention passes.
//
// "Scaling Video Generation Across NVL72 rack with TensorRT-LLM",
// "Attention2D Parallelism" / "Merge phase": the partials for the same query
// rows over complementary key spans are merged in one batched kernel; "Ring
// Attention" / "Online-softmax merge": the merge runs in fp32 and reproduces
// one global pass.  Per row (b, i, h):
//     M = max_k L_k,  w_k = exp(L_k - M),  O = sum_k w_k O_k / sum_k w_k,
//     LSE = M + ln sum_k w_k;
// chunks with L_k = -inf have weight 0 and are not read; an all -inf row gives
// O = 0 and LSE = -inf.
//
// HBM-bound: each row of D fp32 is read once per chunk with 128-bit streaming
// loads and written once.  D/4 lanes own a row (a full warp for D = 128,
// a half warp for D = 64); all chunk loads of a lane are issued before use.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMaxChunks = 64;
constexpr int kGroup = 8;  // chunk loads in flight per lane

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const MergeArgs a, int64_t n_pos) {
    constexpr int LPR = D / 4;            // lanes per row
    constexpr int RPW = 32 / LPR;         // rows (heads) per warp step
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;           // head slot within the warp step
    const int col = (lane % LPR) * 4;     // first channel of this lane
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
    const int64_t warp_stride = (static_cast<int64_t>(gridDim.x) * kMergeThreads) >> 5;
    const int n = a.n_chunks;
    const int H = a.H;

    // One warp per sequence position p = b*Nq + i; its H rows are contiguous.
    for (int64_t p = warp_global; p < n_pos; p += warp_stride) {
        const int64_t bb = p / a.Nq;
        const int64_t i = p - bb * a.Nq;
        for (int h0 = 0; h0 < H; h0 += RPW) {
            const int hh = h0 + sub;
            const bool live = hh < H;
            const int64_t r = p * H + (live ? hh : 0);
            const int64_t lse_idx = (bb * H + (live ? hh : 0)) * a.Nq + i;

            float M = -INFINITY;
            for (int k = 0; k < n; ++k) M = fmaxf(M, __ldg(a.lse_parts + k * a.lse_chunk_stride + lse_idx));

            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float lam = 0.f;
            if (M != -INFINITY) {
                const float* orow = a.o_parts + r * D + col;
                for (int k0 = 0; k0 < n; k0 += kGroup) {
                    float w[kGroup];
                    float4 v[kGroup];
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        const int k = k0 + g;
                        w[g] = 0.f;
                        v[g] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (k < n) {
                            const float L = __ldg(a.lse_parts + k * a.lse_chunk_stride + lse_idx);
                            w[g] = expf(L - M);
                            if (w[g] > 0.f && live)
                                v[g] = __ldcs(reinterpret_cast<const float4*>(orow + k * a.o_chunk_stride));
                        }
                    }
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        lam += w[g];
                        acc.x = fmaf(w[g], v[g].x, acc.x);
                        acc.y = fmaf(w[g], v[g].y, acc.y);
                        acc.z = fmaf(w[g], v[g].z, acc.z);
                        acc.w = fmaf(w[g], v[g].w, acc.w);
                    }
                }
                const float inv = 1.f / lam;
                acc.x *= inv;
                acc.y *= inv;
                acc.z *= inv;
                acc.w *= inv;
            }
            if (live) {
                if constexpr (OUT_BF16) {
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x, acc.y);
                    pk.y = pack_bf16x2(acc.z, acc.w);
                    __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + r * D + col), pk);
                } else {
                    __stcs(reinterpret_cast<float4*>(static_cast<float*>(a.out) + r * D + col), acc);
                }
                if (a.lse_out != nullptr && (lane % LPR) == 0)
                    a.lse_out[lse_idx] = (M == -INFINITY) ? -INFINITY : M + logf(lam);
            }
        }
    }
}

template <int D, bool BF16>
cudaError_t merge_impl(const MergeArgs& a, cudaStream_t stream) {
    const int64_t n_pos = static_cast<int64_t>(a.B) * a.Nq;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count(dev);
    const int64_t pos_per_block = kMergeThreads / 32;
    int64_t blocks = (n_pos + pos_per_block - 1) / pos_per_block;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    lse_merge_kernel<D, BF16><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a, n_pos);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, int D, bool out_bf16, cudaStream_t stream) {
    static_assert(kMaxChunks >= kGroup, "group");
    if (D == 128) return out_bf16 ? merge_impl<128, true>(a, stream) : merge_impl<128, false>(a, stream);
    return out_bf16 ? merge_impl<64, true>(a, stream) : merge_impl<64, false>(a, stream);
}

}  // namespace dit
