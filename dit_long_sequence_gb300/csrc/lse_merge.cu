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
// HBM-bound.  One warp owns one sequence position (b, i).  Phase 1: lane h computes the normalised chunk
// weights of head h (LSE reads once per row, not once per lane) into shared
// memory.  Phase 2: the warp streams the H rows, D/4 lanes per row, with
// 128-bit streaming loads of every chunk issued before they are used.  With
// the chunks interleaved per row (o_row_stride = n*D) those loads are one
// contiguous n*D*4-byte run per row; chunk-major partials are n separate streams,
// which DRAM serves markedly slower.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kMergeWarps = 4;
constexpr int kMergeThreads = 32 * kMergeWarps;
constexpr int kMaxChunks = 64;
constexpr int kGroup = 16;  // chunk loads in flight per lane and row

// Blocks for need_blocks block-rounds of grid-stride work: no more than fit on
// the GPU at once (per_sm resident blocks per SM), spread so that every block
// runs the same number of rounds, give or take one.  The merge's per-position
// work is coarse, so a grid of several waves (or a partly empty last round)
// shows in its tail; the pure streaming kernels (layout, cast, norm + RoPE)
// measured faster with oversubscribed grids.
inline int64_t balanced_blocks(int64_t need_blocks, int per_sm, int sms) {
    if (need_blocks < 1) return 1;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    const int64_t rounds = (need_blocks + cap - 1) / cap;
    return (need_blocks + rounds - 1) / rounds;
}

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(const MergeArgs a, int64_t n_pos) {
    constexpr int LPR = D / 4;    // lanes per row
    constexpr int RPW = 32 / LPR; // rows per warp step
    // weights of 32 heads x up to kMaxChunks chunks, per warp (0 = chunk skipped)
    __shared__ float w_s[kMergeWarps][32][kMaxChunks];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int col = (lane % LPR) * 4;
    const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
    const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * kMergeWarps;
    const int n = a.n_chunks;
    const int H = a.H;
    float (*w)[kMaxChunks] = w_s[warp];

    for (int64_t p = warp_global; p < n_pos; p += warp_stride) {
        const int64_t bb = p / a.Nq;
        const int64_t i = p - bb * a.Nq;
        for (int h0 = 0; h0 < H; h0 += 32) {
            // ---- phase 1: lane = head h0 + lane
            const int hl = h0 + lane;
            if (hl < H) {
                const float* lp = a.lse_parts + (bb * H + hl) * a.Nq + i;
                float M = -INFINITY;
                for (int k = 0; k < n; ++k) M = fmaxf(M, __ldg(lp + k * a.lse_chunk_stride));
                float lam = 0.f;
                if (M != -INFINITY) {
                    for (int k = 0; k < n; ++k) {
                        const float e = expf(__ldg(lp + k * a.lse_chunk_stride) - M);
                        w[lane][k] = e;
                        lam += e;
                    }
                    const float inv = 1.f / lam;
                    for (int k = 0; k < n; ++k) w[lane][k] *= inv;
                } else {
                    for (int k = 0; k < n; ++k) w[lane][k] = 0.f;
                }
                if (a.lse_out != nullptr)
                    a.lse_out[(bb * H + hl) * a.Nq + i] = (M == -INFINITY) ? -INFINITY : M + logf(lam);
            }
            __syncwarp();
            // ---- phase 2: stream rows (p, h0 .. h0+31), RPW rows per step
            const int hn = min(32, H - h0);
            for (int hh = sub; hh < hn; hh += RPW) {
                const int64_t r = p * H + h0 + hh;
                const float* orow = a.o_parts + r * a.o_row_stride + col;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int k0 = 0; k0 < n; k0 += kGroup) {
                    float wk[kGroup];
                    float4 v[kGroup];
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        const int k = k0 + g;
                        wk[g] = (k < n) ? w[hh][k] : 0.f;
                        v[g] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (wk[g] > 0.f) v[g] = __ldcs(reinterpret_cast<const float4*>(orow + k * a.o_chunk_stride));
                    }
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        acc.x = fmaf(wk[g], v[g].x, acc.x);
                        acc.y = fmaf(wk[g], v[g].y, acc.y);
                        acc.z = fmaf(wk[g], v[g].z, acc.z);
                        acc.w = fmaf(wk[g], v[g].w, acc.w);
                    }
                }
                if constexpr (OUT_BF16) {
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x, acc.y);
                    pk.y = pack_bf16x2(acc.z, acc.w);
                    __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + r * D + col), pk);
                } else {
                    __stcs(reinterpret_cast<float4*>(static_cast<float*>(a.out) + r * D + col), acc);
                }
            }
            __syncwarp();
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
    // Positions are dealt to warps round-robin: resident blocks only, every
    // warp the same count of positions (give or take one).
    auto kern = lse_merge_kernel<D, BF16>;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMergeThreads, 0);
    if (e != cudaSuccess) return e;
    const int64_t blocks = balanced_blocks((n_pos + kMergeWarps - 1) / kMergeWarps, per_sm, sms);
    kern<<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a, n_pos);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, int D, bool out_bf16, cudaStream_t stream) {
    if (a.n_chunks > kMaxChunks) return cudaErrorInvalidValue;
    if (D == 128) return out_bf16 ? merge_impl<128, true>(a, stream) : merge_impl<128, false>(a, stream);
    return out_bf16 ? merge_impl<64, true>(a, stream) : merge_impl<64, false>(a, stream);
}

}  // namespace dit
