// qkv_norm_rope.cu -- the QKV split of qkv_layout.cu with the per-head Q/K
// RMSNorm and rotary embedding fused in: one pass over the fused
// [B, N, 3, H, D] projection writes head-major q', k', v [B, H, N, D].
//
// "CUDA IPC Ulysses：在 H100 上重叠 Attention 通信", "基线与瓶颈" (and the
// "模型调度" schedule): Q and K are normalised and rotated before attention, V
// is not.  The pages give neither formula; the reading implemented (and the
// oracle's) is RMSNorm over the head dimension with an optional per-channel
// weight, y = x / sqrt(mean(x^2) + eps) * w, then the RoFormer rotation of
// consecutive channel pairs (2i, 2i+1) by caller-tabulated angles
// (cos/sin [N, D/2] fp32, so 1-D and 3-D video positions are the same call).
//
// HBM-bound: 2 bytes read and 2 written per element (the fp32 tables, N*D*4
// bytes, are read once per sequence row).  A row of D channels is held by D/8
// lanes, 8 channels (one 16-byte vector) each; the mean square is reduced
// across those lanes with shuffles, and every rotary pair lies inside one
// lane.  One warp owns 32/(D/8) consecutive sequence rows and walks all 3*H
// planes of them (contiguous source reads), so a row's cos/sin are loaded once
// and reused by every q and k head.  The loads are software pipelined: the
// next kUnroll planes are requested before the current ones are processed, so
// loads stay in flight through the arithmetic and the stores (+2.5% on the
// LTX-2 shape over loading each group when it is needed).  Latency hiding
// comes from resident warps rather than deep unrolling: four 256-thread
// blocks per SM with 4 planes in flight measured 5.56 TB/s on the LTX-2
// shape, against 4.75 TB/s for one block with 8 and 3.47 TB/s with 16.
// Computed in fp32, rounded to bf16 once.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dit {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 4) qkv_norm_rope_kernel(const NormRopeArgs a) {
    constexpr int LPR = D / 8;          // lanes per row
    constexpr int RPW = 32 / LPR;       // sequence rows per warp unit
    constexpr int kUnroll = 4;          // planes in flight per lane
    const int lane = threadIdx.x & 31;
    const int c = lane % LPR;           // this lane's 8-channel vector
    const int rsub = lane / LPR;        // row within the unit
    const int planes = 3 * a.H;
    const int64_t n_units = (a.N + RPW - 1) / RPW;
    const int64_t units = static_cast<int64_t>(a.B) * n_units;
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t ws = static_cast<int64_t>(gridDim.x) * (kThreads / 32);

    const bool norm_q = a.weight[0] != nullptr, norm_k = a.weight[1] != nullptr;
    const bool rope = a.cos != nullptr;
    const float inv_d = 1.f / D;

    for (int64_t u = w0; u < units; u += ws) {
        const int64_t b = u / n_units;
        const int n = static_cast<int>((u - b * n_units) * RPW) + rsub;
        const bool live = n < a.N;
        // this row's rotation, shared by every q and k head
        float cr[4] = {1.f, 1.f, 1.f, 1.f}, sr[4] = {0.f, 0.f, 0.f, 0.f};
        if (rope && live) {
            const float4 cs = __ldg(reinterpret_cast<const float4*>(a.cos + static_cast<int64_t>(n) * (D / 2) + 4 * c));
            const float4 sn = __ldg(reinterpret_cast<const float4*>(a.sin + static_cast<int64_t>(n) * (D / 2) + 4 * c));
            cr[0] = cs.x; cr[1] = cs.y; cr[2] = cs.z; cr[3] = cs.w;
            sr[0] = sn.x; sr[1] = sn.y; sr[2] = sn.z; sr[3] = sn.w;
        }
        const uint16_t* src = a.qkv + b * a.stride_b + static_cast<int64_t>(live ? n : 0) * a.stride_n + 8 * c;
        const int64_t dst_off = (b * a.H * static_cast<int64_t>(a.N) + n) * D + 8 * c;   // + h * N * D
        // software pipelined: the next group's loads are issued before this
        // group is processed, so kUnroll loads stay in flight throughout
        uint4 nxt[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
            nxt[k] = (live && k < planes) ? __ldcs(reinterpret_cast<const uint4*>(src + k * D))
                                          : make_uint4(0u, 0u, 0u, 0u);
        for (int p0 = 0; p0 < planes; p0 += kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) v[k] = nxt[k];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k)
                nxt[k] = (live && p0 + kUnroll + k < planes)
                             ? __ldcs(reinterpret_cast<const uint4*>(src + (p0 + kUnroll + k) * D))
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int p = p0 + k;
                if (p >= planes) break;                 // uniform across the warp
                const int t = p / a.H;                  // 0 q, 1 k, 2 v
                const bool norm = t == 0 ? norm_q : (t == 1 ? norm_k : false);
                if (t < 2 && (norm || rope)) {
                    float x[8] = {lo_f(v[k].x), hi_f(v[k].x), lo_f(v[k].y), hi_f(v[k].y),
                                  lo_f(v[k].z), hi_f(v[k].z), lo_f(v[k].w), hi_f(v[k].w)};
                    if (norm) {
                        float ss = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
                        for (int off = LPR / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                        const float r = rsqrtf(fmaf(ss, inv_d, a.eps));
                        // this lane's 8 weights (L1-resident after the first row)
                        const float4* wp = reinterpret_cast<const float4*>((t == 0 ? a.weight[0] : a.weight[1]) + 8 * c);
                        const float4 w0 = __ldg(wp), w1 = __ldg(wp + 1);
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) x[i] = x[i] * r * wv[i];
                    }
                    if (rope) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float y0 = x[2 * i], y1 = x[2 * i + 1];
                            x[2 * i] = y0 * cr[i] - y1 * sr[i];
                            x[2 * i + 1] = y0 * sr[i] + y1 * cr[i];
                        }
                    }
                    v[k] = make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
                }
                if (live) {
                    const int hh = p - t * a.H;
                    uint16_t* plane = t == 0 ? a.out[0] : (t == 1 ? a.out[1] : a.out[2]);
                    __stcs(reinterpret_cast<uint4*>(plane + dst_off + static_cast<int64_t>(hh) * a.N * D), v[k]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_qkv_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int rpw = 32 / (a.D / 8);
    const int64_t units = static_cast<int64_t>(a.B) * ((a.N + rpw - 1) / rpw);
    int64_t blocks = static_cast<int64_t>(device_sm_count(dev)) * 8;
    const int64_t need = (units + kThreads / 32 - 1) / (kThreads / 32);
    if (blocks > need) blocks = need;
    if (blocks < 1) blocks = 1;
    if (a.D == 128)
        qkv_norm_rope_kernel<128><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
    else
        qkv_norm_rope_kernel<64><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dit
