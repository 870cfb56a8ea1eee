// mask_occupancy.cu -- pre-pass of dit_attn_fwd_masked: which key tiles of
// each 256-row query block does the general mask leave anything in?
//
// One bit per (b, 256-row block, 128-key tile): set when some row of the
// block may attend some key of the tile.  Rows i >= mask_rows attend every
// valid key ("8 卡怎么分 token", "构造 padding mask": pad query rows see all
// valid keys), so their blocks are fully occupied.  The attention kernel then
// loads and multiplies only occupied tiles; for block-local masks most tiles
// are empty.  Reads the mask once (HBM-bound): one warp per (b, block, 32
// tiles), lane = tile, each lane reading its tile's four words of every row
// (a warp's loads cover 512 consecutive bytes of a mask row).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dit {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 256;   // query rows per attention CTA
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) mask_occupancy_kernel(const OccArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int64_t units = static_cast<int64_t>(a.B) * a.row_blocks * a.occ_words;
    if (unit >= units) return;
    const int g = static_cast<int>(unit % a.occ_words);
    const int64_t rest = unit / a.occ_words;
    const int rb = static_cast<int>(rest % a.row_blocks);
    const int b = static_cast<int>(rest / a.row_blocks);
    const int t = g * 32 + lane;                     // this lane's key tile
    const int r0 = rb * kRowsPerBlock;
    const int r1 = min(r0 + kRowsPerBlock, a.Nq);
    bool occupied = false;
    if (t < a.n_kv_tiles) {
        if (r1 > a.mask_rows) {
            occupied = true;                         // a pad-rule row attends every valid key
        } else {
            const uint4* base = reinterpret_cast<const uint4*>(a.mask + static_cast<int64_t>(b) * a.mask_sb) + t;
            const int64_t row_step = a.mask_si / 4;  // uint4 per row
            for (int r = r0; r < r1 && !occupied; r += kUnroll) {
                uint4 w[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    w[u] = (r + u < r1) ? __ldcs(base + static_cast<int64_t>(r + u) * row_step) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) occupied |= (w[u].x | w[u].y | w[u].z | w[u].w) != 0u;
            }
        }
    }
    const uint32_t word = __ballot_sync(0xffffffffu, occupied);
    if (lane == 0) a.occ[(static_cast<int64_t>(b) * a.row_blocks + rb) * a.occ_words + g] = word;
}

}  // namespace

cudaError_t launch_mask_occupancy(const OccArgs& a, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(a.B) * a.row_blocks * a.occ_words;
    const int64_t blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
    if (blocks <= 0) return cudaSuccess;
    mask_occupancy_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace dit
