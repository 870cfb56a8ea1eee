// internal.h -- launch-side declarations shared by the kernel translation
// units and the C-ABI layer (api.cu).  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dit {

// Warp roles and wait sites reported by the watchdog (status words 2 and 3).
enum WatchRole : uint32_t { ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3 };
enum WatchSite : uint32_t {
    SITE_Q_FULL = 1, SITE_KV_FULL = 2, SITE_KV_EMPTY = 3, SITE_S_FULL = 4, SITE_P_FULL = 5,
    SITE_O_FINAL = 6, SITE_DRAIN = 7, SITE_LOAD_DRAIN = 8
};
// Sites of the debug library's bounds checks (status word 3 with code 6).
enum BoundSite : uint32_t {
    BND_ITEM = 101,   // work item decoded outside (B, H, Nq)
    BND_KEY = 102,    // key tile outside [0, kv_len)
    BND_SMEM = 103,   // shared-memory operand or staging address outside its buffer
    BND_TMEM = 104,   // tensor-memory column outside the 512 allocated
    BND_OUT = 105,    // O element outside the extent its strides reach
    BND_LSE = 106,    // LSE element outside [B, H, Nq]
    BND_WS = 107,     // workspace element outside the split pieces' partials
    BND_MASK = 108,   // mask word outside the extent its strides reach
};
// Faults the debug library can inject (one withheld producer signal).
enum DebugFault : uint32_t {
    FAULT_NONE = 0,
    FAULT_SKIP_LOAD = 1,       // the TMA thread skips K/V load `index` (no arrive, no copy)
    FAULT_SKIP_S_COMMIT = 2,   // the MMA thread skips the completion signal of S_0 number `index`
    FAULT_SKIP_P_ARRIVE = 3,   // softmax warp 0 skips its P-ready arrive at key tile `index`
};

struct AttnArgs {
    int Nq;            // query rows
    int H;             // heads
    int kv_len;        // valid keys (keys >= kv_len are masked)
    int n_kv_tiles;    // ceil(kv_len / 128)
    float scale_log2;  // scale * log2(e)
    void* out;         // O, fp32 or bf16
    int64_t o_sb, o_sn, o_sh;  // O element strides
    float* lse;        // [B, H, Nq]
    float o_scale;     // FP8 path: O multiplied by this (descale of V); unused by bf16
    const uint32_t* mask;      // general mask bits (nullptr = none): bit j&31 of word
    int64_t mask_sb, mask_si;  //   mask[b*mask_sb + i*mask_si + j/32], rows i < mask_rows
    int mask_rows;
    const uint32_t* occ;       // MASK: occupancy bits per (b, 256-row block), occ_words each; nullptr = all tiles
    int occ_words;
    unsigned int* status;      // device status word (4 x u32)
    unsigned long long timeout_ns;
    // Work items are (b, h, 256-row block), counted block fastest, then head,
    // then batch (the bf16 kernel's grid order).  Items >= split_first (the
    // last partial wave) are each split into split_f key ranges run by a
    // second, 1-D launch (piece slot = (item - split_first) * split_f + piece)
    // that writes normalised partials (O, LSE) to ws_o [slot][256][D] and
    // ws_lse [slot][256]; launch_attn_tail_merge combines them into out / lse.
    // No split: split_first = items, split_f = 1, n_split_ctas = 0.  Unused by
    // the FP8 kernel.
    int n_qblk;                // ceil(Nq / 256)
    int split_first;
    int split_f;
    int n_split_ctas;          // (items - split_first) * split_f
    float* ws_o;
    float* ws_lse;
    int B;                     // batch count
    // Debug library only (zero in the product library): one injected fault
    // and the extents the in-kernel bounds checks compare against.
    uint32_t dbg_fault;        // DebugFault
    int dbg_fault_cta;         // linear block index of the CTA that injects it
    int dbg_fault_index;       // which load / commit / arrive is withheld
    int64_t dbg_o_elems;       // O elements reachable through its strides
    int64_t dbg_mask_words;    // mask words reachable through its strides
};

// Most pieces one split item is cut into (the tail merge kernel's unrolled
// bound); the plan itself lives in split_plan.h (host only).
constexpr int kMaxSplit = 8;

// Attention forward.  grid = (ceil(Nq/256), H, B), 384 threads, plus the
// split items' pieces (n_split_ctas CTAs) as a programmatic dependent launch.
// accumulate: merge into the fp32 (out, lse) already there instead of
// overwriting them (no split).
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnArgs& args, int B, int D, bool out_bf16, bool accumulate, cudaStream_t stream);

// Combine of the split pieces' partials into out / lse (after launch_attn_fwd
// on the same stream).  Nothing to do when args.n_split_ctas == 0.
cudaError_t launch_attn_tail_merge(const AttnArgs& args, int D, bool out_bf16, cudaStream_t stream);

// FP8 (E4M3) attention forward, D = 128.  Grid (ceil(Nq/256), H, B); the roles of the bf16
// kernel; scale_log2 already includes the Q and K descales.
cudaError_t launch_attn_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const AttnArgs& args, int B, bool out_bf16, cudaStream_t stream);

// Watchdog self-test: one CTA waits on a barrier nothing arrives on.
cudaError_t launch_watchdog_selftest(unsigned int* status, unsigned long long limit_ns, cudaStream_t stream);

struct MergeArgs {
    const float* o_parts;
    int64_t o_chunk_stride;
    int64_t o_row_stride;
    const float* lse_parts;
    int64_t lse_chunk_stride;
    int n_chunks;
    int B, Nq, H;
    void* out;
    float* lse_out;
};

cudaError_t launch_lse_merge(const MergeArgs& args, int D, bool out_bf16, cudaStream_t stream);

struct LayoutArgs {
    const uint16_t* qkv;
    int64_t stride_b, stride_n;
    int B, N, H, D;
    uint16_t* out[3];
};

cudaError_t launch_qkv_to_head_major(const LayoutArgs& args, cudaStream_t stream);

struct CastArgs {
    const uint16_t* qkv;        // bf16 [B, N, 3, H, D], (3, H, D) contiguous
    int64_t stride_b, stride_n; // elements
    int N;
    uint32_t hd;                // H * D (multiple of 16)
    uint32_t chunks_per_row;    // 3 * H * D / 16
    uint64_t total_chunks;      // B * N * chunks_per_row (< 2^32)
    float scale[3];             // q, k, v
    uint8_t* out;               // E4M3 [B, N, 3, H, D] contiguous
};

cudaError_t launch_qkv_cast_fp8(const CastArgs& args, cudaStream_t stream);

struct NormRopeArgs {
    const uint16_t* qkv;        // bf16 [B, N, 3, H, D], (3, H, D) contiguous
    int64_t stride_b, stride_n; // elements
    int B, N, H, D;
    const float* weight[2];     // RMSNorm weights [D] for q, k; nullptr = no norm for that tensor
    float eps;
    const float* cos;           // [N, D/2] fp32, nullptr = no rotation
    const float* sin;
    uint16_t* out[3];           // head-major [B, H, N, D]
};

cudaError_t launch_qkv_norm_rope(const NormRopeArgs& args, cudaStream_t stream);

// Occupancy pre-pass of the masked attention: bit t of occ[(b*RB + rb)*occ_words + t/32]
// is set when any row of the 256-row block rb attends any key of key tile t.
struct OccArgs {
    const uint32_t* mask;       // bit words, as AttnArgs
    int64_t mask_sb, mask_si;
    int mask_rows;
    int B, Nq, kv_len, n_kv_tiles, row_blocks, occ_words;
    uint32_t* occ;
};

cudaError_t launch_mask_occupancy(const OccArgs& args, cudaStream_t stream);

int device_sm_count(int device);

}  // namespace dit
