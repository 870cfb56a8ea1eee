// attn_fwd_fp8.cu -- attention forward on E4M3 Q/K/V (head dim 128), sm_103a,
// TMA + tcgen05 kind::f8f6f4, fp32 accumulators in TMEM.
//
// The FP8 attention that "Scaling Video Generation Across NVL72 rack with
// TensorRT-LLM" ("Ulysses Parallelism", paragraph "Fused vs. unfused QKV
// all-to-all") feeds with the one-pass cast of the stacked QKV buffer: the
// cast output is read in place through (b, n, h) strides.  Q, K, V stand for
// q8 * descale_q, k8 * descale_k, v8 * descale_v; the kernel computes
//     O = softmax(scale * Q K^T) V,   LSE = ln sum_j exp(scale * q . k_j)
// exactly as the bf16 kernel does, with S = q8 . k8 accumulated in fp32 and
// scale * descale_q * descale_k folded into the exponent.
//
// Same CTA shape, warp roles, TMEM map and product order as the bf16 kernel
// (256 query rows of one head as two 128-row tiles; warps 0-7 softmax, warp 8
// MMA, warp 9 TMA).  A 128 x 128 E4M3 tile is 16 KB and exactly one 128-byte
// swizzle column wide, so every tile moves in one TMA copy and the ring holds
// eight stages.  Each product is four K = 32 instructions.
//
// P is fed to the PV product as E4M3 (four keys per 32-bit TMEM column, the
// lowest key in the lowest byte), so it must stay <= 448.  P = 2^(x - m + 7),
// x = s * scale * log2(e), with m the running row max; m moves only when a
// tile's max exceeds it by more than 1.75, so P <= 2^8.75 < 448, and the
// smallest kept values (2^-9) are ~2^-16 below the row max.  Unlike the bf16
// kernel, this needs the tile max every tile.  The row sum l accumulates the
// unrounded fp32 P; O = (sum P v8) * descale_v / l.
//
// The epilogue stages O through the idle Q buffer and stores whole 128-byte
// lines, and the grid's last partial wave can be split over key ranges
// (PIECE, a programmatic dependent launch), exactly as in the bf16 kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "debug.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kD = 128;
constexpr int kThreads = 384;
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kOtherRegs = 88;
static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * 168, "register split");
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kPOffset = 7.f;   // P = 2^(x - m + kPOffset)
constexpr float kStale = 1.75f;   // keep m while the tile max is <= m + kStale

constexpr int kTile = kBM * kD;   // bytes of one 128 x 128 E4M3 tile
constexpr int kStages = 8;
constexpr int kQFull = 0;
constexpr int kKVFull = 2;
constexpr int kKVEmpty = kKVFull + kStages;
constexpr int kSFull = kKVEmpty + kStages;
constexpr int kPFull = kSFull + 2;
constexpr int kOFinal = kPFull + 2;
constexpr int kDrain = kOFinal + 2;
constexpr int kLoadDrain = kDrain + 1;
constexpr int kNumBars = kLoadDrain + 1;
constexpr int kBarOffset = (2 + kStages) * kTile;
constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(256 + 2 * kD <= 512, "S0, S1, O0, O1 fit the 512 TMEM columns");

__device__ __forceinline__ float max64(const float* v) {
    float t8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t8[k] = max3f(v[k], v[8 + k], v[16 + k]);
#pragma unroll
    for (int k = 0; k < 8; ++k) t8[k] = max3f(t8[k], v[24 + k], v[32 + k]);
#pragma unroll
    for (int k = 0; k < 8; ++k) t8[k] = max3f(t8[k], v[40 + k], v[48 + k]);
#pragma unroll
    for (int k = 0; k < 8; ++k) t8[k] = fmaxf(t8[k], v[56 + k]);
    return max3f(max3f(t8[0], t8[1], t8[2]), max3f(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7]));
}

// PIECE: the kernel of the split items' key-range pieces (1-D grid, partials
// to the workspace); the whole-item kernel is compiled without any of it.
template <bool OUT_BF16, bool PIECE = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
    constexpr int S = kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t sQ = s_base;                  // Q tile t at sQ + t*kTile
    const uint32_t sRing = s_base + 2 * kTile;   // slot s at sRing + s*kTile
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
    auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work item of this CTA: (256-row block, head, batch) = (x, y, z) for a
    // whole item; a piece decodes its item and first key tile from its 1-D
    // index (items counted block fastest, then head, then batch).
    int k_begin = 0, n_tiles = a.n_kv_tiles;
    int h, b, q_row0;
    if constexpr (PIECE) {
        const int slot = static_cast<int>(blockIdx.x);
        const int piece = slot % a.split_f;
        const int item = a.split_first + slot / a.split_f;
        k_begin = static_cast<int>(static_cast<int64_t>(piece) * a.n_kv_tiles / a.split_f);
        n_tiles = static_cast<int>(static_cast<int64_t>(piece + 1) * a.n_kv_tiles / a.split_f) - k_begin;
        q_row0 = (item % a.n_qblk) * (2 * kBM);
        h = (item / a.n_qblk) % a.H;
        b = item / a.n_qblk / a.H;
    } else {
        h = blockIdx.y;
        b = blockIdx.z;
        q_row0 = blockIdx.x * (2 * kBM);
        // The piece kernel (if any) may start once every CTA here has begun;
        // the items it covers are the last in grid order and left to it.
        if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) >= a.split_first) return;
    }
    // (debug library) the item and its key range lie inside the problem
    if (!in_bounds(h >= 0 && h < a.H && b >= 0 && b < a.B && q_row0 >= 0 && q_row0 < a.Nq && k_begin >= 0 &&
                       n_tiles >= 0 && k_begin + n_tiles <= a.n_kv_tiles,
                   a.status, 0, BND_ITEM))
        return;

    if (threadIdx.x == 0) {
        mbar_init(bar(kQFull + 0), 1);
        mbar_init(bar(kQFull + 1), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(kKVFull + s), 1);
            mbar_init(bar(kKVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(kSFull + t), 1);
            mbar_init(bar(kPFull + t), 128);
            mbar_init(bar(kOFinal + t), 1);
        }
        mbar_init(bar(kDrain), 1);
        mbar_init(bar(kLoadDrain), 1);
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{a.status, a.timeout_ns, abort_flag};
    const Watchdog wd_drain{a.status, a.timeout_ns, never_flag};

    if (warp >= 10) {
        regs_decrease<kOtherRegs>();
    } else if (warp == 9) {
        regs_decrease<kOtherRegs>();
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            for (int t = 0; t < 2; ++t) {
                mbar_arrive_expect_tx(bar(kQFull + t), kTile);
                tma_load_4d(sQ + t * kTile, &tm_q, bar(kQFull + t), 0, q_row0 + t * kBM, h, b);
            }
            const int total = 2 * n_tiles;
            int issued = 0;
            int withheld = -1;   // (debug library) the load skipped on request
            for (int i = 0; i < total; ++i) {
                const int slot = i % S;
                const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
                const int key0 = (k_begin + (i >> 1)) * kBN;
                if (!in_bounds(key0 >= 0 && key0 < a.kv_len, a.status, ROLE_LOAD, BND_KEY)) break;
                if (!wait_bounded(bar(kKVEmpty + slot), ph ^ 1u, wd, ROLE_LOAD, SITE_KV_EMPTY)) break;
                issued = i + 1;
                if (inject(a, FAULT_SKIP_LOAD, i)) {
                    withheld = i;   // neither the arrive nor the copy: the slot never fills
                    continue;
                }
                mbar_arrive_expect_tx(bar(kKVFull + slot), kTile);
                tma_load_4d(sRing + slot * kTile, (i & 1) ? &tm_v : &tm_k, bar(kKVFull + slot), 0, key0, h, b);
            }
            if (issued < total || *abort_flag) {
                for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
                    if (i != withheld)
                        wait_bounded(bar(kKVFull + i % S), static_cast<uint32_t>(i / S) & 1u, wd_drain, ROLE_LOAD,
                                     SITE_LOAD_DRAIN);
                wait_bounded(bar(kQFull + 0), 0, wd_drain, ROLE_LOAD, SITE_LOAD_DRAIN);
                wait_bounded(bar(kQFull + 1), 0, wd_drain, ROLE_LOAD, SITE_LOAD_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        regs_decrease<kOtherRegs>();
        // ------------------------------------------------------------- MMA issuer
        // The whole warp runs this block and one elected lane issues each
        // product and commit (the *_warp forms): the issue loop stays
        // warp-uniform and keeps pace with the tensor pipe while the softmax
        // warps keep every SM sub-partition's issue slots busy.
        if (n_tiles > 0) {
            constexpr uint32_t kIdescQK = idesc_e4m3_f32(kBM, kBN, false);
            constexpr uint32_t kIdescPV = idesc_e4m3_f32(kBM, kD, true);
            const uint32_t tS0 = tmem, tS1 = tmem + 128;
            const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + kD;

            // S_t = Q_t K^T: both K-major, 32 channels (32 bytes) per instruction.
            auto issue_qk = [&](uint32_t tS, uint32_t q_addr, uint32_t k_addr) {
                const uint64_t dq = sdesc_sw128(q_addr, 16, 1024), dk = sdesc_sw128(k_addr, 16, 1024);
                static_for<kD / 32>([&](auto kk) {
                    umma_ss_f8_warp<kk.value * 32>(tS, dq, dk, kIdescQK, kk.value > 0 ? 1u : 0u);
                });
            };
            // O_t (+)= P_t V: P from TMEM (8 columns = 32 keys per instruction),
            // V MN-major, 32 keys = four 8-row swizzle atoms = 4096 bytes.
            auto issue_pv = [&](uint32_t tO, uint32_t tP, uint32_t v_addr, bool accumulate) {
                const uint64_t dv = sdesc_sw128(v_addr, 16384, 1024);
                static_for<kBN / 32>([&](auto kk) {
                    umma_ts_f8_warp<kk.value * 4096>(tO, tP + kk.value * 8, dv, kIdescPV,
                                                     (accumulate || kk.value > 0) ? 1u : 0u);
                });
            };

            bool ok = wait_bounded_warp(bar(kQFull + 0), 0, wd, ROLE_MMA, SITE_Q_FULL) &&
                      wait_bounded_warp(bar(kQFull + 1), 0, wd, ROLE_MMA, SITE_Q_FULL) &&
                      wait_bounded_warp(bar(kKVFull + 0), 0, wd, ROLE_MMA, SITE_KV_FULL);
            // S_0 number n is ready (the debug library can withhold one signal)
            auto commit_s0 = [&](int n) {
                if (!inject(a, FAULT_SKIP_S_COMMIT, n)) umma_commit_warp(bar(kSFull + 0));
            };
            if (ok) {
                tc_fence_after();
                issue_qk(tS0, sQ, sRing);
                commit_s0(0);
                issue_qk(tS1, sQ + kTile, sRing);
                umma_commit_warp(bar(kSFull + 1));
                umma_commit_warp(bar(kKVEmpty + 0));
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int iv = 2 * j + 1, ik = 2 * j + 2;
                const uint32_t v_addr = sRing + (iv % S) * kTile;
                const uint32_t k_addr = sRing + (ik % S) * kTile;
                const bool more = j + 1 < n_tiles;
                const uint32_t ph = static_cast<uint32_t>(j) & 1u;
                if (!in_bounds(v_addr >= sRing && v_addr + kTile <= sRing + S * kTile && k_addr >= sRing &&
                                   k_addr + kTile <= sRing + S * kTile,
                               a.status, ROLE_MMA, BND_SMEM))
                    break;
                // K of the next tile as well as V of this one: both land long before P_0
                // is ready, and waiting for them here keeps the K wait out of the chain
                // that P_0 starts (P.V_0 -> Q.K_0 -> S_0 -> the softmax).
                ok = wait_bounded_warp(bar(kKVFull + iv % S), static_cast<uint32_t>(iv / S) & 1u, wd, ROLE_MMA,
                                       SITE_KV_FULL) &&
                     (!more || wait_bounded_warp(bar(kKVFull + ik % S), static_cast<uint32_t>(ik / S) & 1u, wd,
                                                 ROLE_MMA, SITE_KV_FULL)) &&
                     wait_bounded_warp(bar(kPFull + 0), ph, wd, ROLE_MMA, SITE_P_FULL);
                if (!ok) break;
                tc_fence_after();
                issue_pv(tO0, tS0, v_addr, j > 0);
                if (more) {
                    issue_qk(tS0, sQ, k_addr);
                    commit_s0(j + 1);
                } else {
                    umma_commit_warp(bar(kOFinal + 0));
                }
                ok = wait_bounded_warp(bar(kPFull + 1), ph, wd, ROLE_MMA, SITE_P_FULL);
                if (!ok) break;
                tc_fence_after();
                issue_pv(tO1, tS1, v_addr, j > 0);
                umma_commit_warp(bar(kKVEmpty + iv % S));
                if (more) {
                    issue_qk(tS1, sQ + kTile, k_addr);
                    umma_commit_warp(bar(kSFull + 1));
                    umma_commit_warp(bar(kKVEmpty + ik % S));
                } else {
                    umma_commit_warp(bar(kOFinal + 1));
                }
            }
            umma_commit_warp(bar(kDrain));
            wait_bounded_warp(bar(kDrain), 0, wd_drain, ROLE_MMA, SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- softmax warps
        regs_increase<kSoftmaxRegs>();
        const int t = warp >> 2;
        const int wq = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * kD;
        const int row = q_row0 + t * kBM + wq * 32 + lane;
        const float sl2 = a.scale_log2;
        float m = -INFINITY;  // running max of x = s * sl2 (possibly stale by <= kStale)
        float l = 0.f;        // running sum of 2^(x - m + kPOffset)
        bool ok = true;

        // P for 64 scores -> 16 TMEM columns of four E4M3 at tP; returns sum P.
        auto exp_store = [&](const float* v, uint32_t tP, float neg) {
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float x0, x1, x2, x3;
                ffma2_bc(x0, x1, v[4 * i], v[4 * i + 1], sl2, neg);
                ffma2_bc(x2, x3, v[4 * i + 2], v[4 * i + 3], sl2, neg);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                fadd2_acc(a0, a1, p0, p1);
                fadd2_acc(b0, b1, p2, p3);
                pk[i] = pack_e4m3x4(p0, p1, p2, p3);
            }
            tmem_st16(tP, pk);
            return (a0 + a1) + (b0 + b1);
        };

        for (int j = 0; j < n_tiles; ++j) {
            ok = wait_bounded(bar(kSFull + t), static_cast<uint32_t>(j) & 1u, wd, ROLE_SOFTMAX, SITE_S_FULL);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();

            // The S row with its maximum: each load also reduces its 32 columns.
            uint32_t sr[4][32];
            float pm[4];
            tmem_ld32_max(tS + 0, sr[0], pm[0]);
            tmem_ld32_max(tS + 32, sr[1], pm[1]);
            tmem_ld32_max(tS + 64, sr[2], pm[2]);
            tmem_ld32_max(tS + 96, sr[3], pm[3]);
            tmem_ld_wait_dep(sr[0]);
            reg_dep(sr[1]);
            reg_dep(sr[2]);
            reg_dep(sr[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) reg_dep(pm[i]);
            const int valid = a.kv_len - (k_begin + j) * kBN;   // >= 1
            float s[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
            float mx = fmaxf(max3f(pm[0], pm[1], pm[2]), pm[3]);
            if (valid < 128) {
                // last tile: the columns past the valid keys hold scores of the
                // zero-filled key rows, so the maximum is taken over the valid ones
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= valid) s[c] = -INFINITY;
                mx = fmaxf(max64(s), max64(s + 64));
            }
            mx *= sl2;
            const bool need = mx > m + kStale;   // always true on the first tile
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mx : m;
                const float alpha = ex2_approx(m - m_new);
                l *= alpha;
                if (j > 0) {
                    // O holds PV(j-1): S(j) was committed after it.
#pragma unroll
                    for (int cc = 0; cc < kD / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait_dep(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + cc * 32, o);
                    }
                }
                m = m_new;
            }
            const float neg = kPOffset - m;
            l += exp_store(s, tS, neg) + exp_store(s + 64, tS + 16, neg);
            tmem_st_wait();
            tc_fence_before();
            if (!(warp == 0 && inject(a, FAULT_SKIP_P_ARRIVE, j))) mbar_arrive(bar(kPFull + t));
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && n_tiles > 0) {
            ok = wait_bounded(bar(kOFinal + t), 0, wd, ROLE_SOFTMAX, SITE_O_FINAL);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok) {
            const bool in_range = row < a.Nq;
            const int64_t lse_idx = (static_cast<int64_t>(b) * a.H + h) * a.Nq + row;
            const float c_new = n_tiles > 0 ? a.o_scale / l : 0.f;
            // Each 32-column chunk goes through this warp's 4 KB of the Q_t buffer
            // (idle since QK_t(last) completed): a thread writes its row, then the
            // warp stores four rows per instruction as whole 128-byte lines.  Rows
            // sit 128 bytes apart with the 16-byte groups XOR-swizzled by the row.
            float4* stg = reinterpret_cast<float4*>(smem + t * kTile + wq * 4096);
            const int k4 = lane & 7;        // 16-byte group this lane moves in the store phase
            const int r_sub = lane >> 3;    // row within each group of four
#pragma unroll 1
            for (int cc = 0; cc < kD / 32; ++cc) {
                uint32_t o[32];
                if (n_tiles > 0) {
                    tmem_ld32(tO + cc * 32, o);
                    tmem_ld_wait_dep(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                    stg[lane * 8 + (v4 ^ (lane & 7))] =
                        make_float4(__uint_as_float(o[4 * v4 + 0]) * c_new, __uint_as_float(o[4 * v4 + 1]) * c_new,
                                    __uint_as_float(o[4 * v4 + 2]) * c_new, __uint_as_float(o[4 * v4 + 3]) * c_new);
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int r = it * 4 + r_sub;                   // row within the warp's 32
                    const float4 val = stg[r * 8 + (k4 ^ (r & 7))];
                    const int grow = q_row0 + t * kBM + wq * 32 + r;
                    if (PIECE && grow < a.Nq) {
                        // a piece's fp32 partial, row-major [256][D] in its workspace slot
                        const int64_t wi = (static_cast<int64_t>(blockIdx.x) * (2 * kBM) + (grow - q_row0)) * kD + cc * 32 + 4 * k4;
                        if (in_bounds(wi >= 0 && wi + 4 <= static_cast<int64_t>(a.n_split_ctas) * (2 * kBM) * kD, a.status,
                                      ROLE_SOFTMAX, BND_WS))
                            *reinterpret_cast<float4*>(a.ws_o + wi) = val;
                    } else if (grow < a.Nq) {
                        const int64_t off = static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(grow) * a.o_sn +
                                            static_cast<int64_t>(h) * a.o_sh + cc * 32 + 4 * k4;
                        if (!in_bounds(off >= 0 && off + 4 <= a.dbg_o_elems, a.status, ROLE_SOFTMAX, BND_OUT)) continue;
                        if constexpr (OUT_BF16)
                            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + off) =
                                make_uint2(pack_bf16x2(val.x, val.y), pack_bf16x2(val.z, val.w));
                        else
                            *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) = val;
                    }
                }
                __syncwarp();
            }
            const float lse_out = n_tiles > 0 ? (m - kPOffset + log2f(l)) * kLn2 : -INFINITY;
            if (in_range) {
                if (PIECE) {
                    const int64_t wi = static_cast<int64_t>(blockIdx.x) * (2 * kBM) + (row - q_row0);
                    if (in_bounds(wi >= 0 && wi < static_cast<int64_t>(a.n_split_ctas) * (2 * kBM), a.status,
                                  ROLE_SOFTMAX, BND_WS))
                        a.ws_lse[wi] = lse_out;
                } else if (in_bounds(lse_idx >= 0 && lse_idx < static_cast<int64_t>(a.B) * a.H * a.Nq, a.status,
                                     ROLE_SOFTMAX, BND_LSE)) {
                    a.lse[lse_idx] = lse_out;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // A piece completes only after the whole-item grid it was launched beside
    // (whose outputs are the stream's too); by then that grid has no CTA left
    // to schedule, so the wait holds nothing back.
    if constexpr (PIECE) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool BF16>
cudaError_t launch_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& args,
                        int B, cudaStream_t stream) {
    auto kern = attn_fwd_fp8_kernel<BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((args.Nq + 2 * kBM - 1) / (2 * kBM), args.H, B);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, args);
    e = cudaGetLastError();
    if (e != cudaSuccess || args.n_split_ctas == 0) return e;
    // The split items' pieces: a programmatic dependent launch, so that its
    // CTAs take SMs as the last whole items drain instead of after the grid.
    auto piece = attn_fwd_fp8_kernel<BF16, true>;
    e = cudaFuncSetAttribute(piece, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(args.n_split_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, piece, tq, tk, tv, args);
}

}  // namespace

cudaError_t launch_attn_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const AttnArgs& args, int B, bool out_bf16, cudaStream_t stream) {
    return out_bf16 ? launch_impl<true>(tq, tk, tv, args, B, stream) : launch_impl<false>(tq, tk, tv, args, B, stream);
}

}  // namespace dit
