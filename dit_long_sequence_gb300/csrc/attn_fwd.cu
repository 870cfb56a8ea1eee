// attn_fwd.cu -- dense bidirectional attention forward with per-row LSE,
// sm_103a, TMA + tcgen05 (TMEM accumulators), warp-specialised.
//
// Computes, for every (b, h) head and query row i,
//     O[b,i,h,:] = sum_j softmax_j(scale * q_i . k_j) v_j,
//     LSE[b,h,i] = ln sum_j exp(scale * q_i . k_j),
// over the valid keys j < kv_len -- the inner attention of "Scaling Video
// Generation Across NVL72 rack with TensorRT-LLM" ("The Scaling Challenge in
// Video Generation": dense, unmasked, bidirectional; "Attention2D
// Parallelism" / "Local Attention": output plus LSE so partial passes merge).
// The key-only tail mask follows "8 卡怎么分 token：LTX-2 序列并行的 all2all
// 到底搬了什么" ("构造 padding mask").
//
// CTA = 256 query rows of one (b, h) -- a work item -- as two 128-row tiles,
// 12 warps:
//   warps 0-3  softmax for query tile 0 (one TMEM lane = one row per thread)
//   warps 4-7  softmax for query tile 1
//   warp  8    tcgen05.mma issuer (the whole warp runs the issue loop, one
//              elected lane issues); owns the TMEM allocation
//   warp  9    TMA producer (one thread): Q once, then K_0, V_0, K_1, V_1, ...
//              through a ring of STAGES shared-memory slots
//   warps 10-11 idle (they complete the third warpgroup)
// Registers: launched at 168 per thread (3 warps per SM sub-partition); the
// softmax warpgroups raise theirs to 208 and the third warpgroup drops to 88,
// which sums to the launch budget exactly (256*208 + 128*88 = 384*168).
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
// P_t (bf16, 64 columns) is written by the softmax warps over the first half of
// S_t and fed to the PV product as the TMEM A operand.
//
// Per KV tile j the MMA warp issues, in order,
//   PV0(j) and QK0(j+1) once P0(j) is ready, then PV1(j) and QK1(j+1) once
//   P1(j) is ready -- so the tensor pipe runs one tile's products while the
//   other tile's softmax runs.  Products issued by one lane execute in order,
//   which makes writing S_t(j+1) over P_t(j) safe after PV_t(j).
//
// Online softmax in log2 units with a lazy rescale: the running max m of a row
// is set by the first key tile and only moves (O and l rescaled by
// 2^(m_old - m_new)) when a later tile's row sum of 2^(s*sl2 - m) exceeds 2^39;
// otherwise every P <= 2^39, which bf16 P and the fp32 accumulators carry with
// unchanged relative precision, and the final O / l and LSE = ln2 * (m + log2 l)
// are exact whatever m is.  So the steady state needs no per-tile row max at
// all: the exponents are computed straight away and the already-needed row sum
// doubles as the overflow check; the rare warps that fail it recompute P.
//
// Keys j >= kv_len are outside the K/V tensor maps (zero fill) and masked to
// -inf in the last tile, so pad rows are never read.
//
// Grid: (256-row blocks, H, B), one CTA per work item.  With a workspace the
// items of the last partial wave (items mod SMs of them, the last in grid
// order) are left by this grid to a second launch of the same kernel body
// (PIECE) that runs each of them as f key-range pieces.  That launch is a
// programmatic dependent launch: every CTA here signals at its start, so the
// pieces may be scheduled once the last whole item has begun, and they take
// SMs as the last whole items drain -- the end of the work is balanced at
// 1/f of an item's time instead of a whole item (SMs also differ in speed by
// ~1-2%, which a fine-grained end absorbs too).  Each piece writes its
// normalised partial O and LSE to the workspace, and attn_tail_merge_kernel
// combines each item's f partials exactly as the (O, LSE) merge does.  The
// whole-item kernel is compiled without any of the piece logic: its softmax
// loop sits at the edge of its register budget, where one more value held
// across the loop costs ~2% of the loop's time.
//
// MASK variant: a general (B, T, T) mask -- one bit per (query, key), shared by
// the heads -- also sets masked scores to -inf; rows i >= mask_rows attend every
// valid key (the pad-row rule of "8 卡怎么分 token", "构造 padding mask").  Each
// softmax thread loads its row's 128 mask bits per key tile with one 16-byte
// load, issued a tile ahead.  A row whose keys are all masked so far has
// m = -inf: its exponentials use 0 as the offset (all its P are 0), every
// later tile takes the slow path until one sets a finite m (rescale factor 1
// while m stays -inf), and a row with no allowed key at all ends with O = 0,
// LSE = -inf.  With an occupancy map (one bit per (256-row block, key tile):
// does any row of the block attend any key of the tile), every role walks only
// the occupied key tiles -- the TMA producer loads, the MMA warp multiplies
// and the softmax warps exponentiate nothing else.  The masked kernel splits
// its last partial wave the same way: a piece walks the occupied tiles of its
// own key range, and a piece whose range holds no key a row may attend gives
// that row LSE = -inf, i.e. weight 0 in the merge.
#include <cuda.h>
#include <cuda_runtime.h>

#include "debug.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dit {
namespace {

// Walks the set bits of one CTA's occupancy words in [begin, end) (the key
// tiles to process; begin < end when there is a map); without a map every
// tile is occupied.
struct TileCursor {
    const uint32_t* words;   // nullptr: all tiles of the range
    int n_words, n, w;
    uint32_t bits;
    int next_all;
    __device__ TileCursor(const uint32_t* occ, int begin, int end)
        : words(occ), n_words((end + 31) / 32), n(end), w(begin >> 5),
          bits(occ ? occ[begin >> 5] & (~0u << (begin & 31)) : 0u), next_all(begin) {}
    // The next key tile to process, or -1.
    __device__ int next() {
        if (words == nullptr) return next_all < n ? next_all++ : -1;
        while (bits == 0u) {
            if (++w >= n_words) return -1;
            bits = words[w];
        }
        const int t = w * 32 + __ffs(static_cast<int>(bits)) - 1;
        bits &= bits - 1u;
        return t < n ? t : -1;
    }
};

// Occupied key tiles in [begin, end) (all of them without a map).
__device__ __forceinline__ int count_tiles(const uint32_t* occ, int begin, int end) {
    if (occ == nullptr) return end - begin;
    int c = 0;
    for (int w = begin >> 5; w < (end + 31) >> 5; ++w) {
        uint32_t bits = occ[w];
        if (w == (begin >> 5)) bits &= ~0u << (begin & 31);
        if (w == ((end - 1) >> 5) && (end & 31) != 0) bits &= (1u << (end & 31)) - 1u;
        c += __popc(bits);
    }
    return c;
}

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per KV tile
constexpr int kThreads = 384;
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kOtherRegs = 88;
static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * 168, "register split");
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSumLimit = 549755813888.0f;  // 2^39: largest tile row sum kept without a rescale

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kBM * D * 2;          // one 128 x D bf16 tile
    static constexpr int kStages = (D == 128) ? 4 : 8;      // K/V ring slots
    static constexpr int kBlockBytes = kBM * 128;           // 128 rows x 64 bf16 (one swizzle column)
    // barriers
    static constexpr int kQFull = 0;
    static constexpr int kKVFull = 2;
    static constexpr int kKVEmpty = kKVFull + kStages;
    static constexpr int kSFull = kKVEmpty + kStages;
    static constexpr int kPFull = kSFull + 2;
    static constexpr int kOFinal = kPFull + 2;
    static constexpr int kDrain = kOFinal + 2;
    static constexpr int kLoadDrain = kDrain + 1;
    static constexpr int kNumBars = kLoadDrain + 1;
    static constexpr int kBarOffset = (2 + kStages) * kTileBytes;
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kBarOffset + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(256 + 2 * D <= 512, "S0, S1, O0, O1 fit the 512 TMEM columns");
};

// ACCUM: fold this pass into an existing fp32 (O, LSE) pair instead of
// overwriting it (streaming merge over key chunks).  MASK: apply the bit mask.
// PIECE: the kernel of the split items' key-range pieces (1-D grid, partials
// to the workspace); the whole-item kernel is compiled without any of it.
template <int D, bool OUT_BF16, bool ACCUM, bool MASK, bool PIECE = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
    using C = Cfg<D>;
    constexpr int S = C::kStages;
    constexpr int TILE = C::kTileBytes;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t sQ = s_base;                 // Q tile t at sQ + t*TILE
    const uint32_t sRing = s_base + 2 * TILE;   // slot s at sRing + s*TILE
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // stays 0
    auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work item of this CTA: (256-row block, head, batch) = (x, y, z) for a
    // whole item; a piece decodes its item and key range from its 1-D index
    // (items counted block fastest, then head, then batch).
    static_assert(!PIECE || !ACCUM, "only overwriting passes are split");
    struct W { int h, b, q_row0, qblk; };
    int k_begin = 0, k_end = a.n_kv_tiles;   // key tiles [k_begin, k_end) of this CTA
    auto item_w = [&]() {
        W w;
        if constexpr (PIECE) {
            const int slot = static_cast<int>(blockIdx.x);
            const int piece = slot % a.split_f;
            const int item = a.split_first + slot / a.split_f;
            k_begin = static_cast<int>(static_cast<int64_t>(piece) * a.n_kv_tiles / a.split_f);
            k_end = static_cast<int>(static_cast<int64_t>(piece + 1) * a.n_kv_tiles / a.split_f);
            w.qblk = item % a.n_qblk;
            w.h = (item / a.n_qblk) % a.H;
            w.b = item / a.n_qblk / a.H;
        } else {
            w.qblk = blockIdx.x;
            w.h = blockIdx.y;
            w.b = blockIdx.z;
        }
        w.q_row0 = w.qblk * (2 * kBM);
        return w;
    };
    const W wk = item_w();
    const int h = wk.h;
    const int b = wk.b;
    const int q_row0 = wk.q_row0;
    // (debug library) the item and its key range lie inside the problem
    if (!in_bounds(h >= 0 && h < a.H && b >= 0 && b < a.B && q_row0 >= 0 && q_row0 < a.Nq && k_begin >= 0 &&
                       k_begin <= k_end && k_end <= a.n_kv_tiles,
                   a.status, 0, BND_ITEM))
        return;
    if constexpr (!PIECE && !ACCUM) {
        // The piece kernel (if any) may start once every CTA here has begun;
        // the items it covers are the last in grid order and left to it.
        if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)) >= a.split_first) return;
    }
    // MASK with an occupancy map: this item's row of tile bits
    const uint32_t* occ = (MASK && a.occ != nullptr)
                              ? a.occ + (static_cast<int64_t>(b) * a.n_qblk + wk.qblk) * a.occ_words
                              : nullptr;
    const int n_tiles = count_tiles(occ, k_begin, k_end);   // key tiles this CTA processes

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kQFull + 0), 1);
        mbar_init(bar(C::kQFull + 1), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(C::kKVFull + s), 1);
            mbar_init(bar(C::kKVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::kSFull + t), 1);
            mbar_init(bar(C::kPFull + t), 128);
            mbar_init(bar(C::kOFinal + t), 1);
        }
        mbar_init(bar(C::kDrain), 1);
        mbar_init(bar(C::kLoadDrain), 1);
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
    // A second watchdog view that ignores the abort flag: used only to wait
    // (bounded) for work already in flight while winding down.
    const Watchdog wd_drain{a.status, a.timeout_ns, never_flag};

    if (warp >= 10) {
        regs_decrease<kOtherRegs>();  // idle warps
    } else if (warp == 9) {
        regs_decrease<kOtherRegs>();
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            for (int t = 0; t < 2; ++t) {
                mbar_arrive_expect_tx(bar(C::kQFull + t), TILE);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sQ + t * TILE + c * C::kBlockBytes, &tm_q, bar(C::kQFull + t), c * 64,
                                q_row0 + t * kBM, h, b);
            }
            const int total = 2 * n_tiles;
            int issued = 0;
            int withheld = -1;   // (debug library) the load skipped on request
            TileCursor cur(occ, k_begin, k_end);
            int key0 = 0;
            for (int i = 0; i < total; ++i) {
                if ((i & 1) == 0) key0 = cur.next() * kBN;
                if (!in_bounds(key0 >= 0 && key0 < a.kv_len, a.status, ROLE_LOAD, BND_KEY)) break;
                const int slot = i % S;
                const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
                if (!wait_bounded(bar(C::kKVEmpty + slot), ph ^ 1u, wd, ROLE_LOAD, SITE_KV_EMPTY)) break;
                issued = i + 1;
                if (inject(a, FAULT_SKIP_LOAD, i)) {
                    withheld = i;   // neither the arrive nor the copy: the slot never fills
                    continue;
                }
                mbar_arrive_expect_tx(bar(C::kKVFull + slot), TILE);
                const CUtensorMap* tm = (i & 1) ? &tm_v : &tm_k;
                const uint32_t dst = sRing + slot * TILE;
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(dst + c * C::kBlockBytes, tm, bar(C::kKVFull + slot), c * 64, key0, h, b);
            }
            if (issued < total || *abort_flag) {
                // Winding down: wait (bounded) until every copy issued has landed.
                for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
                    if (i != withheld)
                        wait_bounded(bar(C::kKVFull + i % S), static_cast<uint32_t>(i / S) & 1u, wd_drain,
                                     ROLE_LOAD, SITE_LOAD_DRAIN);
                wait_bounded(bar(C::kQFull + 0), 0, wd_drain, ROLE_LOAD, SITE_LOAD_DRAIN);
                wait_bounded(bar(C::kQFull + 1), 0, wd_drain, ROLE_LOAD, SITE_LOAD_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        regs_decrease<kOtherRegs>();
        // ------------------------------------------------------------- MMA issuer
        // The whole warp runs this block and one elected lane issues each
        // product and commit (the *_warp forms), so the issue loop stays
        // warp-uniform and keeps pace with the tensor pipe while the softmax
        // warps keep every SM sub-partition's issue slots busy.
        if (n_tiles > 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, true);
            const uint32_t tS0 = tmem, tS1 = tmem + 128;
            const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;

            // S_t = Q_t K^T : A = Q (K-major), B = K (K-major), K-dim = D.
            auto issue_qk = [&](uint32_t tS, uint32_t q_addr, uint32_t k_addr) {
                const uint64_t dq = sdesc_sw128(q_addr, 16, 1024), dk = sdesc_sw128(k_addr, 16, 1024);
                static_for<D / 16>([&](auto kk) {
                    constexpr uint32_t off = (kk.value >> 2) * C::kBlockBytes + (kk.value & 3) * 32;
                    umma_ss_warp<off>(tS, dq, dk, kIdescQK, kk.value > 0 ? 1u : 0u);
                });
            };
            // O_t (+)= P_t V : A = P (TMEM, bf16 pairs), B = V (MN-major), K-dim = 128 keys.
            auto issue_pv = [&](uint32_t tO, uint32_t tP, uint32_t v_addr, bool accumulate) {
                const uint64_t dv = sdesc_sw128(v_addr, C::kBlockBytes, 1024);
                static_for<kBN / 16>([&](auto kk) {
                    umma_ts_warp<kk.value * 16 * 128>(tO, tP + kk.value * 8, dv, kIdescPV,
                                                      (accumulate || kk.value > 0) ? 1u : 0u);
                });
            };

            bool ok = wait_bounded_warp(bar(C::kQFull + 0), 0, wd, ROLE_MMA, SITE_Q_FULL) &&
                      wait_bounded_warp(bar(C::kQFull + 1), 0, wd, ROLE_MMA, SITE_Q_FULL) &&
                      wait_bounded_warp(bar(C::kKVFull + 0), 0, wd, ROLE_MMA, SITE_KV_FULL);
            // S_0 number n is ready (the debug library can withhold one signal)
            auto commit_s0 = [&](int n) {
                if (!inject(a, FAULT_SKIP_S_COMMIT, n)) umma_commit_warp(bar(C::kSFull + 0));
            };
            if (ok) {
                tc_fence_after();
                issue_qk(tS0, sQ, sRing);
                commit_s0(0);
                issue_qk(tS1, sQ + TILE, sRing);
                umma_commit_warp(bar(C::kSFull + 1));
                umma_commit_warp(bar(C::kKVEmpty + 0));
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int iv = 2 * j + 1, ik = 2 * j + 2;
                const uint32_t v_addr = sRing + (iv % S) * TILE;
                const uint32_t k_addr = sRing + (ik % S) * TILE;
                const bool more = j + 1 < n_tiles;
                const uint32_t ph = static_cast<uint32_t>(j) & 1u;
                if (!in_bounds(v_addr >= sRing && v_addr + TILE <= sRing + S * TILE && k_addr >= sRing &&
                                   k_addr + TILE <= sRing + S * TILE,
                               a.status, ROLE_MMA, BND_SMEM))
                    break;
                ok = wait_bounded_warp(bar(C::kKVFull + iv % S), static_cast<uint32_t>(iv / S) & 1u, wd, ROLE_MMA,
                                       SITE_KV_FULL) &&
                     wait_bounded_warp(bar(C::kPFull + 0), ph, wd, ROLE_MMA, SITE_P_FULL);
                if (!ok) break;
                tc_fence_after();
                issue_pv(tO0, tS0, v_addr, j > 0);
                if (more) {
                    ok = wait_bounded_warp(bar(C::kKVFull + ik % S), static_cast<uint32_t>(ik / S) & 1u, wd,
                                           ROLE_MMA, SITE_KV_FULL);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(tS0, sQ, k_addr);
                    commit_s0(j + 1);
                } else {
                    umma_commit_warp(bar(C::kOFinal + 0));
                }
                ok = wait_bounded_warp(bar(C::kPFull + 1), ph, wd, ROLE_MMA, SITE_P_FULL);
                if (!ok) break;
                tc_fence_after();
                issue_pv(tO1, tS1, v_addr, j > 0);
                umma_commit_warp(bar(C::kKVEmpty + iv % S));
                if (more) {
                    issue_qk(tS1, sQ + TILE, k_addr);
                    umma_commit_warp(bar(C::kSFull + 1));
                    umma_commit_warp(bar(C::kKVEmpty + ik % S));
                } else {
                    umma_commit_warp(bar(C::kOFinal + 1));
                }
            }
            // Every product issued must finish before TMEM is released.
            umma_commit_warp(bar(C::kDrain));
            wait_bounded_warp(bar(C::kDrain), 0, wd_drain, ROLE_MMA, SITE_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- softmax warps
        regs_increase<kSoftmaxRegs>();
        const int t = warp >> 2;    // query tile
        const int wq = warp & 3;    // TMEM lane quadrant
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * D;
        const int row = q_row0 + t * kBM + wq * 32 + lane;
        const float sl2 = a.scale_log2;
        float m = -INFINITY;  // running max of scale*log2(e)*s (possibly stale)
        float l = 0.f;        // running sum of 2^(s*sl2 - m)
        bool ok = true;
        // MASK: this row's bit words (all ones for rows past mask_rows)
        const bool row_masked = MASK && row < a.mask_rows;
        const uint32_t* mrow = MASK ? a.mask + static_cast<int64_t>(b) * a.mask_sb + static_cast<int64_t>(row_masked ? row : 0) * a.mask_si
                                    : nullptr;
        TileCursor cur(occ, k_begin, k_end);
        int tile_next = n_tiles > 0 ? cur.next() : -1;   // key tile of the next iteration
        uint4 mw = make_uint4(~0u, ~0u, ~0u, ~0u);
        // (debug library) the four words of a key tile lie inside the mask's extent
        auto mask_ok = [&](int tile) {
            const int64_t w0 = static_cast<int64_t>(b) * a.mask_sb + static_cast<int64_t>(row) * a.mask_si + 4 * tile;
            return in_bounds(tile >= 0 && w0 >= 0 && w0 + 4 <= a.dbg_mask_words, a.status, ROLE_SOFTMAX, BND_MASK);
        };
        if (MASK && row_masked && n_tiles > 0 && mask_ok(tile_next))
            mw = __ldg(reinterpret_cast<const uint4*>(mrow) + tile_next);
        // offset used in the exponent: 0 while no key of the row has been seen
        auto m_off = [&](float mm) { return (MASK && mm == -INFINITY) ? 0.f : mm; };

        // max over 64 scores: eight 3-input max chains, then a small tree.
        auto max64 = [](const float* v) {
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
        };
        // P = 2^(s*sl2 - m_use) for 64 scores -> 32 bf16x2 TMEM columns at tP; returns sum P.
        auto exp_store = [&](const float* v, uint32_t tP, float m_use) {
            const float neg_m = -m_use;
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    ffma2_bc(x0, x1, v[32 * cc + 2 * i], v[32 * cc + 2 * i + 1], sl2, neg_m);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    if (i & 1) fadd2_acc(b0, b1, p0, p1);
                    else fadd2_acc(a0, a1, p0, p1);
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tP + cc * 16, pk);
            }
            return (a0 + a1) + (b0 + b1);
        };

        for (int j = 0; j < n_tiles; ++j) {
            ok = wait_bounded(bar(C::kSFull + t), static_cast<uint32_t>(j) & 1u, wd, ROLE_SOFTMAX, SITE_S_FULL);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();

            // S row in two halves; the second lands while the first is processed.
            uint32_t sr[4][32];
            tmem_ld32(tS + 0, sr[0]);
            tmem_ld32(tS + 32, sr[1]);
            tmem_ld_wait_dep(sr[0]);
            reg_dep(sr[1]);
            tmem_ld32(tS + 64, sr[2]);
            tmem_ld32(tS + 96, sr[3]);
            const int tile = tile_next;
            tile_next = j + 1 < n_tiles ? cur.next() : -1;
            const int valid = a.kv_len - tile * kBN;   // >= 1
            uint4 mcur = mw;
            if (MASK && row_masked && j + 1 < n_tiles && mask_ok(tile_next))
                mw = __ldg(reinterpret_cast<const uint4*>(mrow) + tile_next);
            float s[128];
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
            if (valid < 64) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c >= valid) s[c] = -INFINITY;
            }
            if constexpr (MASK) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (!(((c < 32 ? mcur.x : mcur.y) >> (c & 31)) & 1u)) s[c] = -INFINITY;
            }
            if (j == 0) {
                const float mxA = max64(s);
                // First tile: no running max yet, so take the tile max first.
                tmem_ld_wait_dep(sr[2]);
                reg_dep(sr[3]);
#pragma unroll
                for (int c = 64; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
                if (valid < 128) {
#pragma unroll
                    for (int c = 64; c < 128; ++c)
                        if (c >= valid) s[c] = -INFINITY;
                }
                if constexpr (MASK) {
#pragma unroll
                    for (int c = 64; c < 128; ++c)
                        if (!(((c < 96 ? mcur.z : mcur.w) >> (c & 31)) & 1u)) s[c] = -INFINITY;
                }
                m = fmaxf(mxA, max64(s + 64)) * sl2;
                l = exp_store(s, tS, m_off(m)) + exp_store(s + 64, tS + 32, m_off(m));
            } else {
                // Exponents with the running max m, no tile max: if the tile's row
                // sum stays <= 2^39 then every P <= 2^39, which bf16 P and the fp32
                // O / l accumulators hold exactly as well as P <= 1.  Rows whose sum
                // exceeds it (their max grew by more than ~32 in log2 units) take
                // the slow path: tile max, O rescale, P recomputed.
                float lA = exp_store(s, tS, m_off(m));
                tmem_ld_wait_dep(sr[2]);
                reg_dep(sr[3]);
#pragma unroll
                for (int c = 64; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
                if (valid < 128) {
#pragma unroll
                    for (int c = 64; c < 128; ++c)
                        if (c >= valid) s[c] = -INFINITY;
                }
                if constexpr (MASK) {
#pragma unroll
                    for (int c = 64; c < 128; ++c)
                        if (!(((c < 96 ? mcur.z : mcur.w) >> (c & 31)) & 1u)) s[c] = -INFINITY;
                }
                float lB = exp_store(s + 64, tS + 32, m_off(m));
                // also true for inf / NaN; MASK: a row with no key seen yet (m = -inf)
                // always takes the slow path, which sets m from this tile's max
                const bool need = !(lA + lB <= kSumLimit) || (MASK && m == -INFINITY);
                bool slow = __any_sync(0xffffffffu, need);
                float m_new = m;
                if (slow) {
                    const float m_tile = fmaxf(max64(s), max64(s + 64)) * sl2;
                    m_new = need ? fmaxf(m_tile, m) : m;
                    // MASK: rows that still have no allowed key keep m = -inf;
                    // when no row of the warp moves, its O and P stand as they are
                    if constexpr (MASK) slow = __any_sync(0xffffffffu, m_new != m);
                }
                if (slow) {
                    // O holds PV(j-1) already (S(j) was committed after it).
                    tmem_st_wait();
                    const float alpha = (MASK && m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
                    l *= alpha;
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait_dep(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + cc * 32, o);
                    }
                    m = m_new;
                    lA = exp_store(s, tS, m_off(m));
                    lB = exp_store(s + 64, tS + 32, m_off(m));
                }
                l += lA + lB;
            }
            tmem_st_wait();
            tc_fence_before();
            if (!(warp == 0 && inject(a, FAULT_SKIP_P_ARRIVE, j))) mbar_arrive(bar(C::kPFull + t));
        }

        // ---------------------------------------------------------------- epilogue
        if (ok && n_tiles > 0) {
            ok = wait_bounded(bar(C::kOFinal + t), 0, wd, ROLE_SOFTMAX, SITE_O_FINAL);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok) {
            static_assert(!(ACCUM && OUT_BF16), "accumulation keeps O in fp32");
            const bool in_range = row < a.Nq;
            const int64_t lse_idx = (static_cast<int64_t>(b) * a.H + h) * a.Nq + row;
            const bool any_key = n_tiles > 0 && (!MASK || l > 0.f);
            const float lse_new = any_key ? (m + log2f(l)) * kLn2 : -INFINITY;
            // out = c_prev * O_prev + c_new * O_tmem
            float c_new = any_key ? 1.f / l : 0.f;
            float c_prev = 0.f;
            float lse_out = lse_new;
            if constexpr (ACCUM) {
                // Merge with the pass already in (out, lse): the same combine as
                // dit_attn_lse_merge, for two partials.
                const float lse_prev =
                    (in_range && in_bounds(lse_idx >= 0 && lse_idx < static_cast<int64_t>(a.B) * a.H * a.Nq, a.status,
                                           ROLE_SOFTMAX, BND_LSE))
                        ? a.lse[lse_idx]
                        : -INFINITY;
                const float mx = fmaxf(lse_prev, lse_new);
                if (mx == -INFINITY) {
                    c_new = 0.f;
                    lse_out = -INFINITY;
                } else {
                    const float wp = expf(lse_prev - mx);
                    const float wn = expf(lse_new - mx);
                    const float inv = 1.f / (wp + wn);
                    c_prev = wp * inv;
                    c_new = n_tiles > 0 ? wn * inv / l : 0.f;
                    lse_out = mx + logf(wp + wn);
                }
            }
            // Each 32-column chunk goes through this warp's 4 KB of the Q_t buffer
            // (idle since QK_t(last) completed, which S_t(last) signalled): a
            // thread writes its row, then the warp stores four rows per
            // instruction as whole 128-byte lines instead of 32 scattered pieces.
            // Rows sit 128 bytes apart with the 16-byte groups XOR-swizzled by
            // the row, so both phases are free of bank conflicts.
            float4* stg = reinterpret_cast<float4*>(smem + t * TILE + wq * 4096);
            const int k4 = lane & 7;        // 16-byte group this lane moves in the store phase
            const int r_sub = lane >> 3;    // row within each group of four
            float* const out_f = static_cast<float*>(a.out);
            uint16_t* const out_h = static_cast<uint16_t*>(a.out);
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
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
                    float4 val = stg[r * 8 + (k4 ^ (r & 7))];
                    const float cp = ACCUM ? __shfl_sync(0xffffffffu, c_prev, r) : 0.f;
                    const int grow = q_row0 + t * kBM + wq * 32 + r;
                    if (PIECE && grow < a.Nq) {
                        // a piece's fp32 partial, row-major [256][D] in its workspace slot
                        const int64_t wi = (static_cast<int64_t>(blockIdx.x) * (2 * kBM) + (grow - q_row0)) * D + cc * 32 + 4 * k4;
                        if (in_bounds(wi >= 0 && wi + 4 <= static_cast<int64_t>(a.n_split_ctas) * (2 * kBM) * D, a.status,
                                      ROLE_SOFTMAX, BND_WS))
                            *reinterpret_cast<float4*>(a.ws_o + wi) = val;
                    } else if (grow < a.Nq) {
                        const int64_t off = static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(grow) * a.o_sn +
                                            static_cast<int64_t>(h) * a.o_sh + cc * 32 + 4 * k4;
                        if (!in_bounds(off >= 0 && off + 4 <= a.dbg_o_elems, a.status, ROLE_SOFTMAX, BND_OUT)) continue;
                        if constexpr (OUT_BF16) {
                            *reinterpret_cast<uint2*>(out_h + off) =
                                make_uint2(pack_bf16x2(val.x, val.y), pack_bf16x2(val.z, val.w));
                        } else {
                            float4* dst = reinterpret_cast<float4*>(out_f + off);
                            if (ACCUM && cp > 0.f) {
                                const float4 pv = *dst;
                                val.x = fmaf(cp, pv.x, val.x);
                                val.y = fmaf(cp, pv.y, val.y);
                                val.z = fmaf(cp, pv.z, val.z);
                                val.w = fmaf(cp, pv.w, val.w);
                            }
                            *dst = val;
                        }
                    }
                }
                __syncwarp();
            }
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

template <int D, bool BF16, bool ACCUM, bool MASK = false>
cudaError_t launch_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& args,
                        int B, cudaStream_t stream) {
    auto kern = attn_fwd_kernel<D, BF16, ACCUM, MASK>;
    const int smem = Cfg<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(args.n_qblk, args.H, B);
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, args);
    e = cudaGetLastError();
    if (e != cudaSuccess || ACCUM || args.n_split_ctas == 0) return e;
    // The split items' pieces: a programmatic dependent launch, so that its
    // CTAs take SMs as the last whole items drain instead of after the grid.
    auto piece = attn_fwd_kernel<D, BF16, false, MASK, true>;
    e = cudaFuncSetAttribute(piece, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(args.n_split_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, piece, tq, tk, tv, args);
}

// Combine the split pieces: per (split item, row) the f normalised partials
// (O_p, LSE_p) give O = sum_p w_p O_p, LSE = M + ln sum_p e^(LSE_p - M), with
// w_p = e^(LSE_p - M) / sum_q e^(LSE_q - M) and M = max_p LSE_p.  A piece whose
// range holds no key the row may attend (general mask) has LSE_p = -inf and
// weight 0; a row with none in any piece gets O = 0, LSE = -inf.  D/4 lanes per
// row, one float4 of O each: coalesced reads of the row-major partials and of
// the output row.
template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(256) attn_tail_merge_kernel(const AttnArgs a) {
    constexpr int LPR = D / 4;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t unit = g / LPR;                     // (split item, row)
    const int c4 = static_cast<int>(g % LPR);
    const int f = a.split_f;
    if (unit >= static_cast<int64_t>(a.n_split_ctas / f) * (2 * kBM)) return;
    const int it = static_cast<int>(unit / (2 * kBM));
    const int r = static_cast<int>(unit % (2 * kBM));
    const int item = a.split_first + it;
    const int qblk = item % a.n_qblk;
    const int h = (item / a.n_qblk) % a.H;
    const int b = item / a.n_qblk / a.H;
    const int grow = qblk * (2 * kBM) + r;
    if (grow >= a.Nq) return;
    const int64_t piece0 = static_cast<int64_t>(it) * f;
    // (debug library) the item, its pieces' partials and the output lie in bounds
    const int64_t n_ws_rows = static_cast<int64_t>(a.n_split_ctas) * (2 * kBM);
    if (!in_bounds(h < a.H && b < a.B && f >= 1 && f <= kMaxSplit && (piece0 + f) * (2 * kBM) <= n_ws_rows, a.status,
                   0, BND_WS))
        return;
    float lp[kMaxSplit];
    float mx = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMaxSplit; ++p) {
        lp[p] = p < f ? a.ws_lse[(piece0 + p) * (2 * kBM) + r] : -INFINITY;
        mx = fmaxf(mx, lp[p]);
    }
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // A masked row may have no allowed key in some pieces (LSE -inf, weight 0)
    // or in all of them (O = 0, LSE = -inf).
#pragma unroll
    for (int p = 0; p < kMaxSplit; ++p) {
        if (p < f && mx != -INFINITY) {
            const float w = expf(lp[p] - mx);
            wsum += w;
            const float4 o = __ldcs(reinterpret_cast<const float4*>(a.ws_o + ((piece0 + p) * (2 * kBM) + r) * D) + c4);
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
        }
    }
    const float inv = mx != -INFINITY ? 1.f / wsum : 0.f;
    const int64_t off = static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(grow) * a.o_sn +
                        static_cast<int64_t>(h) * a.o_sh + 4 * c4;
    if (!in_bounds(off >= 0 && off + 4 <= a.dbg_o_elems, a.status, 0, BND_OUT)) return;
    if constexpr (OUT_BF16) {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + off) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (c4 == 0) a.lse[(static_cast<int64_t>(b) * a.H + h) * a.Nq + grow] = mx != -INFINITY ? mx + logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_attn_tail_merge(const AttnArgs& args, int D, bool out_bf16, cudaStream_t stream) {
    if (args.n_split_ctas == 0) return cudaSuccess;
    const int64_t threads = static_cast<int64_t>(args.n_split_ctas / args.split_f) * (2 * kBM) * (D / 4);
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    if (D == 128) {
        if (out_bf16) attn_tail_merge_kernel<128, true><<<blocks, 256, 0, stream>>>(args);
        else attn_tail_merge_kernel<128, false><<<blocks, 256, 0, stream>>>(args);
    } else {
        if (out_bf16) attn_tail_merge_kernel<64, true><<<blocks, 256, 0, stream>>>(args);
        else attn_tail_merge_kernel<64, false><<<blocks, 256, 0, stream>>>(args);
    }
    return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnArgs& args, int B, int D, bool out_bf16, bool accumulate, cudaStream_t stream) {
    if (args.mask != nullptr) {
        if (accumulate) return cudaErrorInvalidValue;
        if (D == 128) return out_bf16 ? launch_impl<128, true, false, true>(tq, tk, tv, args, B, stream)
                                      : launch_impl<128, false, false, true>(tq, tk, tv, args, B, stream);
        return out_bf16 ? launch_impl<64, true, false, true>(tq, tk, tv, args, B, stream)
                        : launch_impl<64, false, false, true>(tq, tk, tv, args, B, stream);
    }
    if (accumulate) {
        if (out_bf16) return cudaErrorInvalidValue;
        return D == 128 ? launch_impl<128, false, true>(tq, tk, tv, args, B, stream)
                        : launch_impl<64, false, true>(tq, tk, tv, args, B, stream);
    }
    if (D == 128) return out_bf16 ? launch_impl<128, true, false>(tq, tk, tv, args, B, stream)
                                  : launch_impl<128, false, false>(tq, tk, tv, args, B, stream);
    return out_bf16 ? launch_impl<64, true, false>(tq, tk, tv, args, B, stream)
                    : launch_impl<64, false, false>(tq, tk, tv, args, B, stream);
}

}  // namespace dit

