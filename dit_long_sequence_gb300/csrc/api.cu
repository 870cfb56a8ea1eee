// api.cu -- the extern "C" entry points of libditattn.so (include/dit_attn.h).
//
// Host side only: argument / stride / alignment validation before anything is
// enqueued, TMA descriptor encoding for the strided Q/K/V views, the device
// status word read by dit_check_watchdog(), and the kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "dit_attn.h"
#ifdef DIT_DEBUG
#include "dit_attn_debug.h"
#endif
#include "internal.h"
#include "split_plan.h"

namespace dit {

// Device status word: [0] code, [1] block, [2] warp role, [3] wait site.
__device__ unsigned int g_status_word[4];

// Occupancy scratch of dit_attn_fwd_masked_noalloc: one per device, for
// callers that cannot provide a workspace.  65,536 words cover every
// configuration measured here (LTX-2 576 words, Wan 11,248, the 147,456-token
// ring workload 20,736).
constexpr int64_t kNoAllocOccWords = 65536;
static __device__ __align__(256) uint32_t g_noalloc_occ[kNoAllocOccWords];

namespace {

constexpr unsigned long long kWatchdogNs = 2000000000ull;  // 2 s per bounded wait
constexpr int kMaxDevices = 64;

#ifdef DIT_DEBUG
// Debug library: the fault, wait limit and O-extent shrink the next calls use
// (dit_debug_configure).
std::atomic<uint32_t> g_dbg_fault{0};
std::atomic<int> g_dbg_block{0};
std::atomic<int> g_dbg_index{0};
std::atomic<unsigned long long> g_dbg_limit_ns{0};
std::atomic<int64_t> g_dbg_out_shrink{0};
#endif

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The current context's unique id (cuCtxGetCurrent + cuCtxGetId through the
// driver entry points), 0 if there is none.  A device's primary context is
// replaced by cudaDeviceReset; module globals then live at new addresses, so
// cached symbol addresses are keyed on this id and looked up again for a new
// context.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id + 1;   // never 0 for a live context
}

// Per-device cache of a module global's device address, valid for one context.
struct SymbolCache {
    std::mutex mu;
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};

struct DeviceCache {
    SymbolCache status;
    SymbolCache noalloc_occ;
    std::atomic<int> sm_count{0};
};
DeviceCache g_dev[kMaxDevices];

// Device address of `symbol` in the current context of the current device:
// looked up with cudaGetSymbolAddress once per context (the first lookup also
// makes the runtime set up the device's primary context if it has not yet).
template <typename T>
T* symbol_address(SymbolCache& c, const void* symbol) {
    unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(c.mu);
    if (id != 0 && c.addr != nullptr && c.ctx_id == id) return static_cast<T*>(c.addr);
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, symbol) != cudaSuccess) return nullptr;
    c.addr = addr;
    c.ctx_id = current_context_id();   // 0 (never matches) if it cannot be read
    return static_cast<T*>(addr);
}

unsigned int* status_word(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    return symbol_address<unsigned int>(g_dev[dev].status, g_status_word);
}

// Device address of the no-alloc occupancy scratch in the current context.
uint32_t* noalloc_scratch(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    return symbol_address<uint32_t>(g_dev[dev].noalloc_occ, g_noalloc_occ);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every buffer a kernel will touch must be memory of the current device (or
// managed memory), and the stream one of the current device's: a host address
// or another device's memory handed to a TMA copy or a store is refused here,
// before anything is enqueued, instead of faulting the GPU.  Null entries are
// skipped (the caller has already decided which buffers are required).
dit_status_t check_placement(std::initializer_list<const void*> ptrs, dit_stream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DIT_ERR_CUDA;
    for (const void* p : ptrs) {
        if (p == nullptr) continue;
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return DIT_ERR_INVALID_ARG;
        }
        const bool here = (at.type == cudaMemoryTypeDevice && at.device == dev) || at.type == cudaMemoryTypeManaged;
        if (!here) return DIT_ERR_INVALID_ARG;
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread) {
        int sdev = -1;
        if (cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
            (void)cudaGetLastError();
            return DIT_ERR_INVALID_ARG;
        }
        if (sdev != dev) return DIT_ERR_INVALID_ARG;
    }
    return DIT_OK;
}

// A [B, N, H, D] view as a 4-D TMA map (D, N, H, B) with 128-byte swizzle and
// a box of one swizzle column (64 bf16 or 128 E4M3 channels) by 128 rows.
// Rows n >= n_rows are outside the map and read as zeros.
dit_status_t encode_view(CUtensorMap* map, const void* base, const dit_strides4_t& s, int B, int n_rows, int H,
                         int D, bool fp8 = false) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return DIT_ERR_CUDA;
    const cuuint64_t eb = fp8 ? 1 : 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(n_rows > 0 ? n_rows : 1),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.n) * eb, static_cast<cuuint64_t>(s.h) * eb,
                                   static_cast<cuuint64_t>(s.b) * eb};
    const cuuint32_t box[4] = {fp8 ? 128u : 64u, 128, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DIT_OK : DIT_ERR_INVALID_ARG;
}

// b, n, h strides of a TMA operand: positive, 16-byte multiples, < 2^39 elements.
dit_status_t check_tma_strides(const dit_strides4_t& s, bool fp8 = false) {
    if (s.d != 1) return DIT_ERR_UNSUPPORTED;
    const int64_t st[3] = {s.b, s.n, s.h};
    for (int64_t x : st) {
        if (x <= 0 || x >= (int64_t(1) << 39)) return DIT_ERR_INVALID_ARG;
        if (x % (fp8 ? 16 : 8) != 0) return DIT_ERR_ALIGNMENT;
    }
    return DIT_OK;
}

}  // namespace

int device_sm_count(int dev) {
    if (dev >= 0 && dev < kMaxDevices) {
        int c = g_dev[dev].sm_count.load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 148;
    if (dev >= 0 && dev < kMaxDevices) g_dev[dev].sm_count.store(c, std::memory_order_relaxed);
    return c;
}

}  // namespace dit

using namespace dit;

namespace {

struct MaskSpec {
    const uint32_t* bits;
    int64_t batch_stride, row_stride;   // in 32-bit words
    int rows;
    uint32_t* occ;                      // occupancy map (workspace) or nullptr
};

int64_t occ_words_of(int key_valid_len) { return ((key_valid_len + 127) / 128 + 31) / 32; }
int64_t occ_bytes_of(int B, int Nq, int key_valid_len) {
    return static_cast<int64_t>(B) * ((Nq + 255) / 256) * occ_words_of(key_valid_len) * 4;
}
// A masked call's workspace: the occupancy map, then (from this offset) the
// tail split's partials.
int64_t occ_region_of(int B, int Nq, int key_valid_len) { return (occ_bytes_of(B, Nq, key_valid_len) + 255) / 256 * 256; }

// fp8: E4M3 inputs (D = 128 only), descales[3] = (q, k, v); otherwise bf16.
// mask: the general bit mask of dit_attn_fwd_masked (bf16 only).
dit_status_t attn_fwd_common(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides, int B,
                             int Nq, int Nkv, int H, int D, int key_valid_len, float scale, void* out,
                             dit_dtype_t out_dtype, float* lse, bool accumulate, dit_stream_t stream,
                             const float* descales = nullptr, const MaskSpec* mask = nullptr,
                             void* workspace = nullptr, size_t workspace_bytes = 0, bool split_optional = false) {
    const bool fp8 = descales != nullptr;
    if (strides == nullptr) return DIT_ERR_INVALID_ARG;
    if (B < 0 || Nq < 0 || Nkv < 0 || H < 0) return DIT_ERR_INVALID_ARG;
    if (key_valid_len < 0 || key_valid_len > Nkv) return DIT_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return DIT_ERR_INVALID_ARG;
    if (out_dtype != DIT_BF16 && out_dtype != DIT_F32) return DIT_ERR_INVALID_ARG;
    double sl2 = static_cast<double>(scale) * 1.4426950408889634;
    if (fp8) {
        for (int i = 0; i < 3; ++i)
            if (!(descales[i] > 0.f) || !std::isfinite(descales[i])) return DIT_ERR_INVALID_ARG;
        sl2 *= static_cast<double>(descales[0]) * static_cast<double>(descales[1]);
        if (!(sl2 > 1e-30 && sl2 < 1e30)) return DIT_ERR_INVALID_ARG;
        if (D != 128) return DIT_ERR_UNSUPPORTED;
    }
    if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return DIT_ERR_UNSUPPORTED;
    // The work items (b, h, 256-row block) are counted in 32-bit ints on the
    // device (grid order, the split boundary).
    if (static_cast<int64_t>(B) * H * ((static_cast<int64_t>(Nq) + 255) / 256) > 0x7fffffffLL)
        return DIT_ERR_UNSUPPORTED;
    if (B == 0 || Nq == 0 || H == 0) return DIT_OK;
    if (out == nullptr || lse == nullptr) return DIT_ERR_INVALID_ARG;
    const bool any_keys = key_valid_len > 0;
    if (any_keys && (q == nullptr || k == nullptr || v == nullptr)) return DIT_ERR_INVALID_ARG;

    // Output: d contiguous; b, n, h strides non-negative 16-byte multiples.
    const dit_strides4_t& so = strides->o;
    if (so.d != 1) return DIT_ERR_UNSUPPORTED;
    const int64_t o_align = out_dtype == DIT_F32 ? 4 : 8;
    if (so.b < 0 || so.n < 0 || so.h < 0) return DIT_ERR_INVALID_ARG;
    if (so.b % o_align || so.n % o_align || so.h % o_align) return DIT_ERR_ALIGNMENT;
    if (!aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return DIT_ERR_ALIGNMENT;

    CUtensorMap tq, tk, tv;
    std::memset(&tq, 0, sizeof tq);
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    if (any_keys) {
        dit_status_t st;
        if ((st = check_tma_strides(strides->q, fp8)) != DIT_OK) return st;
        if ((st = check_tma_strides(strides->k, fp8)) != DIT_OK) return st;
        if ((st = check_tma_strides(strides->v, fp8)) != DIT_OK) return st;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return DIT_ERR_ALIGNMENT;
        if ((st = encode_view(&tq, q, strides->q, B, Nq, H, D, fp8)) != DIT_OK) return st;
        if ((st = encode_view(&tk, k, strides->k, B, key_valid_len, H, D, fp8)) != DIT_OK) return st;
        if ((st = encode_view(&tv, v, strides->v, B, key_valid_len, H, D, fp8)) != DIT_OK) return st;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DIT_ERR_CUDA;
    {
        const bool with_mask = mask != nullptr && mask->rows > 0 && any_keys;
        const dit_status_t st =
            check_placement({any_keys ? q : nullptr, any_keys ? k : nullptr, any_keys ? v : nullptr, out, lse,
                             workspace, with_mask ? mask->bits : nullptr, with_mask ? mask->occ : nullptr},
                            stream);
        if (st != DIT_OK) return st;
    }
    // Work items (b, h, 256-row block) of the 1-D bf16 grid, and the tail split
    // when the caller gave a workspace for it (plain, unmasked, overwrite only).
    const int64_t items = static_cast<int64_t>(B) * H * ((static_cast<int64_t>(Nq) + 255) / 256);
    SplitPlan split{items, 1, 0};
    if (workspace != nullptr && !accumulate && any_keys) {
        split = plan_tail_split(items, (key_valid_len + 127) / 128, device_sm_count(dev));
        if (workspace_bytes < static_cast<size_t>(split_workspace_bytes(split, D))) {
            if (!split_optional) return DIT_ERR_INVALID_ARG;
            split = SplitPlan{items, 1, 0};   // a masked call's workspace without room for the split
        }
        if (!aligned16(workspace)) return DIT_ERR_ALIGNMENT;
    }
    AttnArgs a;
    a.status = status_word(dev);
    a.timeout_ns = kWatchdogNs;
    if (a.status == nullptr) return DIT_ERR_CUDA;   // checked before anything is enqueued
    a.Nq = Nq;
    a.H = H;
    a.kv_len = key_valid_len;
    a.n_kv_tiles = (key_valid_len + 127) / 128;
    a.scale_log2 = static_cast<float>(sl2);
    a.o_scale = fp8 ? descales[2] : 1.f;
    a.mask = nullptr;
    a.mask_sb = a.mask_si = 0;
    a.mask_rows = 0;
    a.occ = nullptr;
    a.occ_words = 0;
    if (mask != nullptr && mask->rows > 0 && any_keys) {
        a.mask = mask->bits;
        a.mask_sb = mask->batch_stride;
        a.mask_si = mask->row_stride;
        a.mask_rows = mask->rows;
        if (mask->occ != nullptr) {
            OccArgs o;
            o.mask = mask->bits;
            o.mask_sb = mask->batch_stride;
            o.mask_si = mask->row_stride;
            o.mask_rows = mask->rows;
            o.B = B;
            o.Nq = Nq;
            o.kv_len = key_valid_len;
            o.n_kv_tiles = a.n_kv_tiles;
            o.row_blocks = (Nq + 255) / 256;
            o.occ_words = static_cast<int>(occ_words_of(key_valid_len));
            o.occ = mask->occ;
            cudaError_t e = launch_mask_occupancy(o, reinterpret_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) return DIT_ERR_CUDA;
            a.occ = mask->occ;
            a.occ_words = o.occ_words;
        }
    }
    a.out = out;
    a.o_sb = so.b;
    a.o_sn = so.n;
    a.o_sh = so.h;
    a.lse = lse;
    a.n_qblk = static_cast<int>((static_cast<int64_t>(Nq) + 255) / 256);
    a.split_first = static_cast<int>(split.first);
    a.split_f = split.f;
    a.n_split_ctas = static_cast<int>(split.n_ctas);
    a.ws_o = split.n_ctas > 0 ? static_cast<float*>(workspace) : nullptr;
    a.ws_lse = split.n_ctas > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                          split.n_ctas * 256 * D * 4)
                                : nullptr;
    a.B = B;
    // extents of the debug library's bounds checks (unused by the product kernels)
    a.dbg_fault = FAULT_NONE;
    a.dbg_fault_cta = 0;
    a.dbg_fault_index = 0;
    a.dbg_o_elems = static_cast<int64_t>(B - 1) * so.b + static_cast<int64_t>(Nq - 1) * so.n +
                    static_cast<int64_t>(H - 1) * so.h + D;
    a.dbg_mask_words = a.mask == nullptr ? 0
                                         : static_cast<int64_t>(B - 1) * a.mask_sb +
                                               static_cast<int64_t>(a.mask_rows - 1) * a.mask_si + 4 * a.n_kv_tiles;
#ifdef DIT_DEBUG
    a.dbg_fault = g_dbg_fault.load();
    a.dbg_fault_cta = g_dbg_block.load();
    a.dbg_fault_index = g_dbg_index.load();
    if (g_dbg_limit_ns.load() != 0) a.timeout_ns = g_dbg_limit_ns.load();
    a.dbg_o_elems -= g_dbg_out_shrink.load();
#endif
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = fp8 ? launch_attn_fwd_fp8(tq, tk, tv, a, B, out_dtype == DIT_BF16, cs)
                        : launch_attn_fwd(tq, tk, tv, a, B, D, out_dtype == DIT_BF16, accumulate, cs);
    if (e == cudaSuccess) e = launch_attn_tail_merge(a, D, out_dtype == DIT_BF16, cs);
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

}  // namespace

extern "C" {

dit_status_t dit_attn_fwd(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides, int B,
                          int Nq, int Nkv, int H, int D, int key_valid_len, float scale, void* out,
                          dit_dtype_t out_dtype, float* lse, dit_stream_t stream) {
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, out_dtype, lse, false,
                           stream);
}

size_t dit_attn_fwd_workspace_bytes(int B, int Nq, int H, int D, int key_valid_len) {
    if (B <= 0 || Nq <= 0 || H <= 0 || key_valid_len <= 0 || (D != 64 && D != 128)) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int64_t items = static_cast<int64_t>(B) * H * ((static_cast<int64_t>(Nq) + 255) / 256);
    const SplitPlan p = plan_tail_split(items, (key_valid_len + 127) / 128, device_sm_count(dev));
    return static_cast<size_t>(split_workspace_bytes(p, D));
}

dit_status_t dit_attn_fwd_ws(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides, int B,
                             int Nq, int Nkv, int H, int D, int key_valid_len, float scale, void* out,
                             dit_dtype_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                             dit_stream_t stream) {
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, out_dtype, lse, false,
                           stream, nullptr, nullptr, workspace, workspace_bytes);
}

dit_status_t dit_attn_fwd_accumulate(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides,
                                     int B, int Nq, int Nkv, int H, int D, int key_valid_len, float scale, float* out,
                                     float* lse, dit_stream_t stream) {
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, DIT_F32, lse, true,
                           stream);
}

size_t dit_attn_masked_workspace_bytes(int B, int Nq, int key_valid_len) {
    if (B <= 0 || Nq <= 0 || key_valid_len <= 0) return 0;
    return static_cast<size_t>(occ_bytes_of(B, Nq, key_valid_len));
}

dit_status_t dit_attn_fwd_masked(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides,
                                 int B, int Nq, int Nkv, int H, int D, int key_valid_len, const uint32_t* mask,
                                 int64_t mask_batch_stride, int64_t mask_row_stride, int mask_rows, float scale,
                                 void* out, dit_dtype_t out_dtype, float* lse, void* workspace,
                                 size_t workspace_bytes, dit_stream_t stream) {
    if (mask_rows < 0 || mask_rows > Nq) return DIT_ERR_INVALID_ARG;
    if (workspace != nullptr) {
        if (B > 0 && Nq > 0 && key_valid_len > 0 &&
            workspace_bytes < static_cast<size_t>(occ_bytes_of(B, Nq, key_valid_len)))
            return DIT_ERR_INVALID_ARG;
        if (!aligned16(workspace)) return DIT_ERR_ALIGNMENT;
    }
    if (mask_rows > 0) {
        if (mask == nullptr) return DIT_ERR_INVALID_ARG;
        const int64_t words_read = 4 * static_cast<int64_t>((key_valid_len + 127) / 128);
        if (mask_row_stride < words_read || mask_batch_stride < 0) return DIT_ERR_INVALID_ARG;
        if (mask_row_stride % 4 || mask_batch_stride % 4 || !aligned16(mask)) return DIT_ERR_ALIGNMENT;
    }
    const MaskSpec spec{mask, mask_batch_stride, mask_row_stride, mask_rows, static_cast<uint32_t*>(workspace)};
    // Beyond the occupancy map, room for the tail split's partials (if any) lets
    // the call split the grid's last partial wave as dit_attn_fwd_ws does.
    void* split_ws = nullptr;
    size_t split_bytes = 0;
    if (workspace != nullptr && B > 0 && Nq > 0 && key_valid_len > 0) {
        const int64_t region = occ_region_of(B, Nq, key_valid_len);
        if (workspace_bytes > static_cast<size_t>(region)) {
            split_ws = static_cast<uint8_t*>(workspace) + region;
            split_bytes = workspace_bytes - static_cast<size_t>(region);
        }
    }
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, out_dtype, lse, false,
                           stream, nullptr, &spec, split_ws, split_bytes, true);
}

size_t dit_attn_masked_split_workspace_bytes(int B, int Nq, int H, int D, int key_valid_len) {
    if (B <= 0 || Nq <= 0 || H <= 0 || key_valid_len <= 0 || (D != 64 && D != 128)) return 0;
    const size_t split = dit_attn_fwd_workspace_bytes(B, Nq, H, D, key_valid_len);
    if (split == 0) return static_cast<size_t>(occ_bytes_of(B, Nq, key_valid_len));
    return static_cast<size_t>(occ_region_of(B, Nq, key_valid_len)) + split;
}

dit_status_t dit_attn_fwd_masked_noalloc(const void* q, const void* k, const void* v,
                                         const dit_attn_strides_t* strides, int B, int Nq, int Nkv, int H, int D,
                                         int key_valid_len, const uint32_t* mask, int64_t mask_batch_stride,
                                         int64_t mask_row_stride, int mask_rows, float scale, void* out,
                                         dit_dtype_t out_dtype, float* lse, dit_stream_t stream) {
    const int64_t need = (B > 0 && Nq > 0 && key_valid_len > 0) ? occ_bytes_of(B, Nq, key_valid_len) : 0;
    if (need > kNoAllocOccWords * 4) return DIT_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DIT_ERR_CUDA;
    uint32_t* scratch = noalloc_scratch(dev);
    if (scratch == nullptr) return DIT_ERR_CUDA;
    // exactly the occupancy map's bytes: the fixed array never holds split partials
    return dit_attn_fwd_masked(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, mask, mask_batch_stride,
                               mask_row_stride, mask_rows, scale, out, out_dtype, lse, scratch,
                               static_cast<size_t>(need > 0 ? need : 16), stream);
}

dit_status_t dit_attn_fwd_fp8(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides,
                              int B, int Nq, int Nkv, int H, int D, int key_valid_len, float scale, float descale_q,
                              float descale_k, float descale_v, void* out, dit_dtype_t out_dtype, float* lse,
                              dit_stream_t stream) {
    const float descales[3] = {descale_q, descale_k, descale_v};
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, out_dtype, lse, false,
                           stream, descales);
}

dit_status_t dit_attn_fwd_fp8_ws(const void* q, const void* k, const void* v, const dit_attn_strides_t* strides,
                                 int B, int Nq, int Nkv, int H, int D, int key_valid_len, float scale,
                                 float descale_q, float descale_k, float descale_v, void* out, dit_dtype_t out_dtype,
                                 float* lse, void* workspace, size_t workspace_bytes, dit_stream_t stream) {
    const float descales[3] = {descale_q, descale_k, descale_v};
    return attn_fwd_common(q, k, v, strides, B, Nq, Nkv, H, D, key_valid_len, scale, out, out_dtype, lse, false,
                           stream, descales, nullptr, workspace, workspace_bytes);
}

dit_status_t dit_qkv_cast_fp8(const void* qkv, int64_t stride_b, int64_t stride_n, int B, int N, int H, int D,
                              float scale_q, float scale_k, float scale_v, void* out, dit_stream_t stream) {
    if (B < 0 || N < 0 || H < 0 || D < 0) return DIT_ERR_INVALID_ARG;
    const float sc[3] = {scale_q, scale_k, scale_v};
    for (float x : sc)
        if (!(x > 0.f) || !std::isfinite(x)) return DIT_ERR_INVALID_ARG;
    if (D % 16 != 0) return DIT_ERR_UNSUPPORTED;
    if (B == 0 || N == 0 || H == 0 || D == 0) return DIT_OK;
    if (qkv == nullptr || out == nullptr) return DIT_ERR_INVALID_ARG;
    const uint64_t hd = static_cast<uint64_t>(H) * static_cast<uint64_t>(D);
    const uint64_t chunks = 3 * hd / 16;
    if (3 * hd > (uint64_t(1) << 28) || static_cast<uint64_t>(B) * N * chunks >= (uint64_t(1) << 32))
        return DIT_ERR_UNSUPPORTED;
    if (stride_b < 0 || stride_n < 0) return DIT_ERR_INVALID_ARG;
    if (stride_b % 8 || stride_n % 8) return DIT_ERR_ALIGNMENT;
    if (!aligned16(qkv) || !aligned16(out)) return DIT_ERR_ALIGNMENT;
    if (const dit_status_t st = check_placement({qkv, out}, stream); st != DIT_OK) return st;
    CastArgs a;
    a.qkv = static_cast<const uint16_t*>(qkv);
    a.stride_b = stride_b;
    a.stride_n = stride_n;
    a.N = N;
    a.hd = static_cast<uint32_t>(hd);
    a.chunks_per_row = static_cast<uint32_t>(chunks);
    a.total_chunks = static_cast<uint64_t>(B) * N * chunks;
    for (int i = 0; i < 3; ++i) a.scale[i] = sc[i];
    a.out = static_cast<uint8_t*>(out);
    cudaError_t e = launch_qkv_cast_fp8(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

dit_status_t dit_attn_lse_merge(const float* o_parts, int64_t o_chunk_stride, int64_t o_row_stride,
                                const float* lse_parts, int64_t lse_chunk_stride, int n_chunks, int B, int Nq, int H,
                                int D, void* out, dit_dtype_t out_dtype, float* lse_out, dit_stream_t stream) {
    if (n_chunks < 1 || n_chunks > 64) return DIT_ERR_INVALID_ARG;
    if (B < 0 || Nq < 0 || H < 0) return DIT_ERR_INVALID_ARG;
    if (out_dtype != DIT_BF16 && out_dtype != DIT_F32) return DIT_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
    if (B == 0 || Nq == 0 || H == 0) return DIT_OK;
    if (o_parts == nullptr || lse_parts == nullptr || out == nullptr) return DIT_ERR_INVALID_ARG;
    const int64_t rows = static_cast<int64_t>(B) * Nq * H;
    if (o_row_stride < D || o_chunk_stride < 0 || lse_chunk_stride < 0) return DIT_ERR_INVALID_ARG;
    if (n_chunks > 1) {
        // chunks must not overlap: either chunk-major or interleaved within a row
        const bool chunk_major = o_chunk_stride >= (rows - 1) * o_row_stride + D;
        const bool interleaved = o_chunk_stride >= D && o_row_stride >= n_chunks * o_chunk_stride;
        if (!chunk_major && !interleaved) return DIT_ERR_INVALID_ARG;
        if (lse_chunk_stride < rows) return DIT_ERR_INVALID_ARG;
    }
    if (o_chunk_stride % 4 != 0 || o_row_stride % 4 != 0) return DIT_ERR_ALIGNMENT;
    if (!aligned16(o_parts) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse_out) & 3u))
        return DIT_ERR_ALIGNMENT;
    if (const dit_status_t st = check_placement({o_parts, lse_parts, out, lse_out}, stream); st != DIT_OK) return st;
    MergeArgs a;
    a.o_parts = o_parts;
    a.o_chunk_stride = o_chunk_stride;
    a.o_row_stride = o_row_stride;
    a.lse_parts = lse_parts;
    a.lse_chunk_stride = lse_chunk_stride;
    a.n_chunks = n_chunks;
    a.B = B;
    a.Nq = Nq;
    a.H = H;
    a.out = out;
    a.lse_out = lse_out;
    cudaError_t e = launch_lse_merge(a, D, out_dtype == DIT_BF16, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

dit_status_t dit_qkv_to_head_major(const void* qkv, int64_t stride_b, int64_t stride_n, int B, int N, int H, int D,
                                   void* q_out, void* k_out, void* v_out, dit_stream_t stream) {
    if (B < 0 || N < 0 || H < 0 || D < 0) return DIT_ERR_INVALID_ARG;
    if (D % 8 != 0) return DIT_ERR_UNSUPPORTED;
    if (B == 0 || N == 0 || H == 0 || D == 0) return DIT_OK;
    if (qkv == nullptr || q_out == nullptr || k_out == nullptr || v_out == nullptr) return DIT_ERR_INVALID_ARG;
    if (static_cast<int64_t>(3) * H * D > (int64_t(1) << 28)) return DIT_ERR_UNSUPPORTED;
    if (stride_b < 0 || stride_n < 0) return DIT_ERR_INVALID_ARG;
    if (stride_b % 8 || stride_n % 8) return DIT_ERR_ALIGNMENT;
    if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out)) return DIT_ERR_ALIGNMENT;
    if (const dit_status_t st = check_placement({qkv, q_out, k_out, v_out}, stream); st != DIT_OK) return st;
    LayoutArgs a;
    a.qkv = static_cast<const uint16_t*>(qkv);
    a.stride_b = stride_b;
    a.stride_n = stride_n;
    a.B = B;
    a.N = N;
    a.H = H;
    a.D = D;
    a.out[0] = static_cast<uint16_t*>(q_out);
    a.out[1] = static_cast<uint16_t*>(k_out);
    a.out[2] = static_cast<uint16_t*>(v_out);
    cudaError_t e = launch_qkv_to_head_major(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

dit_status_t dit_qkv_norm_rope_to_head_major(const void* qkv, int64_t stride_b, int64_t stride_n, int B, int N,
                                             int H, int D, const float* q_weight, const float* k_weight, float eps,
                                             const float* rope_cos, const float* rope_sin, void* q_out, void* k_out,
                                             void* v_out, dit_stream_t stream) {
    if (B < 0 || N < 0 || H < 0 || D < 0) return DIT_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return DIT_ERR_INVALID_ARG;
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return DIT_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
    if (B == 0 || N == 0 || H == 0) return DIT_OK;
    if (qkv == nullptr || q_out == nullptr || k_out == nullptr || v_out == nullptr) return DIT_ERR_INVALID_ARG;
    if (static_cast<int64_t>(3) * H * D > (int64_t(1) << 28)) return DIT_ERR_UNSUPPORTED;
    if (stride_b < 0 || stride_n < 0) return DIT_ERR_INVALID_ARG;
    if (stride_b % 8 || stride_n % 8) return DIT_ERR_ALIGNMENT;
    if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out)) return DIT_ERR_ALIGNMENT;
    if ((q_weight && !aligned16(q_weight)) || (k_weight && !aligned16(k_weight)) ||
        (rope_cos && (!aligned16(rope_cos) || !aligned16(rope_sin))))
        return DIT_ERR_ALIGNMENT;
    if (const dit_status_t st =
            check_placement({qkv, q_out, k_out, v_out, q_weight, k_weight, rope_cos, rope_sin}, stream);
        st != DIT_OK)
        return st;
    NormRopeArgs a;
    a.qkv = static_cast<const uint16_t*>(qkv);
    a.stride_b = stride_b;
    a.stride_n = stride_n;
    a.B = B;
    a.N = N;
    a.H = H;
    a.D = D;
    a.weight[0] = q_weight;
    a.weight[1] = k_weight;
    a.eps = eps;
    a.cos = rope_cos;
    a.sin = rope_sin;
    a.out[0] = static_cast<uint16_t*>(q_out);
    a.out[1] = static_cast<uint16_t*>(k_out);
    a.out[2] = static_cast<uint16_t*>(v_out);
    cudaError_t e = launch_qkv_norm_rope(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

const char* dit_status_string(dit_status_t s) {
    switch (s) {
        case DIT_OK: return "DIT_OK";
        case DIT_ERR_INVALID_ARG: return "DIT_ERR_INVALID_ARG: invalid argument";
        case DIT_ERR_UNSUPPORTED: return "DIT_ERR_UNSUPPORTED: request outside the built configurations";
        case DIT_ERR_ALIGNMENT: return "DIT_ERR_ALIGNMENT: pointer or stride breaks the 16-byte rules";
        case DIT_ERR_CUDA: return "DIT_ERR_CUDA: a CUDA call failed";
        case DIT_ERR_TIMEOUT: return "DIT_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case DIT_ERR_BOUNDS: return "DIT_ERR_BOUNDS: an in-kernel bounds check failed (debug library)";
    }
    return "unknown dit_status_t";
}

dit_status_t dit_watchdog_selftest(uint32_t limit_us, dit_stream_t stream) {
    if (limit_us < 1000 || limit_us > 2000000) return DIT_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DIT_ERR_CUDA;
    unsigned int* st = status_word(dev);
    if (st == nullptr) return DIT_ERR_CUDA;
    cudaError_t e = launch_watchdog_selftest(st, 1000ull * limit_us, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA;
}

dit_status_t dit_check_watchdog(dit_stream_t stream, uint32_t info[4]) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DIT_ERR_CUDA;
    unsigned int host[4] = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(host, g_status_word, sizeof host) != cudaSuccess) return DIT_ERR_CUDA;
    if (host[0] != 0) {
        const unsigned int zero[4] = {0, 0, 0, 0};
        if (cudaMemcpyToSymbol(g_status_word, zero, sizeof zero) != cudaSuccess) return DIT_ERR_CUDA;
    }
    if (info != nullptr)
        for (int i = 0; i < 4; ++i) info[i] = host[i];
    if (host[0] == 0) return DIT_OK;
    return host[0] == static_cast<unsigned int>(DIT_ERR_BOUNDS) ? DIT_ERR_BOUNDS : DIT_ERR_TIMEOUT;
}

uint32_t dit_version(void) { return (0u << 16) | 2u; }

#ifdef DIT_DEBUG
dit_status_t dit_debug_configure(uint32_t fault, int fault_block, int fault_index, uint32_t wait_limit_us,
                                 int64_t out_extent_shrink) {
    if (fault > FAULT_SKIP_P_ARRIVE || fault_block < 0 || fault_index < 0 || out_extent_shrink < 0)
        return DIT_ERR_INVALID_ARG;
    if (wait_limit_us != 0 && (wait_limit_us < 1000 || wait_limit_us > 2000000)) return DIT_ERR_INVALID_ARG;
    g_dbg_fault.store(fault);
    g_dbg_block.store(fault_block);
    g_dbg_index.store(fault_index);
    g_dbg_limit_ns.store(1000ull * wait_limit_us);
    g_dbg_out_shrink.store(out_extent_shrink);
    return DIT_OK;
}

uint32_t dit_debug_build(void) { return 1u; }
#endif

}  // extern "C"
