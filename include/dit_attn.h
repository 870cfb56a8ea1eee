/*
 * dit_attn.h -- C ABI of libditattn.so: dense bidirectional long-sequence
 * attention for DiT video denoising on one NVIDIA GB300 (sm_103a).
 *
 * Entry points, all asynchronous on a caller-supplied CUDA stream:
 *
 *   dit_attn_fwd           softmax(scale * Q K^T) V plus the per-row
 *                          log-sum-exp, Q/K/V read through arbitrary
 *                          (b, n, h) strides, key-only padding mask.
 *   dit_attn_fwd_ws        the same with a workspace that balances the
 *                          grid's last partial wave.
 *   dit_attn_fwd_masked    the same with a general (B, Nq, Nkv) bit mask
 *                          (dit_attn_fwd_masked_noalloc: its scratch inside
 *                          the library instead of a caller workspace).
 *   dit_attn_fwd_accumulate  one more key chunk folded into a running
 *                          (O, LSE) pair.
 *   dit_attn_lse_merge     exact combine of (O, LSE) partials computed over
 *                          disjoint key chunks.
 *   dit_qkv_to_head_major  split of a fused [B, N, 3, H, D] projection
 *                          buffer into three head-major [B, H, N, D] tensors.
 *   dit_qkv_norm_rope_to_head_major  the same split with Q/K RMSNorm and
 *                          rotary embedding fused in (V copied).
 *   dit_qkv_cast_fp8       one-pass scaled bf16 -> E4M3 cast of that stacked
 *                          buffer, and dit_attn_fwd_fp8 (dit_attn_fwd_fp8_ws
 *                          with the balancing workspace), the attention that
 *                          reads its output in place.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   allocates no memory, copies nothing between host and device and keeps no
 *   per-call state; per-device caches hold kernel attributes, the SM count
 *   and the device addresses of the library's own globals.
 * - Every buffer a call reads or writes must be memory of the current device
 *   (cudaMalloc'd, from a memory pool, mapped with the virtual-memory calls,
 *   or managed memory), and `stream` must belong to the current device.  A
 *   host pointer (pageable or pinned), another device's memory or another
 *   device's stream returns DIT_ERR_INVALID_ARG with nothing enqueued.
 * - Strides are in ELEMENTS, not bytes.
 * - Argument, shape, stride and alignment checks run on the host before any
 *   launch.  A failed check returns a non-zero status and enqueues nothing.
 * - DIT_ERR_CUDA means a CUDA call failed while enqueueing; the CUDA error is
 *   left for the caller to query (cudaGetLastError / cudaPeekAtLastError).
 * - Calls are reentrant.  Input buffers must stay valid until the stream has
 *   executed the call; outputs are valid once the stream has passed it.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).
 * - Every spin-wait inside the kernels is bounded (about two seconds).  A wait
 *   that runs out records DIT_ERR_TIMEOUT in a device status word, the kernel
 *   winds down without faulting, and dit_check_watchdog() reports it.
 */
#ifndef DIT_ATTN_H
#define DIT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *dit_stream_t; /* same type as cudaStream_t */

typedef enum {
    DIT_OK = 0,
    DIT_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, ... */
    DIT_ERR_UNSUPPORTED = 2, /* a legal request outside what is built (e.g. D) */
    DIT_ERR_ALIGNMENT = 3,   /* a pointer or stride breaks the 16-byte rules  */
    DIT_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed           */
    DIT_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait ran out (watchdog)   */
    DIT_ERR_BOUNDS = 6       /* an in-kernel bounds check failed (reported by
                                the debug library only, dit_attn_debug.h)     */
} dit_status_t;

typedef enum { DIT_BF16 = 0, DIT_F32 = 1 } dit_dtype_t;

/* Element strides of a [B, N, H, D] view. */
typedef struct {
    int64_t b, n, h, d;
} dit_strides4_t;

typedef struct {
    dit_strides4_t q, k, v, o;
} dit_attn_strides_t;

/*
 * dit_attn_fwd -- O = softmax(scale * Q K^T) V and LSE = ln sum_j exp(scale q.k_j)
 *
 * Defined by "Scaling Video Generation Across NVL72 rack with TensorRT-LLM":
 * section "The Scaling Challenge in Video Generation" (dense, unmasked,
 * bidirectional attention over the full N x N block, every denoising step)
 * and section "Attention2D Parallelism", paragraph "Local Attention" (the
 * inner backend returns the output [B,S,H,D] and an LSE [B,H,S] recording the
 * softmax normaliser, so partial passes over key chunks merge exactly).  The
 * key mask follows "8 卡怎么分 token：LTX-2 序列并行的 all2all 到底搬了什么",
 * "数据流拆解" / "构造 padding mask": a key-only mask, pads at the tail, pad
 * query rows attend all valid keys.  Strided Q/K/V follow "CUDA IPC
 * Ulysses：在 H100 上重叠 Attention 通信", "基线与瓶颈": V of a fused QKV
 * projection is read as a strided view with no packing copy.
 *
 * q      bf16, element (b, i, h, d) at q + b*s.q.b + i*s.q.n + h*s.q.h + d, i < Nq
 * k, v   bf16, same form with s.k / s.v, j < Nkv
 * strides  s.q.d, s.k.d, s.v.d, s.o.d must be 1.  The b, n, h strides of q/k/v
 *          must be positive multiples of 8 elements (16 bytes); those of o
 *          multiples of 16 bytes of out_dtype.  Base pointers 16-byte aligned.
 * B, Nq, Nkv, H  >= 0 (a zero size is a no-op); D in {64, 128}.  B and H at
 *          most 65,535 and B * H * ceil(Nq / 256) below 2^31, else
 *          DIT_ERR_UNSUPPORTED (the same limits hold for every attention call).
 * key_valid_len  keys j >= key_valid_len are masked out; 0 <= key_valid_len <= Nkv.
 *          Masked keys are never read, so pad rows may hold any bits.
 *          key_valid_len == 0 yields O = 0 and LSE = -inf for every row.
 * scale  finite and > 0 (typically 1/sqrt(D)).
 * out    O, out_dtype DIT_F32 or DIT_BF16, addressed with s.o ([B, Nq, H, D]).
 * lse    fp32 [B, H, Nq] contiguous, natural log, includes `scale`.
 * Returns DIT_OK once enqueued.
 */
dit_status_t dit_attn_fwd(const void *q, const void *k, const void *v,
                          const dit_attn_strides_t *strides,
                          int B, int Nq, int Nkv, int H, int D,
                          int key_valid_len, float scale,
                          void *out, dit_dtype_t out_dtype, float *lse,
                          dit_stream_t stream);

/*
 * dit_attn_fwd_ws -- dit_attn_fwd with a caller workspace that balances the
 * last wave of the grid.
 *
 * The GPU runs one CTA per (b, h, 256-row query block) work item.  When the
 * item count is not a multiple of the SM count, the last partial wave leaves
 * most SMs idle for a whole item's time.  With a workspace, each item of that
 * partial wave is split into f contiguous key ranges (f = SMs / leftover items,
 * at most 8, at least 2 behind whole waves; each range at least 16 key tiles of
 * 128; no split for a single partial wave that fills more than half the SMs).  A second kernel,
 * launched as a programmatic dependent launch, runs the ranges so that its
 * CTAs fill the SMs as the last whole items drain; a third combines each
 * item's normalised partial (O, LSE) pairs with the exact merge of "Scaling
 * Video Generation Across NVL72 rack with TensorRT-LLM", "Ring Attention",
 * paragraph "Online-softmax merge" (the pages have no counterpart for the
 * scheduling itself; the combine is that merge).
 *
 * Results: items that are not split are bit-identical to dit_attn_fwd's.
 * Split items differ by the bf16 rounding of the probabilities P (each range
 * rounds them against its own running maximum) -- a few 1e-4 at most at 8k
 * keys, both within the same tolerance of the exact result -- and their LSE by
 * fp32 rounding.  The call is deterministic (fixed merge order).
 *
 * workspace  NULL (then exactly dit_attn_fwd), or device memory of at least
 *        dit_attn_fwd_workspace_bytes(B, Nq, H, D, key_valid_len) bytes, 16-byte
 *        aligned, owned by the caller and not used by anything else until the
 *        stream has passed the call.  A non-NULL workspace smaller than that
 *        is DIT_ERR_INVALID_ARG (nothing is enqueued).
 * Other arguments and results as dit_attn_fwd.  Enqueues one kernel, or three
 * when a split applies; work queued behind the call on the same stream sees
 * all of its outputs.
 */
dit_status_t dit_attn_fwd_ws(const void *q, const void *k, const void *v,
                             const dit_attn_strides_t *strides,
                             int B, int Nq, int Nkv, int H, int D,
                             int key_valid_len, float scale,
                             void *out, dit_dtype_t out_dtype, float *lse,
                             void *workspace, size_t workspace_bytes,
                             dit_stream_t stream);

/*
 * dit_attn_fwd_workspace_bytes -- workspace bytes that dit_attn_fwd_ws (and
 * dit_attn_fwd_fp8_ws, D = 128) use for this shape on the CURRENT device (the
 * plan depends on its SM count): the split pieces' fp32 partial O (256 x D per
 * piece) and LSE (256 per piece).  0 when no split helps (the item count is a
 * multiple of the SM count, the keys are too few, or there is nothing to
 * compute); D outside {64, 128} gives 0.  Host only, one cached device query.
 * The size holds for the device current at query time (and any device with
 * the same SM count): a call on a device with more SMs can plan a larger
 * split and then refuses a workspace sized elsewhere (DIT_ERR_INVALID_ARG).
 */
size_t dit_attn_fwd_workspace_bytes(int B, int Nq, int H, int D, int key_valid_len);

/*
 * dit_attn_fwd_masked -- dit_attn_fwd with a general attention mask.
 *
 * Defined by "8 卡怎么分 token：LTX-2 序列并行的 all2all 到底搬了什么",
 * "数据流拆解", paragraph "构造 padding mask": when the caller passes a
 * (B, T, T) mask it is expanded over the pad rows and columns -- pad keys are
 * masked and pad query rows may attend every valid key, since a row with every
 * key masked would make a plain softmax NaN.  Cross-attention (Nq != Nkv, e.g.
 * video queries over a short text or audio K/V) is the same call with any
 * Nq, Nkv (and dit_attn_fwd without a mask).
 *
 * mask   device array of 32-bit words: query i may attend key j when bit (j & 31)
 *        of mask[b*mask_batch_stride + i*mask_row_stride + (j >> 5)] is 1.  Read
 *        only for rows i < mask_rows and keys j < key_valid_len; the mask is
 *        shared by all heads.  Rows i >= mask_rows attend every key
 *        j < key_valid_len (the pad-row rule); keys j >= key_valid_len are always
 *        masked.  The kernel reads 4 * ceil(key_valid_len / 128) words of each
 *        masked row, so mask_row_stride must be at least that; strides are
 *        multiples of 4 words, mask_batch_stride >= 0 (0 shares one mask across
 *        the batch), base 16-byte aligned, and the array must hold
 *        (B-1)*mask_batch_stride + mask_rows*mask_row_stride words.
 * mask_rows  0 <= mask_rows <= Nq; 0 makes the call dit_attn_fwd (mask unread).
 * A row left with no allowed key gets O = 0 and LSE = -inf (weight 0 in a
 * merge) instead of NaN.
 * workspace  NULL, or device memory of at least dit_attn_masked_workspace_bytes
 *        (16-byte aligned) owned by the caller and not used by anything else
 *        until the stream has passed the call: a pre-pass records which
 *        128-key tiles each 256-row query block attends at all, and the
 *        attention then loads and multiplies only those (block-local masks
 *        skip most tiles).  NULL processes every tile (same results).
 *        With dit_attn_masked_split_workspace_bytes or more, the space past
 *        the occupancy map (which starts the workspace, rounded up to 256
 *        bytes) also holds the tail split of dit_attn_fwd_ws: the grid's last
 *        partial wave runs as key-range pieces, merged exactly.  A smaller
 *        workspace is not an error; the call then runs unsplit.
 * Other arguments as dit_attn_fwd.
 */
dit_status_t dit_attn_fwd_masked(const void *q, const void *k, const void *v,
                                 const dit_attn_strides_t *strides,
                                 int B, int Nq, int Nkv, int H, int D,
                                 int key_valid_len,
                                 const uint32_t *mask, int64_t mask_batch_stride,
                                 int64_t mask_row_stride, int mask_rows,
                                 float scale, void *out, dit_dtype_t out_dtype, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 dit_stream_t stream);

/*
 * dit_attn_fwd_masked_noalloc -- dit_attn_fwd_masked with its tile-occupancy
 * scratch taken from a fixed array inside the library instead of a
 * caller-provided workspace.  The pages have no counterpart: it serves callers
 * that cannot allocate device memory at call time, e.g. an engine that hands
 * all free device memory to its own pool at start-up, or a plain C host
 * program with no device allocator of its own.
 *
 * Same arguments and results as dit_attn_fwd_masked without the workspace.
 * Limits: one scratch array (65,536 words) per device and process, so
 *   - DIT_ERR_UNSUPPORTED when dit_attn_masked_workspace_bytes(B, Nq,
 *     key_valid_len) exceeds 262,144 bytes (checked before anything is enqueued);
 *   - calls on one device must be ordered (the same stream, or streams joined
 *     by events): two in flight at once would share the array.
 * Allocates nothing.  The array's device address is looked up with
 * cudaGetSymbolAddress on the first call in each CUDA context of a device
 * and cached for that context; after cudaDeviceReset (a new primary context,
 * where the array has a new address) the next call looks it up again.
 */
dit_status_t dit_attn_fwd_masked_noalloc(const void *q, const void *k, const void *v,
                                         const dit_attn_strides_t *strides,
                                         int B, int Nq, int Nkv, int H, int D,
                                         int key_valid_len,
                                         const uint32_t *mask, int64_t mask_batch_stride,
                                         int64_t mask_row_stride, int mask_rows,
                                         float scale, void *out, dit_dtype_t out_dtype, float *lse,
                                         dit_stream_t stream);

/*
 * dit_attn_masked_split_workspace_bytes -- bytes of `workspace` that let
 * dit_attn_fwd_masked both skip empty key tiles and split the grid's last
 * partial wave (the occupancy map rounded up to 256 bytes, then the split's
 * partials, dit_attn_fwd_workspace_bytes of them); the bare occupancy map's
 * size when no split helps.  Like dit_attn_fwd_workspace_bytes, the size holds
 * for the device current at query time (its SM count sets the split).  0 when
 * there is nothing to compute or D is not 64 or 128.  Host only.
 */
size_t dit_attn_masked_split_workspace_bytes(int B, int Nq, int H, int D, int key_valid_len);

/*
 * dit_attn_masked_workspace_bytes -- bytes of `workspace` that let
 * dit_attn_fwd_masked skip key tiles the mask leaves empty: one bit per
 * (batch, 256-row query block, 128-key tile), written by a pre-pass on the
 * same stream.  0 when there is nothing to compute.  Host only, no CUDA call.
 */
size_t dit_attn_masked_workspace_bytes(int B, int Nq, int key_valid_len);

/*
 * dit_attn_fwd_accumulate -- one more key chunk folded into a running result.
 *
 * The streaming form of the merge: "Scaling Video Generation Across NVL72 rack
 * with TensorRT-LLM", "Ring Attention", paragraph "Online-softmax merge" (each
 * ring step's partial output and LSE are merged into the running output in
 * fp32, block by block, until it equals one global pass) and the "Difference
 * from Ring" table of "Attention2D Parallelism" (streaming merge after every
 * step, in place on the local rank).  Computes this call's (O_c, LSE_c) exactly
 * as dit_attn_fwd and replaces the fp32 (out, lse) already in memory by
 *   M = max(LSE, LSE_c),  w = exp(LSE - M),  w_c = exp(LSE_c - M),
 *   out = (w out + w_c O_c) / (w + w_c),  lse = M + ln(w + w_c),
 * so a sequence of calls over disjoint key chunks ends at the single-pass
 * result.  Start from lse = -inf everywhere: rows whose lse is -inf take this
 * call's result and their old `out` is not read (it may hold any bits).
 * Arguments as dit_attn_fwd; `out` is fp32 only and is read and written.
 */
dit_status_t dit_attn_fwd_accumulate(const void *q, const void *k, const void *v,
                                     const dit_attn_strides_t *strides,
                                     int B, int Nq, int Nkv, int H, int D,
                                     int key_valid_len, float scale,
                                     float *out, float *lse, dit_stream_t stream);

/*
 * dit_attn_lse_merge -- combine n_chunks partial (O_k, LSE_k) computed for the
 * same queries over disjoint key spans into the single-pass result.
 *
 * Defined by "Scaling Video Generation Across NVL72 rack with TensorRT-LLM",
 * "Attention2D Parallelism", paragraph "Merge phase" (one batched combine of
 * the col_size received (output, LSE) pairs) and "Ring Attention", paragraph
 * "Online-softmax merge" (fp32 merge until the result equals one global pass):
 *   M = max_k LSE_k,  w_k = exp(LSE_k - M),  O = sum_k w_k O_k / sum_k w_k,
 *   LSE = M + ln sum_k w_k.  Chunks with LSE_k = -inf get weight 0 (their O_k
 *   is not read); a row whose chunks are all -inf yields O = 0, LSE = -inf.
 *
 * o_parts    fp32, chunk k, row (b, i, h), channel d at
 *              o_parts + k*o_chunk_stride + ((b*Nq + i)*H + h)*o_row_stride + d.
 *            o_row_stride = D with o_chunk_stride = B*Nq*H*D is the chunk-major
 *            layout [n, B, Nq, H, D]; o_row_stride = n*D with o_chunk_stride = D
 *            interleaves the chunks per row ([B, Nq, H, n, D]), which the kernel
 *            reads as one contiguous stream (dit_attn_fwd can write either
 *            through its output strides).  Strides multiples of 4, chunks must
 *            not overlap.
 * lse_parts  fp32, chunk k at lse_parts + k*lse_chunk_stride, [B, H, Nq] contiguous.
 * n_chunks in [1, 64]; D in {64, 128}.
 * out        [B, Nq, H, D] contiguous, out_dtype DIT_F32 or DIT_BF16.
 * lse_out    fp32 [B, H, Nq] contiguous, may be NULL.
 * All pointers 16-byte aligned.  Output must not overlap any input.
 */
dit_status_t dit_attn_lse_merge(const float *o_parts, int64_t o_chunk_stride, int64_t o_row_stride,
                                const float *lse_parts, int64_t lse_chunk_stride,
                                int n_chunks, int B, int Nq, int H, int D,
                                void *out, dit_dtype_t out_dtype, float *lse_out,
                                dit_stream_t stream);

/*
 * dit_qkv_to_head_major -- bit-exact split/permute of a fused QKV projection.
 *
 * Defined by "Scaling Video Generation Across NVL72 rack with TensorRT-LLM",
 * "Ulysses Parallelism" (the swap from sequence-major [B,S,H,D] to the
 * head-sharded layout before attention; paragraph "Fused vs. unfused QKV
 * all-to-all": the stacked buffer is [B, S, 3, H, D]) and "CUDA IPC
 * Ulysses：在 H100 上重叠 Attention 通信", "Strided Copy Engine scatter"
 * (the source pitch comes straight from the input stride; head and channel
 * must be contiguous within each sequence row).
 *
 * qkv     bf16; element (b, n, t, h, d) at qkv + b*stride_b + n*stride_n +
 *         (t*H + h)*D + d, t = 0 (q), 1 (k), 2 (v).  stride_b, stride_n
 *         multiples of 8 elements; base 16-byte aligned; D a multiple of 8.
 * q_out, k_out, v_out  each [B, H, N, D] contiguous bf16, 16-byte aligned:
 *         out_t[((b*H + h)*N + n)*D + d] = qkv(b, n, t, h, d).
 */
dit_status_t dit_qkv_to_head_major(const void *qkv, int64_t stride_b, int64_t stride_n,
                                   int B, int N, int H, int D,
                                   void *q_out, void *k_out, void *v_out,
                                   dit_stream_t stream);

/*
 * dit_qkv_norm_rope_to_head_major -- dit_qkv_to_head_major with the per-head
 * normalisation and rotary embedding of Q and K fused into the same pass.
 *
 * Defined by "CUDA IPC Ulysses：在 H100 上重叠 Attention 通信", "基线与瓶颈"
 * and "模型调度": after the fused QKV projection, Q and K get normalisation and
 * RoPE, V does not.  The pages give neither formula; this call implements
 * RMSNorm over the head dimension followed by the RoFormer rotation of
 * consecutive channel pairs:
 *   y_d = x_d / sqrt(mean_d(x_d^2) + eps) * w_d                (w = q_weight / k_weight)
 *   (y_2i, y_2i+1) -> (y_2i c - y_2i+1 s, y_2i s + y_2i+1 c),  c = rope_cos[n*D/2 + i],
 *                                                              s = rope_sin[n*D/2 + i],
 * computed in fp32 and rounded to bf16 once.
 *
 * qkv, stride_b, stride_n, B, N, H, q_out, k_out, v_out  as dit_qkv_to_head_major.
 * D          64 or 128.
 * q_weight, k_weight  fp32 [D] device arrays, 16-byte aligned; NULL skips the
 *            normalisation of that tensor.
 * eps        finite, >= 0.
 * rope_cos, rope_sin  fp32 [N, D/2] contiguous device arrays, 16-byte aligned,
 *            one row per sequence position (any 1-D or multi-axis angle table);
 *            both NULL skips the rotation, one NULL is DIT_ERR_INVALID_ARG.
 * v_out receives V bit-exactly.
 */
dit_status_t dit_qkv_norm_rope_to_head_major(const void *qkv, int64_t stride_b, int64_t stride_n,
                                             int B, int N, int H, int D,
                                             const float *q_weight, const float *k_weight, float eps,
                                             const float *rope_cos, const float *rope_sin,
                                             void *q_out, void *k_out, void *v_out,
                                             dit_stream_t stream);

/*
 * dit_qkv_cast_fp8 -- one pass over a stacked bf16 QKV buffer that writes it
 * as FP8 E4M3 in the same stacked layout, q, k and v each scaled first.
 *
 * Defined by "Scaling Video Generation Across NVL72 rack with TensorRT-LLM",
 * "Ulysses Parallelism", paragraph "Fused vs. unfused QKV all-to-all": the
 * stacked QKV buffer is one contiguous allocation, so a single FP8 cast covers
 * all three tensors, and its output goes to the attention kernel without an
 * intermediate copy.  The pages do not say how the scales are chosen; they are
 * the caller's (per-tensor factors, e.g. 448 / amax).
 *
 * qkv     bf16, element (b, n, t, h, d) at qkv + b*stride_b + n*stride_n +
 *         (t*H + h)*D + d; stride_b, stride_n multiples of 8 elements; base
 *         16-byte aligned; D a multiple of 16.
 * out     E4M3 bytes, [B, N, 3, H, D] contiguous, 16-byte aligned:
 *         out(b, n, t, h, d) = e4m3(qkv(b, n, t, h, d) * scale_t), the product
 *         rounded to fp32, then rounded to nearest even E4M3, magnitudes above
 *         448 saturating to +-448 (NaN stays NaN).
 * scale_q, scale_k, scale_v  finite and > 0.
 * DIT_ERR_UNSUPPORTED when 3*H*D > 2^28 or B*N*3*H*D / 16 >= 2^32.
 */
dit_status_t dit_qkv_cast_fp8(const void *qkv, int64_t stride_b, int64_t stride_n,
                              int B, int N, int H, int D,
                              float scale_q, float scale_k, float scale_v,
                              void *out, dit_stream_t stream);

/*
 * dit_attn_fwd_fp8 -- dit_attn_fwd on E4M3 inputs.
 *
 * The FP8 attention kernel that the cast above feeds ("Scaling Video
 * Generation Across NVL72 rack with TensorRT-LLM", "Ulysses Parallelism",
 * "Fused vs. unfused QKV all-to-all").  q, k, v hold E4M3 codes q8, k8, v8
 * standing for Q = q8 * descale_q, K = k8 * descale_k, V = v8 * descale_v
 * (descale = 1 / the cast's scale); the result is dit_attn_fwd's O and LSE
 * for those Q, K, V.  The probabilities P enter the P.V product as E4M3 (their
 * largest value per row ~2^7 to 2^8.75), so O carries a relative error of
 * about 2^-4 / sqrt(number of keys that matter) on top of the inputs'
 * quantisation; LSE is computed from fp32 P.
 *
 * Arguments as dit_attn_fwd, except:
 * q, k, v   E4M3 bytes; strides in elements (= bytes), the b, n, h strides
 *           positive multiples of 16.  For the output of dit_qkv_cast_fp8:
 *           q = out, k = out + H*D, v = out + 2*H*D, strides
 *           (b, n, h, d) = (N*3*H*D, 3*H*D, D, 1).
 * D         128 only (DIT_ERR_UNSUPPORTED otherwise).
 * descale_q, descale_k, descale_v  finite and > 0; scale * descale_q *
 *           descale_k * log2(e) must lie in (1e-30, 1e30).
 */
dit_status_t dit_attn_fwd_fp8(const void *q, const void *k, const void *v,
                              const dit_attn_strides_t *strides,
                              int B, int Nq, int Nkv, int H, int D,
                              int key_valid_len, float scale,
                              float descale_q, float descale_k, float descale_v,
                              void *out, dit_dtype_t out_dtype, float *lse,
                              dit_stream_t stream);

/*
 * dit_attn_fwd_fp8_ws -- dit_attn_fwd_fp8 with the grid-balancing workspace of
 * dit_attn_fwd_ws: the work items of the last partial wave run as key-range
 * pieces (a programmatic dependent launch) beside the last whole items, and
 * their normalised partial (O, LSE) pairs are combined with the exact merge of
 * "Scaling Video Generation Across NVL72 rack with TensorRT-LLM", "Ring
 * Attention", paragraph "Online-softmax merge".  The pages have no counterpart
 * for the scheduling.
 *
 * workspace  NULL (then exactly dit_attn_fwd_fp8), or device memory of at least
 *        dit_attn_fwd_workspace_bytes(B, Nq, H, D, key_valid_len) bytes (the
 *        same plan as the bf16 call), 16-byte aligned, owned by the caller and
 *        not used by anything else until the stream has passed the call.  A
 *        smaller non-zero size is DIT_ERR_INVALID_ARG.
 * Other arguments and results as dit_attn_fwd_fp8.  Items that are not split
 * are bit-identical to dit_attn_fwd_fp8's; split items differ by the E4M3
 * rounding of P (each piece rounds against its own running max).
 */
dit_status_t dit_attn_fwd_fp8_ws(const void *q, const void *k, const void *v,
                                 const dit_attn_strides_t *strides,
                                 int B, int Nq, int Nkv, int H, int D,
                                 int key_valid_len, float scale,
                                 float descale_q, float descale_k, float descale_v,
                                 void *out, dit_dtype_t out_dtype, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 dit_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *dit_status_string(dit_status_t s);

/*
 * dit_check_watchdog -- synchronise `stream`, read and clear the device
 * status word of the current device.  Returns DIT_OK, DIT_ERR_TIMEOUT (a
 * bounded in-kernel wait ran out; `info`, if non-NULL, receives four words:
 * code, block index, warp role, wait site), DIT_ERR_BOUNDS (debug library
 * only: an in-kernel bounds check failed and the access was skipped; `info`
 * then holds the check's site) or DIT_ERR_CUDA.  Only the first report since
 * the last read is kept.
 */
dit_status_t dit_check_watchdog(dit_stream_t stream, uint32_t info[4]);

/*
 * dit_watchdog_selftest -- library self-test of the failure path; the pages
 * have no counterpart.  Launches one CTA whose bounded wait can never be
 * satisfied, so it gives up after `limit_us` microseconds (1,000 to 2,000,000),
 * records DIT_ERR_TIMEOUT in the device status word (wait site 99) and exits
 * normally; the CUDA context stays usable.  Read the result with
 * dit_check_watchdog().  Returns DIT_OK once enqueued.
 */
dit_status_t dit_watchdog_selftest(uint32_t limit_us, dit_stream_t stream);

/* Library version, (major << 16) | minor. */
uint32_t dit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_H */
