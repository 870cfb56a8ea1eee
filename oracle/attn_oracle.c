/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for dense bidirectional
 * multi-head self-attention that also returns the per-row log-sum-exp.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; it exists so that tests, the smoke check and the timed CPU
 * baseline can compare the CUDA library against an independent definition.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (one (b, h) head, a caller-chosen list of query rows i):
 *
 *     J      = { j : 0 <= j < key_valid_len, allow[b,i,j] }  (allow optional)
 *     s_ij   = scale * sum_d q[b,i,h,d] * k[b,j,h,d]       (fp64)
 *     m_i    = max_{j in J} s_ij
 *     l_i    = sum_{j in J} exp(s_ij - m_i)
 *     O[i,:] = sum_{j in J} exp(s_ij - m_i) * v[b,j,h,:] / l_i
 *     LSE_i  = m_i + ln(l_i)
 *
 * Sources:
 *   - "Scaling Video Generation Across NVL72 rack with TensorRT-LLM",
 *     section "The Scaling Challenge in Video Generation": every step runs
 *     dense, unmasked, bidirectional self-attention over the full N x N block.
 *   - same page, "Attention2D Parallelism", paragraph "Local Attention": the
 *     inner backend returns the output [B,S,H,D] and an LSE [B,H,S] that
 *     records the softmax normaliser of that pass.
 *   - "8 卡怎么分 token：LTX-2 序列并行的 all2all 到底搬了什么", section
 *     "数据流拆解", paragraph "构造 padding mask": a key-only mask of shape
 *     (1,1,T) marks valid keys with 1 and pad keys with 0, broadcast over
 *     batch and query rows; pad query rows still attend every valid key.
 *   - "CUDA IPC Ulysses：在 H100 上重叠 Attention 通信", section "基线与瓶颈":
 *     V may be a strided view of a fused QKV projection, so every operand is
 *     addressed through explicit (b, n, h) element strides, d contiguous.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - LSE is the natural log of sum_j exp(scale * q.k), i.e. it includes the
 *     scale; this is the reading under which partial passes merge exactly.
 *   - A row with no valid key (key_valid_len == 0) gets O = 0, LSE = -inf, so
 *     that an empty key chunk has weight zero in a merge.
 *   - Masked keys are the tail j >= key_valid_len (pads are appended at the end
 *     of the sequence and cut again after the gather).
 *   - A general (B, T, T) mask (same page, same paragraph: a user mask is
 *     expanded over the pad rows and columns) enters as `allow`, one byte per
 *     (b, i, j), 1 = may attend; a row whose J is empty gets O = 0, LSE = -inf
 *     (where a plain softmax would produce NaN).
 *
 * Inputs are bf16 bit patterns; each converts exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bits -> the exact value as float (bf16 is the top half of an fp32). */
static float bf16_bits_to_float(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * One head (b, h), a list of n_rows query rows.
 *
 * q, k, v          : base pointers to bf16 bit patterns.
 * q_s, k_s, v_s    : element strides {b, n, h}; d is contiguous.
 * allow            : NULL, or bytes with allow[b*allow_sb + i*allow_si + j] != 0
 *                    when query i may attend key j (j < key_valid_len).
 * o_out            : n_rows x D doubles, row r is query rows[r].
 * lse_out          : n_rows doubles.
 * Returns 0, or -1 when an argument is out of range, -2 on allocation failure.
 */
int oracle_attn_head_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int64_t *q_s, const int64_t *k_s, const int64_t *v_s,
                          int Nq, int Nkv, int D, int key_valid_len, double scale,
                          int b, int h, const int32_t *rows, int n_rows,
                          double *o_out, double *lse_out, int n_threads,
                          const uint8_t *allow, int64_t allow_sb, int64_t allow_si) {
    if (D <= 0 || Nq < 0 || Nkv < 0 || key_valid_len < 0 || key_valid_len > Nkv || n_rows < 0)
        return -1;
    for (int r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= Nq) return -1;

    const int nj = key_valid_len;
    if (nj == 0) {
        for (int r = 0; r < n_rows; ++r) {
            for (int d = 0; d < D; ++d) o_out[(int64_t)r * D + d] = 0.0;
            lse_out[r] = -INFINITY;
        }
        return 0;
    }

    /* The valid keys and values of this head, as exact floats. */
    float *kh = (float *)malloc(sizeof(float) * (size_t)nj * (size_t)D);
    float *vh = (float *)malloc(sizeof(float) * (size_t)nj * (size_t)D);
    if (!kh || !vh) { free(kh); free(vh); return -2; }
    for (int j = 0; j < nj; ++j) {
        const uint16_t *kr = k + (int64_t)b * k_s[0] + (int64_t)j * k_s[1] + (int64_t)h * k_s[2];
        const uint16_t *vr = v + (int64_t)b * v_s[0] + (int64_t)j * v_s[1] + (int64_t)h * v_s[2];
        for (int d = 0; d < D; ++d) {
            kh[(int64_t)j * D + d] = bf16_bits_to_float(kr[d]);
            vh[(int64_t)j * D + d] = bf16_bits_to_float(vr[d]);
        }
    }

    int err = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)nj);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd || !acc) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int r = 0; r < n_rows; ++r) {
                const int i = rows[r];
                const uint16_t *qr = q + (int64_t)b * q_s[0] + (int64_t)i * q_s[1] + (int64_t)h * q_s[2];
                for (int d = 0; d < D; ++d) qd[d] = (double)bf16_bits_to_float(qr[d]);

                /* pass 1: scores of the allowed keys and their maximum */
                const uint8_t *al = allow ? allow + (int64_t)b * allow_sb + (int64_t)i * allow_si : NULL;
                double m = -INFINITY;
                for (int j = 0; j < nj; ++j) {
                    if (al && !al[j]) { s[j] = -INFINITY; continue; }
                    const float *kj = kh + (int64_t)j * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qd[d] * (double)kj[d];
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                if (m == -INFINITY) {          /* no allowed key */
                    for (int d = 0; d < D; ++d) o_out[(int64_t)r * D + d] = 0.0;
                    lse_out[r] = -INFINITY;
                    continue;
                }
                /* pass 2: normaliser and weighted sum of values */
                double l = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int j = 0; j < nj; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const double p = exp(s[j] - m);
                    const float *vj = vh + (int64_t)j * D;
                    l += p;
                    for (int d = 0; d < D; ++d) acc[d] += p * (double)vj[d];
                }
                for (int d = 0; d < D; ++d) o_out[(int64_t)r * D + d] = acc[d] / l;
                lse_out[r] = m + log(l);
            }
        }
        free(s);
        free(qd);
        free(acc);
    }
    free(kh);
    free(vh);
    return err;
}

/* Threads an OpenMP parallel region actually gets (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
