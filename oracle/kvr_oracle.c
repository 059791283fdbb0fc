/*
 * kvr_oracle.c -- fp64 CPU oracle for the precomputed-KV RAG hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * path under rag_precomputed_kv_gb300/csrc.
 *
 * Every function is the plain definition, in double precision, with no
 * blocking, fusion or reordering beyond what the definition states:
 *
 *   kvo_positions   -- target position of each retrieved span and the
 *                      per-token position / source maps.  CoinRAG blog,
 *                      section 2.3 (the Delta_i formula and the C_ctx
 *                      equation); TurboRAG blog, "Position ID" section
 *                      (reordered vs composite positions, Figure 5).
 *   kvo_rope_rows   -- RoPE rotation R(shift) of rows of a key / query.
 *                      CoinRAG blog section 2.3 (Rot(.; Delta_i)); TurboRAG
 *                      blog, "TurboRAG's two key observations" (RoPE only
 *                      depends on relative position) and "Position ID"
 *                      (re-apply RoPE at the new position).
 *   kvo_rope_rows_interleaved
 *                   -- the same rotation on adjacent pairs (x_2i, x_2i+1),
 *                      the other RoPE layout in use; the pages fix no layout.
 *   kvo_query_attention_units
 *                   -- query prefill over a stitched prefix: every query
 *                      token sees the whole prefix and the query tokens
 *                      before it.  CoinRAG blog section 2.3 (KV_CoinRAG =
 *                      C_ctx (+) KV_M(q; C_ctx)); TurboRAG blog, "Attention
 *                      Mask" (independent attention, Figure 4); SemPIC page
 *                      (inline tokens interleaved under a causal mask).
 *
 * Readings of points the pages leave open:
 *   - spans are half-open [start, end), length end - start;
 *   - the rotation applied to a cached span is delta = target - start, since
 *     the cached key already carries its chunk-local position start + t;
 *   - RoPE pairs element i with element i + D/2 (half-split), frequency
 *     theta^(-2i/D), x' = x cos(a) - y sin(a), y' = x sin(a) + y cos(a);
 *     the interleaved layout pairs elements 2i and 2i+1 at the same
 *     frequency theta^(-2i/D);
 *   - query tokens (and their keys) are rotated at P + t, P = prefix length;
 *   - attention scale defaults to 1/sqrt(D); masked keys get weight 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t src;   /* source id (chunk, system prompt entry or inline block) */
    int32_t start; /* first token of the span inside its source            */
    int32_t end;   /* one past the last token                               */
} kvo_span;

/* Number of threads the attention oracle uses. */
int kvo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Positions of the stitched prefix.
 *
 * Reordered positions (composite == 0): span i lands at
 *     target_i = first_pos + sum_{j<i} (end_j - start_j)
 * so the spans sit back to back in retrieval order, each in its in-document
 * order; token t of span i gets position target_i + (t - start_i) and is
 * rotated by delta_i = target_i - start_i.
 *
 * Composite positions (composite != 0): every span keeps its chunk-local ids
 * (position t, delta 0); the rows are still stitched back to back.
 *
 * Outputs (caller-allocated): target[n], delta[n] and, per stitched token in
 * stitched order, pos[P], src_id[P], src_tok[P].  Returns P (total stitched
 * tokens) or -1 on an invalid span (start < 0 or end < start).
 */
int64_t kvo_positions(int n, const kvo_span *spans, int64_t first_pos,
                      int composite, int64_t *target, int64_t *delta,
                      int32_t *pos, int32_t *src_id, int32_t *src_tok)
{
    int64_t next = first_pos; /* position the next reordered span starts at */
    int64_t row = 0;          /* stitched row index                          */
    for (int i = 0; i < n; ++i) {
        const kvo_span s = spans[i];
        if (s.start < 0 || s.end < s.start)
            return -1;
        target[i] = composite ? s.start : next;
        delta[i] = target[i] - s.start;
        for (int32_t t = s.start; t < s.end; ++t) {
            if (pos)
                pos[row] = (int32_t)(target[i] + (t - s.start));
            if (src_id)
                src_id[row] = s.src;
            if (src_tok)
                src_tok[row] = t;
            ++row;
        }
        next += (int64_t)(s.end - s.start);
    }
    return row;
}

/* RoPE frequency of pair i: theta^(-2i/D). */
static double inv_freq(double theta, int D, int i)
{
    return pow(theta, -2.0 * (double)i / (double)D);
}

/*
 * Rotate each row r of x (n_rows x D, row-major) by the positional shift
 * shift[r]: pair (x_i, x_{i+D/2}) turns by angle shift[r] * theta^(-2i/D).
 * out may alias x.
 */
void kvo_rope_rows(int64_t n_rows, int D, const double *x, const double *shift,
                   double theta, double *out)
{
    const int h = D / 2;
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int i = 0; i < h; ++i) {
            const double a = shift[r] * inv_freq(theta, D, i);
            const double c = cos(a), s = sin(a);
            const double x1 = x[r * D + i], x2 = x[r * D + i + h];
            out[r * D + i] = x1 * c - x2 * s;
            out[r * D + i + h] = x1 * s + x2 * c;
        }
    }
}

/*
 * Rotate each row r of x by shift[r] with the interleaved pairing: pair i is
 * (x_{2i}, x_{2i+1}) and turns by angle shift[r] * theta^(-2i/D).  out may
 * alias x.
 */
void kvo_rope_rows_interleaved(int64_t n_rows, int D, const double *x, const double *shift,
                               double theta, double *out)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        const double *xr = x + r * D;
        double *yr = out + r * D;
        for (int i = 0; i < D / 2; ++i) {
            const double ang = shift[r] * inv_freq(theta, D, i);
            const double cs = cos(ang), sn = sin(ang);
            const double ev = xr[2 * i], od = xr[2 * i + 1];
            yr[2 * i] = ev * cs - od * sn;
            yr[2 * i + 1] = ev * sn + od * cs;
        }
    }
}

/* One row through the rotation of the chosen layout. */
static void rope_row(int interleaved, int D, const double *x, double shift, double theta,
                     double *out)
{
    if (interleaved)
        kvo_rope_rows_interleaved(1, D, x, &shift, theta, out);
    else
        kvo_rope_rows(1, D, x, &shift, theta, out);
}

/*
 * Query prefill attention for n_units independent (request, layer, kv-head)
 * units that share the prefix length P and the query length Lq.
 *
 * Per unit u (arrays are unit-major, row-major inside):
 *   kc, vc : [P, D]      stitched prefix; kc already rotated to its positions
 *   q      : [Lq, G, D]  the G query heads that share this kv head, un-rotated
 *   kq, vq : [Lq, D]     the query tokens' own key / value, un-rotated
 *   o      : [Lq, G, D]  output
 *
 * Query token t sits at position P + t: its query and key are rotated by
 * P + t, its key/value row is appended after the prefix, and it attends to
 * the P prefix rows plus query rows 0..t:
 *     s_j = scale * <R(P+t) q_{t,g}, k_j>,  o = sum_j softmax(s)_j v_j
 * (softmax with the maximum subtracted).  scale <= 0 means 1/sqrt(D).
 * interleaved != 0 rotates with kvo_rope_rows_interleaved (kc must then be
 * rotated that way too).  Returns 0, or -1 if memory runs out.
 */
int kvo_query_attention_units(int64_t n_units, int64_t P, int64_t Lq, int G,
                              int D, double theta, int interleaved, double scale,
                              const double *kc, const double *vc,
                              const double *q, const double *kq,
                              const double *vq, double *o)
{
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)D);
    const int64_t N = P + Lq;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < n_units; ++u) {
        double *K = (double *)malloc(sizeof(double) * (size_t)(N * D));
        double *V = (double *)malloc(sizeof(double) * (size_t)(N * D));
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        double *sc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!K || !V || !qr || !sc) {
#pragma omp atomic write
            failed = 1;
            free(K); free(V); free(qr); free(sc);
            continue;
        }
        /* cache = prefix rows, then the query tokens' rotated keys / values */
        memcpy(K, kc + u * P * D, sizeof(double) * (size_t)(P * D));
        memcpy(V, vc + u * P * D, sizeof(double) * (size_t)(P * D));
        for (int64_t t = 0; t < Lq; ++t) {
            const double sh = (double)(P + t);
            rope_row(interleaved, D, kq + (u * Lq + t) * D, sh, theta, K + (P + t) * D);
            memcpy(V + (P + t) * D, vq + (u * Lq + t) * D, sizeof(double) * (size_t)D);
        }
        for (int64_t t = 0; t < Lq; ++t) {
            const double sh = (double)(P + t);
            const int64_t n_vis = P + t + 1; /* prefix + query rows 0..t */
            for (int g = 0; g < G; ++g) {
                rope_row(interleaved, D, q + ((u * Lq + t) * G + g) * D, sh, theta, qr);
                double m = -INFINITY;
                for (int64_t j = 0; j < n_vis; ++j) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qr[d] * K[j * D + d];
                    sc[j] = dot * scale;
                    if (sc[j] > m)
                        m = sc[j];
                }
                double z = 0.0;
                for (int64_t j = 0; j < n_vis; ++j) {
                    sc[j] = exp(sc[j] - m);
                    z += sc[j];
                }
                double *orow = o + ((u * Lq + t) * G + g) * D;
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < n_vis; ++j)
                        acc += sc[j] * V[j * D + d];
                    orow[d] = acc / z;
                }
            }
        }
        free(K); free(V); free(qr); free(sc);
    }
    return failed ? -1 : 0;
}
