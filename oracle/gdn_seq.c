/*
 * Gated delta rule, sequential form, in fp64 on the host.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the oracle that the CUDA path is
 * checked against.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm may load it.  It shares no code, header or
 * constant with the CUDA library.
 *
 * Definition followed (ferrox-core `gdn_chunk.rs`, module docs, "The
 * algebra"; metaltile-std `gated_delta_wy.rs`, module docs, "Algorithm"):
 * for one (batch b, value head hv) with state S (Dv x Dk), per token t
 *
 *     x_t = S_{t-1} k_t
 *     d_t = beta_t (v_t - g_t x_t)
 *     S_t = g_t S_{t-1} + d_t k_t^T
 *     y_t = S_t q_t / sqrt(Dk)
 *
 * with k_t, q_t read from key head hk = hv / (Hv / Hk) (grouped GQA map,
 * metaltile-std `gated_delta_wy.rs`, "Layouts").  The gate g is the
 * multiplicative decay in (0, 1].
 *
 * Layouts (row-major, contiguous):
 *   q, k  [B, T, Hk, Dk]     v, y [B, T, Hv, Dv]     g, beta [B, T, Hv]
 *   s0, s [B, Hv, Dv, Dk]    (s0 may be NULL: zero initial state)
 *
 * Each value row r of S evolves on its own (x_t[r] depends only on row r),
 * so the loop below walks one row at a time; that is the same arithmetic
 * as the matrix form above, in the same order of operations per element.
 */
#include <math.h>
#include <stddef.h>
#include <string.h>

void gdn_seq_f64(int B, int T, int Hk, int Hv, int Dk, int Dv,
                 const double *q, const double *k, const double *v,
                 const double *g, const double *beta,
                 const double *s0, double *s, double *y)
{
    const int group = Hv / Hk;
    const double scale = 1.0 / sqrt((double)Dk);
    const size_t state_elems = (size_t)Dv * (size_t)Dk;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int hv = 0; hv < Hv; ++hv) {
            const int hk = hv / group;
            double *S = s + ((size_t)b * Hv + hv) * state_elems;
            if (s0)
                memcpy(S, s0 + ((size_t)b * Hv + hv) * state_elems,
                       state_elems * sizeof(double));
            else
                memset(S, 0, state_elems * sizeof(double));

            for (int t = 0; t < T; ++t) {
                const size_t tok = (size_t)b * T + t;
                const double *kt = k + (tok * Hk + hk) * Dk;
                const double *qt = q + (tok * Hk + hk) * Dk;
                const double *vt = v + (tok * Hv + hv) * Dv;
                double *yt = y + (tok * Hv + hv) * Dv;
                const double gt = g[tok * Hv + hv];
                const double bt = beta[tok * Hv + hv];

                for (int r = 0; r < Dv; ++r) {
                    double *Sr = S + (size_t)r * Dk;
                    double x = 0.0;
                    for (int c = 0; c < Dk; ++c)
                        x += Sr[c] * kt[c];
                    const double d = bt * (vt[r] - gt * x);
                    double out = 0.0;
                    for (int c = 0; c < Dk; ++c) {
                        Sr[c] = gt * Sr[c] + d * kt[c];
                        out += Sr[c] * qt[c];
                    }
                    yt[r] = out * scale;
                }
            }
        }
    }
}
