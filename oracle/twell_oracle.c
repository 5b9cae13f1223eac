/*
 * twell_oracle.c -- plain, slow fp64 CPU oracle for the activation-sparse gated FFN and the
 * tile-wise ELL (TwELL) / hybrid formats.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
 * reference legs load this library; the product path never does. It shares no code, header,
 * table or helper with the CUDA library: every step here is written out from the pages.
 *
 * Pages cited (title, then section):
 *   [AIM] aimodeling.com news item "TwELL：Sakana AI与NVIDIA联合提出稀疏LLM推理加速20%，解决GPU批处理落地难题",
 *         summary paragraphs 1-5.
 *   [TG]  Telegram post "Sakana AI и NVIDIA представили TwELL ..." (ai_machinelearning_big_data),
 *         sections "Вот тут и решает TwELL", "Инференс", "Обучение".
 *   [PUL] pulsen.vercel.app "Sakana AI og NVIDIA introduserer TwELL ...", paragraphs 1-5.
 *   [TC]  Tencent Cloud "一文读懂 NVIDIA 与 Sakana AI 联手打造的稀疏 LLM 黑科技", sections 1-6.
 *
 * Notation: N tokens, d = d_model, f = d_ff, T = column-tile width, nt = ceil(f/T), K = hybrid
 * capacity. Weights are stored one row per hidden unit: Wg_s, Wu_s, Wd_s are [f, d] row-major,
 * so G = x Wg_s^T, U = x Wu_s^T, y = H Wd_s. All arithmetic is fp64; inputs arrive as fp64
 * copies of bf16- or fp32-exact values.
 *
 * Parity pins (tests/test_oracle.py): every function below is checked against something other
 * than itself -- library routines (torch fp64 matmul/autograd, torch's bf16 conversion),
 * invariants, closed forms, brute force on tiny inputs and central finite differences.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int64_t i64;

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ rounding --------------- */

/* Round a double to the nearest bf16 value (8 significant bits, fp32 exponent range with
 * subnormals), ties to even. This is the definition of IEEE round-to-nearest-even for a format
 * with a 7-bit stored mantissa: the quantum is 2^(e-7) inside binade [2^e, 2^(e+1)) and 2^-133
 * below the normal range; overflow past the largest finite value goes to infinity. The pages
 * fix no precision; bf16 storage with fp32 accumulation is this build's reading. */
EXPORT double oracle_round_bf16(double v)
{
    if (v != v || v == 0.0 || isinf(v)) return v;
    double a = fabs(v);
    int e2;
    frexp(a, &e2);           /* a = m * 2^e2 with m in [0.5, 1) */
    int e = e2 - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;  /* subnormal range keeps the quantum of the lowest binade */
    double q = ldexp(1.0, e - 7);
    double r = nearbyint(a / q) * q; /* default rounding mode: to nearest, ties to even */
    if (r >= ldexp(1.0, 128)) r = INFINITY;
    return copysign(r, v);
}

EXPORT void oracle_round_bf16_array(i64 n, const double* in, double* out)
{
    for (i64 i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}

/* ------------------------------------------------------------------ dense FFN -------------- */

static double dot(const double* a, const double* b, i64 n)
{
    double s = 0.0;
    for (i64 i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* Gate pre-activations G[r, j] = x_r . Wg_s[j] for the selected rows.
 * [TC] §1 (gated FFN as in Llama: the gate projection decides the sparsity pattern). */
EXPORT void oracle_gate_rows(i64 n_sel, const i64* rows, i64 d, i64 f, const double* x,
                             const double* Wg_s, double* G_out)
{
#pragma omp parallel for schedule(dynamic)
    for (i64 s = 0; s < n_sel; ++s) {
        const double* xr = x + rows[s] * d;
        for (i64 j = 0; j < f; ++j) G_out[s * f + j] = dot(xr, Wg_s + j * d, d);
    }
}

/* The layer itself, for the selected rows:
 *   g = x_r Wg_s^T,  a = ReLU(g),  u = x_r Wu_s^T,  h = a * u,  y_r = h Wd_s.
 * Gated FFN framing: [TC] §1; ReLU in place of SiLU on the gate: [AIM] ¶4, [PUL] ¶4.
 * This is the plain dense definition (every hidden unit, zeros included); the TwELL method
 * reaches exactly this result by skipping the zero terms ([AIM] ¶3, [TG] "Инференс").
 * G_out / U_out ([n_sel, f]) may be NULL. */
EXPORT void oracle_ffn_rows(i64 n_sel, const i64* rows, i64 d, i64 f, const double* x,
                            const double* Wg_s, const double* Wu_s, const double* Wd_s,
                            double* y_out, double* G_out, double* U_out)
{
#pragma omp parallel for schedule(dynamic)
    for (i64 s = 0; s < n_sel; ++s) {
        const double* xr = x + rows[s] * d;
        double* yr = y_out + s * d;
        for (i64 c = 0; c < d; ++c) yr[c] = 0.0;
        for (i64 j = 0; j < f; ++j) {
            double g = dot(xr, Wg_s + j * d, d);
            double u = dot(xr, Wu_s + j * d, d);
            double a = g > 0.0 ? g : 0.0;
            double h = a * u;
            if (G_out) G_out[s * f + j] = g;
            if (U_out) U_out[s * f + j] = u;
            const double* wd = Wd_s + j * d;
            for (i64 c = 0; c < d; ++c) yr[c] += h * wd[c];
        }
    }
}

/* ------------------------------------------------------------------ TwELL ------------------ */

/* TwELL pack of a given gate matrix G [N, f] with tile width T.
 * The columns of the gate activation are cut into tiles of T columns; inside each tile only
 * the nonzero values and their in-tile column indices are kept, in local ELL form
 * ([TG] "Вот тут и решает TwELL"; [TC] §2). A gate entry is kept iff g > 0 (ReLU,
 * [AIM] ¶4), scanning each tile's columns in ascending order. The last tile covers
 * columns [(nt-1)T, f) when T does not divide f.
 * Outputs: cnt[N, nt]; vals[N, nt, T] and idx[N, nt, T] hold entries 0..cnt-1 of each
 * (row, tile) slot; entries past cnt are not written. Values are copied unchanged. */
EXPORT void oracle_twell_pack(i64 N, i64 f, i64 T, const double* G, double* vals, uint8_t* idx,
                              uint16_t* cnt)
{
    i64 nt = (f + T - 1) / T;
    for (i64 r = 0; r < N; ++r) {
        for (i64 t = 0; t < nt; ++t) {
            i64 c = 0;
            i64 slot = (r * nt + t) * T;
            for (i64 k = 0; k < T; ++k) {
                i64 j = t * T + k;
                if (j >= f) break;
                double g = G[r * f + j];
                if (g > 0.0) {
                    vals[slot + c] = g;
                    idx[slot + c] = (uint8_t)k;
                    ++c;
                }
            }
            cnt[r * nt + t] = (uint16_t)c;
        }
    }
}

/* Inverse of the pack: a dense [N, f] matrix, zero except at the packed positions. */
EXPORT void oracle_twell_unpack(i64 N, i64 f, i64 T, const double* vals, const uint8_t* idx,
                                const uint16_t* cnt, double* dense)
{
    i64 nt = (f + T - 1) / T;
    memset(dense, 0, (size_t)(N * f) * sizeof(double));
    for (i64 r = 0; r < N; ++r)
        for (i64 t = 0; t < nt; ++t) {
            i64 slot = (r * nt + t) * T;
            for (i64 k = 0; k < cnt[r * nt + t]; ++k)
                dense[r * f + t * T + idx[slot + k]] = vals[slot + k];
        }
}

/* Fused up+down walk over a TwELL matrix of gate activations a ([AIM] ¶3; [TG] "Инференс";
 * [PUL] ¶3; [TC] §2): for every token row, walk its packed nonzeros tile by tile; for each
 * one (column j = t*T + idx, value a) fetch row j of Wu_s and of Wd_s, form u = x_r . Wu_s[j],
 * h = a * u, and accumulate y_r += h * Wd_s[j]. The dense hidden matrix is never formed. */
EXPORT void oracle_twell_walk(i64 N, i64 d, i64 f, i64 T, const double* vals, const uint8_t* idx,
                              const uint16_t* cnt, const double* x, const double* Wu_s,
                              const double* Wd_s, double* y)
{
    i64 nt = (f + T - 1) / T;
#pragma omp parallel for schedule(dynamic)
    for (i64 r = 0; r < N; ++r) {
        const double* xr = x + r * d;
        double* yr = y + r * d;
        for (i64 c = 0; c < d; ++c) yr[c] = 0.0;
        for (i64 t = 0; t < nt; ++t) {
            i64 slot = (r * nt + t) * T;
            for (i64 k = 0; k < cnt[r * nt + t]; ++k) {
                i64 j = t * T + idx[slot + k];
                double a = vals[slot + k];
                double u = dot(xr, Wu_s + j * d, d);
                double h = a * u;
                const double* wd = Wd_s + j * d;
                for (i64 c = 0; c < d; ++c) yr[c] += h * wd[c];
            }
        }
    }
}

/* ------------------------------------------------------------------ hybrid format ---------- */

/* Hybrid routing of a given gate matrix G [N, f] with per-row capacity K ([TG] "Обучение":
 * each row is either squeezed into one globally aligned sparse block or, on rare overflow,
 * falls into a dense backup; [TC] §3: most rows go to a compact sparse matrix, the few very
 * dense rows to a dense backup buffer).
 * Reading of the rule: nnz_r = #{j : G[r,j] > 0}; a row overflows iff nnz_r > K.
 *   - nnz_r <= K: hcnt[r] = nnz_r; slots k < nnz_r of row r hold the kept columns in ascending
 *     order (hcol) and their values (hval_a); slots k >= nnz_r hold value +0 and column 0.
 *   - nnz_r >  K: hcnt[r] = 0xFFFF, no slot of row r is written; r is appended to the backup
 *     list in ascending row order, and its dense activation row max(G_r, 0) goes to A_b.
 *     Rows beyond backup_cap are counted but not stored.
 * *n_backup receives the total number of overflow rows. */
EXPORT void oracle_hybrid_route(i64 N, i64 f, i64 K, const double* G, i64 backup_cap,
                                double* hval_a, uint16_t* hcol, uint16_t* hcnt, int32_t* brows,
                                int32_t* n_backup, double* A_b)
{
    i64 nb = 0;
    for (i64 r = 0; r < N; ++r) {
        const double* gr = G + r * f;
        i64 nnz = 0;
        for (i64 j = 0; j < f; ++j) nnz += gr[j] > 0.0;
        if (nnz <= K) {
            hcnt[r] = (uint16_t)nnz;
            i64 k = 0;
            for (i64 j = 0; j < f; ++j)
                if (gr[j] > 0.0) {
                    hval_a[r * K + k] = gr[j];
                    hcol[r * K + k] = (uint16_t)j;
                    ++k;
                }
            for (; k < K; ++k) {
                hval_a[r * K + k] = 0.0;
                hcol[r * K + k] = 0;
            }
        } else {
            hcnt[r] = 0xFFFF;
            if (nb < backup_cap) {
                brows[nb] = (int32_t)r;
                for (i64 j = 0; j < f; ++j) A_b[nb * f + j] = gr[j] > 0.0 ? gr[j] : 0.0;
            }
            ++nb;
        }
    }
    *n_backup = (int32_t)nb;
}

/* ------------------------------------------------------------------ L1 term ---------------- */

/* L1 regulariser on the hidden activations ([AIM] ¶4; [PUL] ¶4: coefficient 2e-5 on the hidden
 * feed-forward activations). Reading: the penalty is lambda * mean|h| over all N*f entries of
 * h = ReLU(x Wg_s^T) * (x Wu_s^T). Returns lambda * sum|h| / (N f). */
EXPORT double oracle_l1(i64 N, i64 d, i64 f, double lambda, const double* x, const double* Wg_s,
                        const double* Wu_s)
{
    double total = 0.0;
#pragma omp parallel for schedule(dynamic) reduction(+ : total)
    for (i64 r = 0; r < N; ++r) {
        const double* xr = x + r * d;
        double s = 0.0;
        for (i64 j = 0; j < f; ++j) {
            double g = dot(xr, Wg_s + j * d, d);
            if (g > 0.0) s += fabs(g * dot(xr, Wu_s + j * d, d));
        }
        total += s;
    }
    return lambda * total / ((double)N * (double)f);
}

/* ------------------------------------------------------------------ backward --------------- */

/* Gradients of  L = <y, dy> + lambda * mean|h|  (chain rule; the pages give only "L1 on the
 * hidden activations", [PUL] ¶4). With a = ReLU(g), h = a u, mean over the N*f entries of h:
 *   dh = dy_r . Wd_s[j] + lambda * sgn(h) / (N f)
 *   du = dh * a,   dg = dh * u * [g > 0]            (ReLU'(0) = 0, sgn(0) = 0)
 *   dx_r    = sum_j du * Wu_s[j] + dg * Wg_s[j]
 *   dWd_s[j] = sum_r h * dy_r,  dWu_s[j] = sum_r du * x_r,  dWg_s[j] = sum_r dg * x_r.
 * N_total is the N of the mean (the whole batch), even when only some rows are evaluated. */
static void local_grads(const double* xr, const double* dyr, i64 j, i64 d, i64 f, i64 N_total,
                        double lambda, const double* Wg_s, const double* Wu_s, const double* Wd_s,
                        double* h_o, double* du_o, double* dg_o)
{
    double g = dot(xr, Wg_s + j * d, d);
    if (!(g > 0.0)) { /* a = 0: then h = 0, sgn(h) = 0, du = dh * 0 = 0 and dg = 0 exactly */
        *h_o = *du_o = *dg_o = 0.0;
        return;
    }
    double u = dot(xr, Wu_s + j * d, d);
    double a = g;
    double h = a * u;
    double sg = h > 0.0 ? 1.0 : (h < 0.0 ? -1.0 : 0.0);
    double dh = dot(dyr, Wd_s + j * d, d) + lambda * sg / ((double)N_total * (double)f);
    *h_o = h;
    *du_o = dh * a;
    *dg_o = dh * u;
}

/* dx for the selected rows. */
EXPORT void oracle_ffn_bwd_rows(i64 n_sel, const i64* rows, i64 N_total, i64 d, i64 f,
                                double lambda, const double* x, const double* Wg_s,
                                const double* Wu_s, const double* Wd_s, const double* dy,
                                double* dx_out)
{
#pragma omp parallel for schedule(dynamic)
    for (i64 s = 0; s < n_sel; ++s) {
        i64 r = rows[s];
        const double* xr = x + r * d;
        const double* dyr = dy + r * d;
        double* dxr = dx_out + s * d;
        for (i64 c = 0; c < d; ++c) dxr[c] = 0.0;
        for (i64 j = 0; j < f; ++j) {
            double h, du, dg;
            local_grads(xr, dyr, j, d, f, N_total, lambda, Wg_s, Wu_s, Wd_s, &h, &du, &dg);
            const double* wu = Wu_s + j * d;
            const double* wg = Wg_s + j * d;
            for (i64 c = 0; c < d; ++c) dxr[c] += du * wu[c] + dg * wg[c];
        }
    }
}

/* dWg_s, dWu_s, dWd_s for the selected hidden units j, summed over all N rows. */
EXPORT void oracle_ffn_bwd_cols(i64 n_sel, const i64* cols, i64 N, i64 d, i64 f, double lambda,
                                const double* x, const double* Wg_s, const double* Wu_s,
                                const double* Wd_s, const double* dy, double* dWg_out,
                                double* dWu_out, double* dWd_out)
{
#pragma omp parallel for schedule(dynamic)
    for (i64 s = 0; s < n_sel; ++s) {
        i64 j = cols[s];
        double* wg = dWg_out + s * d;
        double* wu = dWu_out + s * d;
        double* wd = dWd_out + s * d;
        for (i64 c = 0; c < d; ++c) wg[c] = wu[c] = wd[c] = 0.0;
        for (i64 r = 0; r < N; ++r) {
            const double* xr = x + r * d;
            const double* dyr = dy + r * d;
            double h, du, dg;
            local_grads(xr, dyr, j, d, f, N, lambda, Wg_s, Wu_s, Wd_s, &h, &du, &dg);
            if (h == 0.0 && du == 0.0 && dg == 0.0) continue; /* adds exact zeros */
            for (i64 c = 0; c < d; ++c) {
                wd[c] += h * dyr[c];
                wu[c] += du * xr[c];
                wg[c] += dg * xr[c];
            }
        }
    }
}

/* Threads used by the parallel loops above (test infrastructure: lets a caller time the oracle on
 * one core or on every core of its affinity mask). */
void oracle_set_threads(int64_t n) { omp_set_num_threads(n > 0 ? (int)n : 1); }
int64_t oracle_max_threads(void) { return (int64_t)omp_get_max_threads(); }
