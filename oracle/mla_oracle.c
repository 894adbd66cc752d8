/*
 * mla_oracle.c -- plain CPU oracle for multi-head latent attention (MLA) computed
 * from the compressed latent.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only in the seeded input generator, which holds none of
 * the method's arithmetic.
 *
 * Everything is evaluated in IEEE double precision with plain loops, one output
 * row at a time, in the order the definitions are written.  OpenMP only spreads
 * independent (batch, head) or (batch, head, query) work over host cores; it never
 * changes the order of any sum.
 *
 * Sources (pages; "LAGA" = "A Training-Memory Regression in MLA Sequence
 * Parallelism: Why Megatron-Core Forbids Absorption, and LAGA -- a
 * Communication-Efficient Fix", arXiv 2607.17644; "TPLA" = "TPLA: Tensor Parallel
 * Latent Attention for Efficient Disaggregated Prefill and Decode Inference",
 * arXiv 2508.15881; "Helix" = "Helix Parallelism: Rethinking Sharding Strategies
 * for Interactive Multi-Million-Token LLM Decoding", arXiv 2507.07120):
 *
 *  - LAGA, "What carries the argument" and Fig. 2: explicit form = per-head K/V
 *    rebuilt from the latent through W_kv_b, head-dim attention; absorbed form =
 *    q_absorbed = W_kv_b^T q_nope, attention in latent space, un-absorb after.
 *  - LAGA, axiom ledger (paper section 2.1): the kv_b up-projection is linear and
 *    shared by all heads; the normalised latent LN(latent) is common to all heads.
 *  - TPLA, "What carries the argument" / Proposition 1: that normalisation is an
 *    RMSNorm of the latent c_KV.
 *  - LAGA, "What carries the argument": only the d_kv latent plus "the small RoPE
 *    band" travel, i.e. RoPE is decoupled and k_pe is shared across heads.
 *  - Helix, "What carries the argument" and "Assumptions" (paper section 2.1.1):
 *    partial attention outputs plus log-sum-exp scalars are rescaled and summed to
 *    give the exact softmax output (the Flash-Decoding combine).
 *
 * Readings where the pages are silent:
 *  - RMSNorm: y = x * w / sqrt(mean(x^2) + eps), no mean subtraction, no bias;
 *    applied to c_KV only, never to k_pe.
 *  - RoPE: half-split pairing (t, t + d_rope/2), theta_t = base^(-2t/d_rope);
 *    query row i sits at absolute position q_offset + i, key j at position j,
 *    a decode query at position kv_len - 1.
 *  - Score scale: 1/sqrt(d_nope + d_rope) unless the caller passes another.
 *  - W_kv_b rows: head h owns rows [h*(d_nope+d_v), (h+1)*(d_nope+d_v)); the first
 *    d_nope rows give K_nope, the next d_v rows give V.  Each row has d_kv entries.
 *  - Causal mask with offset: key j is visible to query i iff j <= q_offset + i.
 *  - LSE is the natural log of the softmax normaliser, scale included.  A row that
 *    sees no key has lse = -inf and output 0.
 *  - Split-KV boundaries: contiguous chunks of ceil(kv_len / n_splits) keys; the
 *    last chunk may be shorter or empty.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- RMSNorm ---- */
/* One row: y_k = x_k * w_k / sqrt((1/d) * sum_k x_k^2 + eps).  TPLA, "What carries
 * the argument" (RMSNorm of the latent); LAGA axiom ledger (LN(latent) shared by all
 * heads). */
static void rmsnorm_row(const double *x, const double *w, int d, double eps, double *y)
{
    double ss = 0.0;
    for (int k = 0; k < d; ++k)
        ss += x[k] * x[k];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int k = 0; k < d; ++k)
        y[k] = x[k] * inv * w[k];
}

void orc_rmsnorm(const double *x, const double *w, long rows, int d, double eps, double *y)
{
    for (long r = 0; r < rows; ++r)
        rmsnorm_row(x + r * d, w, d, eps, y + r * d);
}

/* ------------------------------------------------------------------- RoPE ---- */
/* Rotary embedding of one d_rope-wide band at absolute position pos, half-split
 * pairing: for t < d_rope/2 the pair (x_t, x_{t+d/2}) is rotated by the angle
 * pos * base^(-2t/d).  LAGA, "What carries the argument" ("the small RoPE band"). */
static void rope_row(const double *x, double pos, int d, double base, double *y)
{
    int half = d / 2;
    for (int t = 0; t < half; ++t) {
        double theta = pow(base, -2.0 * (double)t / (double)d);
        double a = pos * theta;
        double c = cos(a), s = sin(a);
        double x0 = x[t], x1 = x[t + half];
        y[t] = x0 * c - x1 * s;
        y[t + half] = x1 * c + x0 * s;
    }
}

void orc_rope(const double *x, const double *pos, long rows, int d, double base, double *y)
{
    for (long r = 0; r < rows; ++r)
        rope_row(x + r * d, pos[r], d, base, y + r * d);
}

/* ------------------------------------------------------ softmax attention ---- */
/* Softmax over the given scores s[0..n): writes p[j] = exp(s_j - m) (unnormalised)
 * and returns the log-sum-exp m + log(sum_j exp(s_j - m)); n == 0 gives -inf. */
static double softmax_weights(const double *s, long n, double *p, double *z_out)
{
    if (n == 0) {
        *z_out = 0.0;
        return -INFINITY;
    }
    double m = s[0];
    for (long j = 1; j < n; ++j)
        if (s[j] > m)
            m = s[j];
    double z = 0.0;
    for (long j = 0; j < n; ++j) {
        p[j] = exp(s[j] - m);
        z += p[j];
    }
    *z_out = z;
    return m + log(z);
}

static double dot(const double *a, const double *b, int n)
{
    double acc = 0.0;
    for (int k = 0; k < n; ++k)
        acc += a[k] * b[k];
    return acc;
}

/* Number of keys query row i (absolute position pos) may attend to. */
static long visible_keys(int causal, long pos, long s_kv)
{
    if (!causal)
        return s_kv;
    long n = pos + 1;
    return n < s_kv ? n : s_kv;
}

/* ----------------------------------------------- explicit form (LAGA / B1) ---- */
/*
 * Explicit MLA forward for batches [0,B), heads [head_begin, head_begin+head_count),
 * queries at absolute positions q_off .. q_off+s_q-1 over a full latent of s_kv keys.
 * LAGA, "What carries the argument" and Fig. 2: rebuild per-head K_nope/V from the
 * normalised latent through W_kv_b (same matmul, reordered views -- the paper's
 * section 3.3 "H_r slice"), then head-dim attention with q = [q_nope ; RoPE(q_pe)],
 * k = [K_nope ; RoPE(k_pe)] (k_pe shared by all heads).
 *
 * Layouts (row-major): q_nope [B,s_q,head_count,Dn]; q_pe [B,s_q,head_count,Dr];
 * c_kv [B,s_kv,Dk]; k_pe [B,s_kv,Dr]; w_kv_b [n_heads*(Dn+Dv), Dk]; rms_w [Dk];
 * out [B,s_q,head_count,Dv]; lse [B,head_count,s_q].
 */
void orc_mla_explicit(int B, int s_q, int s_kv, int q_off, int causal,
                      int n_heads, int head_begin, int head_count,
                      int Dk, int Dn, int Dr, int Dv,
                      double base, double eps, double scale,
                      const double *q_nope, const double *q_pe, const double *c_kv,
                      const double *k_pe, const double *w_kv_b, const double *rms_w,
                      double *out, double *lse)
{
    (void)n_heads;
    long kv_need = causal ? (long)q_off + s_q : s_kv;
    if (kv_need > s_kv)
        kv_need = s_kv;
    int Dh = Dn + Dv;

    /* Step 1 (per batch, shared by every head): normalised latent and rotated k_pe. */
    double *chat = (double *)malloc(sizeof(double) * (size_t)B * (kv_need > 0 ? kv_need : 1) * Dk);
    double *krot = (double *)malloc(sizeof(double) * (size_t)B * (kv_need > 0 ? kv_need : 1) * Dr);
    for (int b = 0; b < B; ++b)
        for (long j = 0; j < kv_need; ++j) {
            rmsnorm_row(c_kv + ((size_t)b * s_kv + j) * Dk, rms_w, Dk, eps,
                        chat + ((size_t)b * kv_need + j) * Dk);
            rope_row(k_pe + ((size_t)b * s_kv + j) * Dr, (double)j, Dr, base,
                     krot + ((size_t)b * kv_need + j) * Dr);
        }

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int hl = 0; hl < head_count; ++hl) {
            int h = head_begin + hl;
            const double *wk = w_kv_b + (size_t)h * Dh * Dk;  /* Dn rows: K_nope */
            const double *wv = wk + (size_t)Dn * Dk;          /* Dv rows: V      */
            long nk = kv_need > 0 ? kv_need : 1;
            double *kn = (double *)malloc(sizeof(double) * nk * Dn);
            double *vv = (double *)malloc(sizeof(double) * nk * Dv);
            double *sc = (double *)malloc(sizeof(double) * nk);
            double *pw = (double *)malloc(sizeof(double) * nk);
            double qr[1024];

            /* Step 2: K_nope_j = W_K(h) chat_j, V_j = W_V(h) chat_j. */
            for (long j = 0; j < kv_need; ++j) {
                const double *cj = chat + ((size_t)b * kv_need + j) * Dk;
                for (int d = 0; d < Dn; ++d)
                    kn[j * Dn + d] = dot(wk + (size_t)d * Dk, cj, Dk);
                for (int d = 0; d < Dv; ++d)
                    vv[j * Dv + d] = dot(wv + (size_t)d * Dk, cj, Dk);
            }

            for (int i = 0; i < s_q; ++i) {
                long pos = (long)q_off + i;
                size_t qrow = ((size_t)b * s_q + i) * head_count + hl;
                const double *qn = q_nope + qrow * Dn;
                rope_row(q_pe + qrow * Dr, (double)pos, Dr, base, qr);
                long n = visible_keys(causal, pos, s_kv);
                /* Step 3: scores over the visible keys. */
                for (long j = 0; j < n; ++j)
                    sc[j] = scale * (dot(qn, kn + j * Dn, Dn) +
                                     dot(qr, krot + ((size_t)b * kv_need + j) * Dr, Dr));
                double z;
                double l = softmax_weights(sc, n, pw, &z);
                /* Step 4: o = sum_j softmax_j V_j. */
                double *o = out + qrow * Dv;
                for (int d = 0; d < Dv; ++d) {
                    double acc = 0.0;
                    for (long j = 0; j < n; ++j)
                        acc += pw[j] * vv[j * Dv + d];
                    o[d] = n > 0 ? acc / z : 0.0;
                }
                lse[((size_t)b * head_count + hl) * s_q + i] = l;
            }
            free(kn);
            free(vv);
            free(sc);
            free(pw);
        }
    free(chat);
    free(krot);
}

/* ----------------------------------------------- absorbed form (B2) ---- */
/*
 * Absorbed MLA forward, same arguments and layouts as orc_mla_explicit.
 * LAGA, "What carries the argument" and Fig. 2 (absorb -> latent-attn -> un-absorb):
 * q_abs = W_K(h)^T q_nope (d_kv wide), scores q_abs . chat_j + RoPE(q_pe) . RoPE(k_pe_j),
 * latent accumulator o_lat = sum_j softmax_j chat_j, then out = W_V(h) o_lat.
 */
void orc_mla_absorbed(int B, int s_q, int s_kv, int q_off, int causal,
                      int n_heads, int head_begin, int head_count,
                      int Dk, int Dn, int Dr, int Dv,
                      double base, double eps, double scale,
                      const double *q_nope, const double *q_pe, const double *c_kv,
                      const double *k_pe, const double *w_kv_b, const double *rms_w,
                      double *out, double *lse)
{
    (void)n_heads;
    long kv_need = causal ? (long)q_off + s_q : s_kv;
    if (kv_need > s_kv)
        kv_need = s_kv;
    int Dh = Dn + Dv;
    long nk = kv_need > 0 ? kv_need : 1;

    double *chat = (double *)malloc(sizeof(double) * (size_t)B * nk * Dk);
    double *krot = (double *)malloc(sizeof(double) * (size_t)B * nk * Dr);
    for (int b = 0; b < B; ++b)
        for (long j = 0; j < kv_need; ++j) {
            rmsnorm_row(c_kv + ((size_t)b * s_kv + j) * Dk, rms_w, Dk, eps,
                        chat + ((size_t)b * kv_need + j) * Dk);
            rope_row(k_pe + ((size_t)b * s_kv + j) * Dr, (double)j, Dr, base,
                     krot + ((size_t)b * kv_need + j) * Dr);
        }

#pragma omp parallel for collapse(3) schedule(dynamic, 16)
    for (int b = 0; b < B; ++b)
        for (int hl = 0; hl < head_count; ++hl)
            for (int i = 0; i < s_q; ++i) {
                int h = head_begin + hl;
                const double *wk = w_kv_b + (size_t)h * Dh * Dk;
                const double *wv = wk + (size_t)Dn * Dk;
                double *qa = (double *)malloc(sizeof(double) * Dk);
                double *ol = (double *)malloc(sizeof(double) * Dk);
                double *sc = (double *)malloc(sizeof(double) * nk);
                double *pw = (double *)malloc(sizeof(double) * nk);
                double qr[1024];
                long pos = (long)q_off + i;
                size_t qrow = ((size_t)b * s_q + i) * head_count + hl;
                const double *qn = q_nope + qrow * Dn;
                /* absorb: q_abs_k = sum_d q_nope_d W_K(h)[d][k] */
                for (int k = 0; k < Dk; ++k) {
                    double acc = 0.0;
                    for (int d = 0; d < Dn; ++d)
                        acc += qn[d] * wk[(size_t)d * Dk + k];
                    qa[k] = acc;
                }
                rope_row(q_pe + qrow * Dr, (double)pos, Dr, base, qr);
                long n = visible_keys(causal, pos, s_kv);
                for (long j = 0; j < n; ++j)
                    sc[j] = scale * (dot(qa, chat + ((size_t)b * kv_need + j) * Dk, Dk) +
                                     dot(qr, krot + ((size_t)b * kv_need + j) * Dr, Dr));
                double z;
                double l = softmax_weights(sc, n, pw, &z);
                /* latent accumulator */
                for (int k = 0; k < Dk; ++k) {
                    double acc = 0.0;
                    for (long j = 0; j < n; ++j)
                        acc += pw[j] * chat[((size_t)b * kv_need + j) * Dk + k];
                    ol[k] = n > 0 ? acc / z : 0.0;
                }
                /* un-absorb: out_d = sum_k W_V(h)[d][k] o_lat_k */
                double *o = out + qrow * Dv;
                for (int d = 0; d < Dv; ++d)
                    o[d] = dot(wv + (size_t)d * Dk, ol, Dk);
                lse[((size_t)b * head_count + hl) * s_q + i] = l;
                free(qa);
                free(ol);
                free(sc);
                free(pw);
            }
    free(chat);
    free(krot);
}

/* ---------------------------------------------------- latent decode ---- */
/*
 * One decode query per sequence at position kv_len-1, all n_heads heads, over a
 * latent cache that already holds normalised c_KV and rotated k_pe (what a prefill
 * writes).  Absorbed-form scores, as the LAGA page says the absorb trick is used only
 * in inference decode ("Core claim", abstract).  The result is the plain softmax over
 * every cached key; part_out/part_lse (when not NULL) receive the same attention
 * restricted to each contiguous split of ceil(kv_len/n_splits) keys: the latent
 * accumulator normalised within the split [n_splits,B,H,Dk] and its log-sum-exp
 * [n_splits,B,H].  The Helix page's rescale-and-sum turns those partials back into
 * the unsplit result; that identity is what orc_lse_combine states.
 *
 * Layouts: q_nope [B,H,Dn]; q_pe [B,H,Dr] (not yet rotated); c_cache [B,kv_len,Dk];
 * kpe_cache [B,kv_len,Dr]; out [B,H,Dv]; lse [B,H].
 */
void orc_mla_decode(int B, int kv_len, int n_splits, int n_heads,
                    int Dk, int Dn, int Dr, int Dv, double base, double scale,
                    const double *q_nope, const double *q_pe, const double *c_cache,
                    const double *kpe_cache, const double *w_kv_b,
                    double *out, double *lse, double *part_out, double *part_lse)
{
    int Dh = Dn + Dv;
    long chunk = n_splits > 0 ? ((long)kv_len + n_splits - 1) / n_splits : kv_len;
    long nk = kv_len > 0 ? kv_len : 1;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < n_heads; ++h) {
            const double *wk = w_kv_b + (size_t)h * Dh * Dk;
            const double *wv = wk + (size_t)Dn * Dk;
            double *qa = (double *)malloc(sizeof(double) * Dk);
            double *ol = (double *)malloc(sizeof(double) * Dk);
            double *sc = (double *)malloc(sizeof(double) * nk);
            double *pw = (double *)malloc(sizeof(double) * nk);
            double qr[1024];
            size_t row = (size_t)b * n_heads + h;
            const double *qn = q_nope + row * Dn;
            for (int k = 0; k < Dk; ++k) {
                double acc = 0.0;
                for (int d = 0; d < Dn; ++d)
                    acc += qn[d] * wk[(size_t)d * Dk + k];
                qa[k] = acc;
            }
            rope_row(q_pe + row * Dr, (double)(kv_len - 1), Dr, base, qr);
            const double *cb = c_cache + (size_t)b * kv_len * Dk;
            const double *kb = kpe_cache + (size_t)b * kv_len * Dr;
            for (long j = 0; j < kv_len; ++j)
                sc[j] = scale * (dot(qa, cb + j * Dk, Dk) + dot(qr, kb + j * Dr, Dr));

            /* unsplit softmax over all cached keys */
            double z;
            double l = softmax_weights(sc, kv_len, pw, &z);
            for (int k = 0; k < Dk; ++k) {
                double acc = 0.0;
                for (long j = 0; j < kv_len; ++j)
                    acc += pw[j] * cb[j * Dk + k];
                ol[k] = kv_len > 0 ? acc / z : 0.0;
            }
            for (int d = 0; d < Dv; ++d)
                out[row * Dv + d] = dot(wv + (size_t)d * Dk, ol, Dk);
            lse[row] = l;

            /* per-split partials: the same attention restricted to each key chunk */
            if (part_out && part_lse)
                for (int s = 0; s < n_splits; ++s) {
                    long j0 = (long)s * chunk, j1 = j0 + chunk;
                    if (j0 > kv_len)
                        j0 = kv_len;
                    if (j1 > kv_len)
                        j1 = kv_len;
                    double zs;
                    double ls = softmax_weights(sc + j0, j1 - j0, pw, &zs);
                    double *po = part_out + ((size_t)s * B * n_heads + row) * Dk;
                    for (int k = 0; k < Dk; ++k) {
                        double acc = 0.0;
                        for (long j = j0; j < j1; ++j)
                            acc += pw[j - j0] * cb[j * Dk + k];
                        po[k] = j1 > j0 ? acc / zs : 0.0;
                    }
                    part_lse[(size_t)s * B * n_heads + row] = ls;
                }
            free(qa);
            free(ol);
            free(sc);
            free(pw);
        }
}

/* ------------------------------------------------- RMSNorm backward ---- */
/*
 * Gradient of y = per-shard RMSNorm(x) * w (orc_rmsnorm on each of g shards of d/g
 * columns; g = 1 the LAGA page's latent norm, g > 1 TPLA's per-shard norm) for an
 * upstream gradient dy [rows, d]: with r the shard's sqrt(mean x^2 + eps) and ds = d/g,
 *   dx_k = dy_k w_k / r - x_k (sum over the shard of dy_m w_m x_m) / (ds r^3)
 *   dw_k = sum over rows of dy_k x_k / r
 */
void orc_rmsnorm_bwd(const double *x, const double *w, long rows, int d, int g, double eps,
                     const double *dy, double *dx, double *dw)
{
    const int ds = d / g;
    for (int k = 0; k < d; ++k)
        dw[k] = 0.0;
    for (long r = 0; r < rows; ++r)
        for (int i = 0; i < g; ++i) {
            const double *xs = x + r * d + (size_t)i * ds, *dys = dy + r * d + (size_t)i * ds;
            const double *ws = w + (size_t)i * ds;
            double ss = 0.0, gs = 0.0;
            for (int k = 0; k < ds; ++k) {
                ss += xs[k] * xs[k];
                gs += dys[k] * ws[k] * xs[k];
            }
            const double rr = sqrt(ss / ds + eps);
            for (int k = 0; k < ds; ++k) {
                dx[r * d + (size_t)i * ds + k] = dys[k] * ws[k] / rr - xs[k] * gs / ((double)ds * rr * rr * rr);
                dw[(size_t)i * ds + k] += dys[k] * xs[k] / rr;
            }
        }
}

/* ------------------------------------------------- explicit backward ---- */
/*
 * Gradients of the explicit forward (orc_mla_explicit) for a given upstream gradient
 * dout [B,s_q,head_count,Dv] of the output; the log-sum-exp is not differentiated.
 * LAGA, "What carries the argument": the sequence-parallel method is claimed to give the
 * same gradients as the baseline (bit-identical at one rank, within 2e-5 / 1e-3 at more),
 * so a backward pass is part of what the method computes; the pages print no backward
 * formulas, so these are the chain rule through the forward's own steps, written in
 * reverse order:
 *   dP_ij = dO_i . V_j,  D_i = dO_i . o_i,  dS_ij = P_ij (dP_ij - D_i)      (softmax)
 *   dq_nope_i = scale sum_j dS_ij K_nope_j,   dq_rot_i = scale sum_j dS_ij k_rot_j
 *   dK_nope_j = scale sum_i dS_ij q_nope_i,   dk_rot_j = scale sum_i dS_ij q_rot_i
 *   dV_j = sum_i P_ij dO_i
 *   RoPE is a rotation, so its transpose rotates by the opposite angle:
 *     dq_pe_i = rope(dq_rot_i, -pos_i),  dk_pe_j = rope(dk_rot_j, -j) (summed over heads)
 *   dW_K(h) = sum_j dK_nope_j chat_j^T,  dW_V(h) = sum_j dV_j chat_j^T,
 *   dchat_j = sum_h W_K(h)^T dK_nope_j + W_V(h)^T dV_j
 *   RMSNorm y = x w / r, r = sqrt(mean x^2 + eps):
 *     dx = (dy . w) / r - x (sum_k dy_k w_k x_k) / (d r^3),  dw = sum_rows dy . x / r
 * Outputs: dq_nope [B,s_q,hc,Dn], dq_pe [B,s_q,hc,Dr], dc_kv [B,s_kv,Dk],
 * dk_pe [B,s_kv,Dr], dw_kv_b [n_heads*(Dn+Dv),Dk] (rows of heads outside the range
 * stay zero), drms_w [Dk].  Keys that no query sees get zero gradients.
 */
void orc_mla_explicit_bwd(int B, int s_q, int s_kv, int q_off, int causal,
                          int n_heads, int head_begin, int head_count,
                          int Dk, int Dn, int Dr, int Dv,
                          double base, double eps, double scale,
                          const double *q_nope, const double *q_pe, const double *c_kv,
                          const double *k_pe, const double *w_kv_b, const double *rms_w,
                          const double *dout,
                          double *dq_nope, double *dq_pe, double *dc_kv, double *dk_pe,
                          double *dw_kv_b, double *drms_w)
{
    long kv_need = causal ? (long)q_off + s_q : s_kv;
    if (kv_need > s_kv)
        kv_need = s_kv;
    const int Dh = Dn + Dv;
    const long nk = kv_need > 0 ? kv_need : 1;
    memset(dc_kv, 0, sizeof(double) * (size_t)B * s_kv * Dk);
    memset(dk_pe, 0, sizeof(double) * (size_t)B * s_kv * Dr);
    memset(dw_kv_b, 0, sizeof(double) * (size_t)n_heads * Dh * Dk);
    memset(drms_w, 0, sizeof(double) * Dk);

    /* forward step 1 again: normalised latent and rotated k_pe */
    double *chat = (double *)malloc(sizeof(double) * (size_t)B * nk * Dk);
    double *krot = (double *)malloc(sizeof(double) * (size_t)B * nk * Dr);
    double *dchat = (double *)calloc((size_t)B * nk * Dk, sizeof(double));
    double *dkrot = (double *)calloc((size_t)B * nk * Dr, sizeof(double));
    for (int b = 0; b < B; ++b)
        for (long j = 0; j < kv_need; ++j) {
            rmsnorm_row(c_kv + ((size_t)b * s_kv + j) * Dk, rms_w, Dk, eps, chat + ((size_t)b * nk + j) * Dk);
            rope_row(k_pe + ((size_t)b * s_kv + j) * Dr, (double)j, Dr, base, krot + ((size_t)b * nk + j) * Dr);
        }

    double *kn = (double *)malloc(sizeof(double) * nk * Dn);
    double *vv = (double *)malloc(sizeof(double) * nk * Dv);
    double *dkn = (double *)malloc(sizeof(double) * nk * Dn);
    double *dvv = (double *)malloc(sizeof(double) * nk * Dv);
    double *sc = (double *)malloc(sizeof(double) * nk);
    double *pw = (double *)malloc(sizeof(double) * nk);
    double qr[1024], dqr[1024], o[1024];
    for (int b = 0; b < B; ++b)
        for (int hl = 0; hl < head_count; ++hl) {
            const int h = head_begin + hl;
            const double *wk = w_kv_b + (size_t)h * Dh * Dk, *wv = wk + (size_t)Dn * Dk;
            double *dwk = dw_kv_b + (size_t)h * Dh * Dk, *dwv = dwk + (size_t)Dn * Dk;
            for (long j = 0; j < kv_need; ++j) {   /* forward step 2 again */
                const double *cj = chat + ((size_t)b * nk + j) * Dk;
                for (int d = 0; d < Dn; ++d)
                    kn[j * Dn + d] = dot(wk + (size_t)d * Dk, cj, Dk);
                for (int d = 0; d < Dv; ++d)
                    vv[j * Dv + d] = dot(wv + (size_t)d * Dk, cj, Dk);
            }
            memset(dkn, 0, sizeof(double) * nk * Dn);
            memset(dvv, 0, sizeof(double) * nk * Dv);
            for (int i = 0; i < s_q; ++i) {
                const long pos = (long)q_off + i;
                const size_t qrow = ((size_t)b * s_q + i) * head_count + hl;
                const double *qn = q_nope + qrow * Dn, *dO = dout + qrow * Dv;
                rope_row(q_pe + qrow * Dr, (double)pos, Dr, base, qr);
                const long n = visible_keys(causal, pos, s_kv);
                for (long j = 0; j < n; ++j)
                    sc[j] = scale * (dot(qn, kn + j * Dn, Dn) + dot(qr, krot + ((size_t)b * nk + j) * Dr, Dr));
                double z;
                softmax_weights(sc, n, pw, &z);
                for (int d = 0; d < Dv; ++d) {
                    double acc = 0.0;
                    for (long j = 0; j < n; ++j)
                        acc += pw[j] * vv[j * Dv + d];
                    o[d] = n > 0 ? acc / z : 0.0;
                }
                const double Di = dot(dO, o, Dv);
                double *dqn = dq_nope + qrow * Dn;
                for (int d = 0; d < Dn; ++d)
                    dqn[d] = 0.0;
                for (int d = 0; d < Dr; ++d)
                    dqr[d] = 0.0;
                for (long j = 0; j < n; ++j) {
                    const double p = pw[j] / z;
                    const double ds = p * (dot(dO, vv + j * Dv, Dv) - Di);
                    const double *kr = krot + ((size_t)b * nk + j) * Dr;
                    double *dkr = dkrot + ((size_t)b * nk + j) * Dr;
                    for (int d = 0; d < Dn; ++d) {
                        dqn[d] += scale * ds * kn[j * Dn + d];
                        dkn[j * Dn + d] += scale * ds * qn[d];
                    }
                    for (int d = 0; d < Dr; ++d) {
                        dqr[d] += scale * ds * kr[d];
                        dkr[d] += scale * ds * qr[d];
                    }
                    for (int d = 0; d < Dv; ++d)
                        dvv[j * Dv + d] += p * dO[d];
                }
                rope_row(dqr, -(double)pos, Dr, base, dq_pe + qrow * Dr);
            }
            /* through the reconstruction: weight gradients and the latent's gradient */
            for (long j = 0; j < kv_need; ++j) {
                const double *cj = chat + ((size_t)b * nk + j) * Dk;
                double *dcj = dchat + ((size_t)b * nk + j) * Dk;
                for (int d = 0; d < Dn; ++d)
                    for (int k = 0; k < Dk; ++k) {
                        dwk[(size_t)d * Dk + k] += dkn[j * Dn + d] * cj[k];
                        dcj[k] += wk[(size_t)d * Dk + k] * dkn[j * Dn + d];
                    }
                for (int d = 0; d < Dv; ++d)
                    for (int k = 0; k < Dk; ++k) {
                        dwv[(size_t)d * Dk + k] += dvv[j * Dv + d] * cj[k];
                        dcj[k] += wv[(size_t)d * Dk + k] * dvv[j * Dv + d];
                    }
            }
        }
    /* through RoPE of the keys and the RMSNorm of the latent */
    for (int b = 0; b < B; ++b)
        for (long j = 0; j < kv_need; ++j) {
            rope_row(dkrot + ((size_t)b * nk + j) * Dr, -(double)j, Dr, base, dk_pe + ((size_t)b * s_kv + j) * Dr);
            const double *x = c_kv + ((size_t)b * s_kv + j) * Dk, *dy = dchat + ((size_t)b * nk + j) * Dk;
            double ss = 0.0, g = 0.0;
            for (int k = 0; k < Dk; ++k) {
                ss += x[k] * x[k];
                g += dy[k] * rms_w[k] * x[k];
            }
            const double r = sqrt(ss / Dk + eps);
            double *dx = dc_kv + ((size_t)b * s_kv + j) * Dk;
            for (int k = 0; k < Dk; ++k) {
                dx[k] = dy[k] * rms_w[k] / r - x[k] * g / ((double)Dk * r * r * r);
                drms_w[k] += dy[k] * x[k] / r;
            }
        }
    free(kn);
    free(vv);
    free(dkn);
    free(dvv);
    free(sc);
    free(pw);
    free(chat);
    free(krot);
    free(dchat);
    free(dkrot);
}

/* ------------------------------------------------- TPLA latent decode ---- */
/*
 * TPLA, "The reading" and "What carries the argument": the latent c_KV and each head's
 * input dimension are split into g shards; every shard attends with all query heads over
 * its own part of the latent (a local softmax over its own scores) and the shards'
 * outputs are summed (the all-reduce).  The page calls the result a grouped latent
 * attention with replicated heads.  Readings where the page is silent:
 *  - no orthogonal reparameterisation (U = I): its Hadamard and PCA forms need
 *    calibration data;
 *  - shard i owns latent dims [i Dk/g, (i+1) Dk/g) and normalises them by its own
 *    RMSNorm with the matching slice of the weight (Condition 1 read as a per-shard
 *    norm);
 *  - every shard also reads the whole RoPE band (576 -> 320 dims per shard at g = 2);
 *  - the score scale stays 1/sqrt(d_nope + d_rope) and the local softmax is not
 *    rescaled (the referee report's second major comment: the deployed form uses an
 *    unscaled local softmax).
 * Inputs as orc_mla_decode, except that c_raw [B,kv_len,Dk] is the latent before any
 * normalisation (rms_w [Dk], eps); with rms_w NULL it is taken as already normalised
 * shard by shard (what a deployed cache holds).  Outputs: out [B,H,Dv], the sum over
 * shards, and shard_lse [g,B,H], each shard's log-sum-exp.
 */
void orc_tpla_decode(int B, int kv_len, int g, int n_heads, int Dk, int Dn, int Dr, int Dv,
                     double base, double scale, double eps,
                     const double *q_nope, const double *q_pe, const double *c_raw,
                     const double *kpe_cache, const double *w_kv_b, const double *rms_w,
                     double *out, double *shard_lse)
{
    int Dh = Dn + Dv, ds = Dk / g;
    long nk = kv_len > 0 ? kv_len : 1;
    /* the per-shard normalised latent of every cached key */
    double *chat = (double *)malloc(sizeof(double) * (size_t)B * nk * Dk);
    for (long r = 0; r < (long)B * kv_len; ++r)
        for (int i = 0; i < g; ++i) {
            if (rms_w)
                rmsnorm_row(c_raw + r * Dk + (size_t)i * ds, rms_w + (size_t)i * ds, ds, eps,
                            chat + r * Dk + (size_t)i * ds);
            else
                memcpy(chat + r * Dk + (size_t)i * ds, c_raw + r * Dk + (size_t)i * ds, sizeof(double) * ds);
        }

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < n_heads; ++h) {
            const double *wk = w_kv_b + (size_t)h * Dh * Dk;
            const double *wv = wk + (size_t)Dn * Dk;
            double *qa = (double *)malloc(sizeof(double) * Dk);
            double *ol = (double *)malloc(sizeof(double) * Dk);
            double *sc = (double *)malloc(sizeof(double) * nk);
            double *pw = (double *)malloc(sizeof(double) * nk);
            double qr[1024];
            size_t row = (size_t)b * n_heads + h;
            const double *qn = q_nope + row * Dn;
            for (int k = 0; k < Dk; ++k) {
                double acc = 0.0;
                for (int d = 0; d < Dn; ++d)
                    acc += qn[d] * wk[(size_t)d * Dk + k];
                qa[k] = acc;
            }
            rope_row(q_pe + row * Dr, (double)(kv_len - 1), Dr, base, qr);
            const double *cb = chat + (size_t)b * kv_len * Dk;
            const double *kb = kpe_cache + (size_t)b * kv_len * Dr;
            for (int d = 0; d < Dv; ++d)
                out[row * Dv + d] = 0.0;
            for (int i = 0; i < g; ++i) {
                const int k0 = i * ds;
                /* this shard's scores: its latent dims plus the whole RoPE band */
                for (long j = 0; j < kv_len; ++j)
                    sc[j] = scale * (dot(qa + k0, cb + j * Dk + k0, ds) + dot(qr, kb + j * Dr, Dr));
                double z;
                double l = softmax_weights(sc, kv_len, pw, &z);
                for (int k = k0; k < k0 + ds; ++k) {
                    double acc = 0.0;
                    for (long j = 0; j < kv_len; ++j)
                        acc += pw[j] * cb[j * Dk + k];
                    ol[k] = kv_len > 0 ? acc / z : 0.0;
                }
                /* this shard's part of the up-projection, summed over the shards */
                for (int d = 0; d < Dv; ++d)
                    out[row * Dv + d] += dot(wv + (size_t)d * Dk + k0, ol + k0, ds);
                shard_lse[(size_t)i * B * n_heads + row] = l;
            }
            free(qa);
            free(ol);
            free(sc);
            free(pw);
        }
    free(chat);
}

/* ------------------------------------------------------ LSE combine ---- */
/*
 * Helix, "What carries the argument" and "Assumptions" (paper section 2.1.1):
 * given per-split outputs o_s (each normalised within its split) and their
 * log-sum-exp l_s, the full result is lse = log sum_s exp(l_s) and
 * o = sum_s exp(l_s - lse) o_s.  Splits with l_s = -inf (no keys) carry no weight;
 * if every split is empty the row gives lse = -inf and o = 0.
 * Layouts: part_out [n_splits,rows,D]; part_lse [n_splits,rows]; out [rows,D]; lse [rows].
 */
void orc_lse_combine(int n_splits, long rows, int D, const double *part_out,
                     const double *part_lse, double *out, double *lse)
{
    for (long r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < n_splits; ++s)
            if (part_lse[(size_t)s * rows + r] > m)
                m = part_lse[(size_t)s * rows + r];
        double *o = out + (size_t)r * D;
        if (m == -INFINITY) {
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int s = 0; s < n_splits; ++s)
            z += exp(part_lse[(size_t)s * rows + r] - m);
        double l = m + log(z);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int s = 0; s < n_splits; ++s)
                acc += exp(part_lse[(size_t)s * rows + r] - l) *
                       part_out[((size_t)s * rows + r) * D + d];
            o[d] = acc;
        }
        lse[r] = l;
    }
}
