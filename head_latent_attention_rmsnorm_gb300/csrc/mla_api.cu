// mla_api.cu -- the C ABI of libmla: argument validation, workspace layout and the
// sequence of kernel launches for each entry point.  See include/mla.h for the
// contract of every call.
//
// Two kernel families sit behind each entry point:
//  * tensor cores (tcgen05 + TMA, tc_*.cu) for bf16 calls at the dimensions they
//    were written for; their intermediates (normalised latent, rotated RoPE bands,
//    K_nope, V^T, q_abs, o_lat) are stored as fp16, whose 11-bit significand keeps
//    every score within ~3e-4 of exact;
//  * CUDA cores (simt.cu) for fp32 calls and any other shape; their intermediates
//    are fp32.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_internal.h"

namespace {

using namespace mla;

thread_local int g_last_path = 0;
thread_local int g_path_override = 0;
thread_local int g_fused_cluster = 0;   // 0: chosen per call

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over the caller's workspace; every sub-buffer is 256-byte aligned.
struct Carve {
    size_t off = 0;
    char *base = nullptr;
    void *take(size_t bytes) {
        off = align_up(off, 256);
        void *p = base ? base + off : nullptr;
        off += bytes;
        return p;
    }
};

bool valid_dtype(mla_dtype dt) { return dt == MLA_F32 || dt == MLA_BF16; }

mla_status check_dims(const mla_dims *d) {
    if (!d) return MLA_ERR_NULL;
    if (d->n_heads <= 0 || d->d_kv <= 0 || d->d_nope <= 0 || d->d_rope <= 0 || d->d_v <= 0 ||
        (d->d_rope & 1) || d->d_rope > 1024 || !(d->rope_base > 0.f) || !(d->rms_eps >= 0.f))
        return MLA_ERR_SHAPE;
    return MLA_OK;
}

float scale_of(const mla_dims *d) {
    return d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / sqrtf((float)(d->d_nope + d->d_rope));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Outputs must not overlap inputs or one another.
mla_status check_alias(const Range *in, int n_in, const Range *out, int n_out) {
    for (int i = 0; i < n_out; ++i) {
        if (out[i].lo == out[i].hi) continue;
        for (int j = 0; j < n_in; ++j)
            if (in[j].lo != in[j].hi && overlap(out[i], in[j])) return MLA_ERR_ALIAS;
        for (int j = i + 1; j < n_out; ++j)
            if (out[j].lo != out[j].hi && overlap(out[i], out[j])) return MLA_ERR_ALIAS;
    }
    return MLA_OK;
}
Range rng(const void *p, size_t bytes) { return Range{(uintptr_t)p, (uintptr_t)p + (p ? bytes : 0)}; }

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }
#define MLA_TRY(x)                                   \
    do {                                             \
        cudaError_t e_ = (x);                        \
        if (e_ != cudaSuccess) return MLA_ERR_CUDA;  \
    } while (0)

// ------------------------------------------------------------ prefill shapes ----
struct Prefill {
    int B, s_q, s_kv, q_offset, causal, head_begin, head_count, hs, n_shards;
    int Dk, Dn, Dr, Dv, H;
    long kv_need, kv_pad;
    bool tc;
    int tin, tmid;   // storage of inputs, of intermediates
};

mla_status prefill_shape(const mla_dims *d, mla_dtype dt, int B, int s_q, int s_kv, int q_offset, int causal,
                         int head_begin, int head_count, int head_shard, bool absorbed, Prefill *p) {
    mla_status st = check_dims(d);
    if (st != MLA_OK) return st;
    if (!valid_dtype(dt)) return MLA_ERR_DTYPE;
    if (B < 0 || s_q < 0 || s_kv < 0 || q_offset < 0 || head_begin < 0 || head_count < 0 || head_shard < 0 ||
        (long)head_begin + head_count > d->n_heads)
        return MLA_ERR_SHAPE;
    if (causal && (long)q_offset + s_q > s_kv) return MLA_ERR_SHAPE;
    p->B = B;
    p->s_q = s_q;
    p->s_kv = s_kv;
    p->q_offset = q_offset;
    p->causal = causal ? 1 : 0;
    p->head_begin = head_begin;
    p->head_count = head_count;
    p->hs = head_shard == 0 ? std::max(head_count, 1) : std::min(head_shard, std::max(head_count, 1));
    p->n_shards = head_count == 0 ? 0 : (head_count + p->hs - 1) / p->hs;
    p->Dk = d->d_kv;
    p->Dn = d->d_nope;
    p->Dr = d->d_rope;
    p->Dv = d->d_v;
    p->H = d->n_heads;
    p->kv_need = causal ? (long)q_offset + s_q : s_kv;
    p->kv_pad = (p->kv_need + 127) / 128 * 128;
    // SIMT register limits of the attention kernel
    if (!absorbed && (p->Dn + p->Dr > 640 || p->Dv > 512)) return MLA_ERR_UNSUPPORTED;
    if (absorbed && (p->Dk + p->Dr > 640 || p->Dk > 512)) return MLA_ERR_UNSUPPORTED;
    p->tc = false;
    if (dt == MLA_BF16 && g_path_override != 1 && p->kv_need >= 1) {
        // the absorbed form's per-head GEMMs tile the query rows by 128
        p->tc = absorbed ? tc_absorbed_supported(p->Dk, p->Dn, p->Dr, p->Dv) && (s_q >= 128 || 128 % s_q == 0)
                         : tc_explicit_supported(p->Dk, p->Dn, p->Dr, p->Dv);
    }
    p->tin = ty_of(dt);
    p->tmid = p->tc ? TY_F16 : TY_F32;
    return MLA_OK;
}

struct PrefillWs {
    void *chat, *kpe, *qpe, *k, *v, *qabs, *olat, *w16;
    float2 *rtab;
    size_t bytes;
};

// RoPE table positions of a prefill call: keys [0, kv_need) and queries
// [q_offset, q_offset + s_q) (beyond kv_need only for non-causal calls).
long rope_positions(const Prefill &p) { return std::max(p.kv_need, (long)p.q_offset + p.s_q); }

// `fused`: the explicit form with the K/V reconstruction inside the attention kernel
// (no per-shard K_nope / V^T).
PrefillWs prefill_ws(const Prefill &p, bool absorbed, void *base, bool fused_kv = false) {
    Carve c;
    c.base = (char *)base;
    PrefillWs w{};
    const size_t es = ty_size(p.tmid);
    w.chat = c.take((size_t)p.B * p.kv_pad * p.Dk * es);
    w.kpe = c.take((size_t)p.B * p.kv_pad * p.Dr * es);
    const bool fused = p.tc && !absorbed;   // the explicit tensor-core path
    w.qpe = c.take((size_t)p.B * p.s_q * p.head_count * p.Dr * es);
    w.rtab = (float2 *)c.take((size_t)rope_positions(p) * (p.Dr / 2) * sizeof(float2));
    // fp16 W_kv_b rows: all heads of the call (explicit), one shard (absorbed transposes)
    if (p.tc) w.w16 = c.take((size_t)(fused ? p.head_count : p.hs) * (p.Dn + p.Dv) * p.Dk * 2);
    if (fused_kv) {
        // nothing per shard: K_nope and V^T tiles live only in shared memory
    } else if (!absorbed) {
        // per-shard K_nope and V (tensor-core path: V stored transposed)
        w.k = c.take((size_t)p.B * p.hs * p.kv_pad * p.Dn * es);
        w.v = c.take((size_t)p.B * p.hs * p.kv_pad * p.Dv * es);
    } else {
        // per-shard absorbed intermediates: q_abs and the latent accumulator, d_kv wide
        w.qabs = c.take((size_t)p.B * p.s_q * p.hs * p.Dk * es);
        w.olat = c.take((size_t)p.B * p.s_q * p.hs * p.Dk * es);
    }
    w.bytes = align_up(c.off, 256);
    return w;
}

mla_status prefill_common_checks(const Prefill &p, bool absorbed, const void *q_nope, const void *q_pe,
                                 const void *c_kv, const void *k_pe, const void *w_kv_b, const void *rms_w,
                                 void *out, float *lse, void *workspace, size_t workspace_bytes,
                                 bool fused_kv = false) {
    const size_t es = ty_size(p.tin);
    const void *ptrs[] = {q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse};
    for (const void *q : ptrs)
        if (!q) return MLA_ERR_NULL;
    for (const void *q : ptrs)
        if (!aligned16(q)) return MLA_ERR_ALIGN;
    PrefillWs w = prefill_ws(p, absorbed, nullptr, fused_kv);
    if (workspace_bytes < w.bytes) return MLA_ERR_WORKSPACE;
    if (w.bytes && !workspace) return MLA_ERR_NULL;
    if (workspace && !aligned16(workspace)) return MLA_ERR_ALIGN;
    size_t nq = (size_t)p.B * p.s_q * p.head_count;
    Range in[] = {rng(q_nope, nq * p.Dn * es),
                  rng(q_pe, nq * p.Dr * es),
                  rng(c_kv, (size_t)p.B * p.s_kv * p.Dk * es),
                  rng(k_pe, (size_t)p.B * p.s_kv * p.Dr * es),
                  rng(w_kv_b, (size_t)p.H * (p.Dn + p.Dv) * p.Dk * es),
                  rng(rms_w, (size_t)p.Dk * es)};
    Range outs[] = {rng(out, nq * p.Dv * es), rng(lse, nq * 4), rng(workspace, w.bytes)};
    return check_alias(in, 6, outs, 3);
}

// Common first steps of both prefill forms: normalised latent, rotated k_pe and q_pe.
mla_status prefill_prep(const Prefill &p, bool absorbed, const mla_dims *d, const void *q_pe, const void *c_kv,
                        const void *k_pe, const void *w_kv_b, const void *rms_w, const PrefillWs &w,
                        cudaStream_t st) {
    if (p.tc && !absorbed) {
        // one launch: table, normalised latent, rotated k_pe and q_pe, fp16 weight copy
        const long Dh = p.Dn + p.Dv;
        return cuda_status(launch_prep_tc(p.B, p.s_kv, (int)p.kv_need, (int)p.kv_pad, p.Dk, rope_positions(p),
                                          d->rope_base, c_kv, k_pe, rms_w, d->rms_eps, w.rtab, w.chat, w.kpe,
                                          (const char *)w_kv_b + (size_t)p.head_begin * Dh * p.Dk * 2, w.w16,
                                          (long)p.head_count * Dh * p.Dk, q_pe, w.qpe, p.s_q, p.q_offset,
                                          p.head_count, st));
    }
    MLA_TRY(launch_rope_table(0, rope_positions(p), p.Dr, d->rope_base, w.rtab, st));
    MLA_TRY(launch_latent_prep(p.tin, p.tmid, p.B, p.s_kv, (int)p.kv_need, (int)p.kv_pad, p.Dk, p.Dr, c_kv, k_pe,
                               rms_w, d->rms_eps, w.rtab, w.chat, w.kpe, st));
    long rows = (long)p.B * p.s_q * p.head_count;
    MLA_TRY(launch_rope_rows(p.tin, p.tmid, rows, p.Dr, q_pe, p.q_offset, p.head_count, p.s_q, w.rtab, 0, w.qpe,
                             st));
    return MLA_OK;
}

// ------------------------------------------------------ explicit, SIMT ----
mla_status explicit_simt(const Prefill &p, float scale, const void *q_nope, const void *w_kv_b, void *out,
                         float *lse, const PrefillWs &w, cudaStream_t st) {
    const long Dh = p.Dn + p.Dv;
    const long kvn = p.kv_need;
    const size_t ein = ty_size(p.tin);
    for (int s = 0; s < p.n_shards; ++s) {
        int h0 = s * p.hs;                        // local head index of the shard
        int nh = std::min(p.hs, p.head_count - h0);
        long hg = p.head_begin + h0;              // global head index
        // K_ws [B][hs][kv][Dn] and V_ws [B][hs][kv][Dv] = chat[b] x W(head rows)^T
        for (int part = 0; part < 2; ++part) {
            GemmArgs g{};
            int Dpart = part == 0 ? p.Dn : p.Dv;
            g.M = (int)kvn;
            g.N = Dpart;
            g.K = p.Dk;
            g.nzb = p.B;
            g.nzh = nh;
            g.A = w.chat;
            g.ta = p.tmid;
            g.a_zb = p.kv_pad * p.Dk;
            g.a_m = p.Dk;
            g.a_k = 1;
            g.B = (const char *)w_kv_b + ((hg * Dh + (part ? p.Dn : 0)) * p.Dk) * ein;
            g.tb = p.tin;
            g.b_zh = Dh * p.Dk;
            g.b_n = p.Dk;
            g.b_k = 1;
            g.C = part == 0 ? w.k : w.v;
            g.tc = p.tmid;
            g.c_zh = kvn * Dpart;
            g.c_zb = (long)p.hs * g.c_zh;
            g.c_m = Dpart;
            g.c_n = 1;
            MLA_TRY(launch_gemm_simt(g, st));
        }
        AttnArgs a{};
        a.n_b = p.B;
        a.n_h = nh;
        a.n_rows = p.s_q;
        a.D1 = p.Dn;
        a.D2 = p.Dr;
        a.Dv = p.Dv;
        a.q1 = (const char *)q_nope + (size_t)h0 * p.Dn * ein;
        a.tq1 = p.tin;
        a.q1_b = (long)p.s_q * p.head_count * p.Dn;
        a.q1_h = p.Dn;
        a.q1_r = (long)p.head_count * p.Dn;
        a.q2 = (const char *)w.qpe + (size_t)h0 * p.Dr * ty_size(p.tmid);
        a.tq2 = p.tmid;
        a.q2_b = (long)p.s_q * p.head_count * p.Dr;
        a.q2_h = p.Dr;
        a.q2_r = (long)p.head_count * p.Dr;
        a.k1 = w.k;
        a.tk1 = p.tmid;
        a.k1_b = (long)p.hs * kvn * p.Dn;
        a.k1_h = kvn * p.Dn;
        a.k1_r = p.Dn;
        a.k2 = w.kpe;
        a.tk2 = p.tmid;
        a.k2_b = p.kv_pad * p.Dr;
        a.k2_r = p.Dr;
        a.v = w.v;
        a.tv = p.tmid;
        a.v_b = (long)p.hs * kvn * p.Dv;
        a.v_h = kvn * p.Dv;
        a.v_r = p.Dv;
        a.kv_len = kvn;
        a.n_splits = 1;
        a.chunk = kvn;
        a.causal = p.causal;
        a.pos0 = p.q_offset;
        a.scale = scale;
        a.out = (char *)out + (size_t)h0 * p.Dv * ein;
        a.to = p.tin;
        a.o_b = (long)p.s_q * p.head_count * p.Dv;
        a.o_h = p.Dv;
        a.o_r = (long)p.head_count * p.Dv;
        a.lse = lse + (size_t)h0 * p.s_q;
        a.l_b = (long)p.head_count * p.s_q;
        a.l_h = p.s_q;
        a.l_r = 1;
        MLA_TRY(launch_attn_simt(a, st));
    }
    return MLA_OK;
}

// ------------------------------------------------------ absorbed, SIMT ----
mla_status absorbed_simt(const Prefill &p, float scale, const void *q_nope, const void *w_kv_b, void *out,
                         float *lse, const PrefillWs &w, cudaStream_t st) {
    const long Dh = p.Dn + p.Dv;
    const size_t ein = ty_size(p.tin);
    for (int s = 0; s < p.n_shards; ++s) {
        int h0 = s * p.hs;
        int nh = std::min(p.hs, p.head_count - h0);
        long hg = p.head_begin + h0;
        // absorb: q_abs[b][i][hl][k] = sum_d q_nope[b][i][h0+hl][d] * W_K(h)[d][k]
        GemmArgs g{};
        g.M = p.s_q;
        g.N = p.Dk;
        g.K = p.Dn;
        g.nzb = p.B;
        g.nzh = nh;
        g.A = (const char *)q_nope + (size_t)h0 * p.Dn * ein;
        g.ta = p.tin;
        g.a_zb = (long)p.s_q * p.head_count * p.Dn;
        g.a_zh = p.Dn;
        g.a_m = (long)p.head_count * p.Dn;
        g.a_k = 1;
        g.B = (const char *)w_kv_b + (size_t)(hg * Dh * p.Dk) * ein;
        g.tb = p.tin;
        g.b_zh = Dh * p.Dk;
        g.b_n = 1;
        g.b_k = p.Dk;
        g.C = w.qabs;
        g.tc = p.tmid;
        g.c_zb = (long)p.s_q * p.hs * p.Dk;
        g.c_zh = p.Dk;
        g.c_m = (long)p.hs * p.Dk;
        g.c_n = 1;
        MLA_TRY(launch_gemm_simt(g, st));
        // latent attention: scores over [q_abs ; q_pe] . [chat ; kpe], values chat
        AttnArgs a{};
        a.n_b = p.B;
        a.n_h = nh;
        a.n_rows = p.s_q;
        a.D1 = p.Dk;
        a.D2 = p.Dr;
        a.Dv = p.Dk;
        a.q1 = w.qabs;
        a.tq1 = p.tmid;
        a.q1_b = (long)p.s_q * p.hs * p.Dk;
        a.q1_h = p.Dk;
        a.q1_r = (long)p.hs * p.Dk;
        a.q2 = (const char *)w.qpe + (size_t)h0 * p.Dr * ty_size(p.tmid);
        a.tq2 = p.tmid;
        a.q2_b = (long)p.s_q * p.head_count * p.Dr;
        a.q2_h = p.Dr;
        a.q2_r = (long)p.head_count * p.Dr;
        a.k1 = w.chat;
        a.tk1 = p.tmid;
        a.k1_b = p.kv_pad * p.Dk;
        a.k1_r = p.Dk;
        a.k2 = w.kpe;
        a.tk2 = p.tmid;
        a.k2_b = p.kv_pad * p.Dr;
        a.k2_r = p.Dr;
        a.v = w.chat;
        a.tv = p.tmid;
        a.v_b = p.kv_pad * p.Dk;
        a.v_r = p.Dk;
        a.kv_len = p.kv_need;
        a.n_splits = 1;
        a.chunk = p.kv_need;
        a.causal = p.causal;
        a.pos0 = p.q_offset;
        a.scale = scale;
        a.out = w.olat;
        a.to = p.tmid;
        a.o_b = (long)p.s_q * p.hs * p.Dk;
        a.o_h = p.Dk;
        a.o_r = (long)p.hs * p.Dk;
        a.lse = lse + (size_t)h0 * p.s_q;
        a.l_b = (long)p.head_count * p.s_q;
        a.l_h = p.s_q;
        a.l_r = 1;
        MLA_TRY(launch_attn_simt(a, st));
        // un-absorb: out[b][i][h0+hl][d] = sum_k o_lat[b][i][hl][k] * W_V(h)[d][k]
        GemmArgs u{};
        u.M = p.s_q;
        u.N = p.Dv;
        u.K = p.Dk;
        u.nzb = p.B;
        u.nzh = nh;
        u.A = w.olat;
        u.ta = p.tmid;
        u.a_zb = (long)p.s_q * p.hs * p.Dk;
        u.a_zh = p.Dk;
        u.a_m = (long)p.hs * p.Dk;
        u.a_k = 1;
        u.B = (const char *)w_kv_b + (size_t)((hg * Dh + p.Dn) * p.Dk) * ein;
        u.tb = p.tin;
        u.b_zh = Dh * p.Dk;
        u.b_n = p.Dk;
        u.b_k = 1;
        u.C = (char *)out + (size_t)h0 * p.Dv * ein;
        u.tc = p.tin;
        u.c_zb = (long)p.s_q * p.head_count * p.Dv;
        u.c_zh = p.Dv;
        u.c_m = (long)p.head_count * p.Dv;
        u.c_n = 1;
        MLA_TRY(launch_gemm_simt(u, st));
    }
    return MLA_OK;
}

// ------------------------------------------------------------ decode shapes ----
struct Decode {
    int B, L, n, H, Dk, Dn, Dr, Dv;
    int g;   // latent shards (TPLA); 1 for plain latent decode
    long chunk;
    bool tc;
    int tin, tmid;
};

mla_status decode_shape(const mla_dims *d, mla_dtype dt, int B, int kv_len, int n_splits, Decode *p, int g = 1) {
    mla_status st = check_dims(d);
    if (st != MLA_OK) return st;
    if (!valid_dtype(dt)) return MLA_ERR_DTYPE;
    if (B < 0 || kv_len < 1 || n_splits < 1 || n_splits > 256) return MLA_ERR_SHAPE;
    if (g < 1 || g > 16 || d->d_kv % g) return MLA_ERR_SHAPE;
    p->g = g;
    p->B = B;
    p->L = kv_len;
    p->n = n_splits;
    p->H = d->n_heads;
    p->Dk = d->d_kv;
    p->Dn = d->d_nope;
    p->Dr = d->d_rope;
    p->Dv = d->d_v;
    p->chunk = ((long)kv_len + n_splits - 1) / n_splits;
    if (p->Dk + p->Dr > 640 || p->Dk > 512) return MLA_ERR_UNSUPPORTED;
    p->tc = dt == MLA_BF16 && g_path_override != 1 && tc_decode_supported(p->Dk, p->Dn, p->Dr, p->Dv, p->H * g);
    p->tin = ty_of(dt);
    p->tmid = p->tc ? TY_F16 : TY_F32;
    return MLA_OK;
}

struct DecodeWs {
    void *qabs, *qpe, *olat;
    void *qx, *qpx;   // TPLA: the g query rows of every head
    float *po, *pl;
    float2 *rtab;
    size_t bytes;
};

DecodeWs decode_ws(const Decode &p, void *base, bool own_partials) {
    Carve c;
    c.base = (char *)base;
    DecodeWs w{};
    const size_t es = ty_size(p.tmid);
    size_t rows = (size_t)p.B * p.H;
    w.qabs = c.take(rows * p.Dk * es);
    w.qpe = c.take(rows * p.Dr * es);
    w.olat = c.take(rows * p.Dk * es);
    w.rtab = (float2 *)c.take((size_t)(p.Dr / 2) * sizeof(float2));
    if (p.g > 1) {
        w.qx = c.take(rows * p.g * p.Dk * es);
        w.qpx = c.take(rows * p.g * p.Dr * es);
    }
    if (own_partials) {
        w.po = (float *)c.take((size_t)p.n * rows * p.g * p.Dk * 4);
        w.pl = (float *)c.take((size_t)p.n * rows * p.g * 4);
    }
    w.bytes = align_up(c.off, 256);
    return w;
}

mla_status decode_simt(const Decode &p, float scale, const mla_dims *d, const void *q_nope, const void *q_pe,
                       const void *c_cache, const void *kpe_cache, const void *w_kv_b, void *out, float *lse,
                       float *po, float *pl, const DecodeWs &w, cudaStream_t st) {
    const size_t ein = ty_size(p.tin);
    const long Dh = p.Dn + p.Dv;
    long rows = (long)p.B * p.H;
    MLA_TRY(launch_rope_rows_at(p.tin, p.tmid, rows, p.Dr, q_pe, p.L - 1, d->rope_base, w.qpe, st));
    GemmArgs g{};
    g.M = p.B;
    g.N = p.Dk;
    g.K = p.Dn;
    g.nzb = 1;
    g.nzh = p.H;
    g.A = q_nope;
    g.ta = p.tin;
    g.a_zh = p.Dn;
    g.a_m = (long)p.H * p.Dn;
    g.a_k = 1;
    g.B = w_kv_b;
    g.tb = p.tin;
    g.b_zh = Dh * p.Dk;
    g.b_n = 1;
    g.b_k = p.Dk;
    g.C = w.qabs;
    g.tc = p.tmid;
    g.c_zh = p.Dk;
    g.c_m = (long)p.H * p.Dk;
    g.c_n = 1;
    MLA_TRY(launch_gemm_simt(g, st));
    // TPLA: g query rows per head, each seeing only its shard of the latent
    const int HX = p.H * p.g;
    if (p.g > 1) MLA_TRY(launch_tpla_expand(p.tmid, p.B, p.H, p.g, p.Dk, p.Dr, w.qabs, w.qpe, w.qx, w.qpx, st));
    AttnArgs a{};
    a.n_b = p.B;
    a.n_h = 1;
    a.n_rows = HX;
    a.D1 = p.Dk;
    a.D2 = p.Dr;
    a.Dv = p.Dk;
    a.q1 = p.g > 1 ? w.qx : w.qabs;
    a.tq1 = p.tmid;
    a.q1_b = (long)HX * p.Dk;
    a.q1_r = p.Dk;
    a.q2 = p.g > 1 ? w.qpx : w.qpe;
    a.tq2 = p.tmid;
    a.q2_b = (long)HX * p.Dr;
    a.q2_r = p.Dr;
    a.k1 = c_cache;
    a.tk1 = p.tin;
    a.k1_b = (long)p.L * p.Dk;
    a.k1_r = p.Dk;
    a.k2 = kpe_cache;
    a.tk2 = p.tin;
    a.k2_b = (long)p.L * p.Dr;
    a.k2_r = p.Dr;
    a.v = c_cache;
    a.tv = p.tin;
    a.v_b = (long)p.L * p.Dk;
    a.v_r = p.Dk;
    a.kv_len = p.L;
    a.n_splits = p.n;
    a.chunk = p.chunk;
    a.causal = 0;
    a.pos0 = p.L - 1;
    a.scale = scale;
    a.part_out = po;
    a.po_s = rows * p.g * p.Dk;
    a.po_b = (long)HX * p.Dk;
    a.po_r = p.Dk;
    a.part_lse = pl;
    a.pl_s = rows * p.g;
    a.pl_b = HX;
    a.pl_r = 1;
    MLA_TRY(launch_attn_simt(a, st));
    if (p.g > 1)
        MLA_TRY(launch_tpla_combine(p.tmid, p.n, p.B, p.H, p.g, p.Dk, po, pl, w.olat, lse, st));
    else
        MLA_TRY(launch_lse_combine(p.tmid, p.n, rows, p.Dk, po, pl, w.olat, lse, st));
    GemmArgs u{};
    u.M = p.B;
    u.N = p.Dv;
    u.K = p.Dk;
    u.nzb = 1;
    u.nzh = p.H;
    u.A = w.olat;
    u.ta = p.tmid;
    u.a_zh = p.Dk;
    u.a_m = (long)p.H * p.Dk;
    u.a_k = 1;
    u.B = (const char *)w_kv_b + (size_t)p.Dn * p.Dk * ein;
    u.tb = p.tin;
    u.b_zh = Dh * p.Dk;
    u.b_n = p.Dk;
    u.b_k = 1;
    u.C = out;
    u.tc = p.tin;
    u.c_zh = p.Dv;
    u.c_m = (long)p.H * p.Dv;
    u.c_n = 1;
    MLA_TRY(launch_gemm_simt(u, st));
    return MLA_OK;
}

// Query tiles of a head that share each rebuilt key tile in the fused kernel.
int fused_cluster(const Prefill &p) {
    if (g_fused_cluster == 4 || g_fused_cluster == 8) return g_fused_cluster;
    return (p.s_q + 127) / 128 >= 8 ? 8 : 4;
}

mla_status prefill_entry(bool absorbed, const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                         int q_offset, int causal, int head_begin, int head_count, int head_shard, const void *q_nope,
                         const void *q_pe, const void *c_kv, const void *k_pe, const void *w_kv_b, const void *rms_w,
                         void *out, float *lse, void *workspace, size_t workspace_bytes, void *cuda_stream,
                         bool fused_kv = false) {
    Prefill p;
    mla_status st = prefill_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, head_begin, head_count, head_shard,
                                  absorbed, &p);
    if (st != MLA_OK) return st;
    if (fused_kv && !p.tc) return MLA_ERR_UNSUPPORTED;   // the fused kernel is the tensor-core path only
    if (B == 0 || s_q == 0 || head_count == 0) return MLA_OK;
    st = prefill_common_checks(p, absorbed, q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, workspace,
                               workspace_bytes, fused_kv);
    if (st != MLA_OK) return st;
    cudaStream_t cs = (cudaStream_t)cuda_stream;
    PrefillWs w = prefill_ws(p, absorbed, workspace, fused_kv);
    float scale = scale_of(dims);
    st = prefill_prep(p, absorbed, dims, q_pe, c_kv, k_pe, w_kv_b, rms_w, w, cs);
    if (st != MLA_OK) return st;
    g_last_path = p.tc ? (fused_kv ? 3 : 2) : 1;
    if (p.tc) {
        TcPrefill t{p.B, p.s_q, p.s_kv, p.q_offset, p.causal, p.head_begin, p.head_count, p.hs, p.n_shards,
                    p.Dk, p.Dn, p.Dr, p.Dv, p.H, p.kv_need, scale};
        if (fused_kv)
            return cuda_status(tc_fused_prefill(t, q_nope, out, lse, w.chat, w.kpe, w.qpe, w.w16, fused_cluster(p), cs));
        cudaError_t e = absorbed ? tc_absorbed_prefill(t, q_nope, w_kv_b, out, lse, w.chat, w.kpe, w.qpe, w.qabs,
                                                       w.olat, w.w16, cs)
                                 : tc_explicit_prefill(t, q_nope, w_kv_b, out, lse, w.chat, w.kpe, w.qpe, w.k,
                                                       w.v, w.w16, cs);
        return cuda_status(e);
    }
    return absorbed ? absorbed_simt(p, scale, q_nope, w_kv_b, out, lse, w, cs)
                    : explicit_simt(p, scale, q_nope, w_kv_b, out, lse, w, cs);
}

// ------------------------------------------------------------------ backward ----
struct BwdWs {
    PrefillWs f;   // the forward's recomputed intermediates (K / V per head shard)
    float *D, *dqr, *dK, *dV, *dkr, *dkr_acc, *dchat, *rms_part;
    void *qn16, *do16, *dkvt, *chatT, *wT;   // tensor-core path
    size_t bytes;
};

BwdWs bwd_ws(const Prefill &p, void *base) {
    BwdWs w{};
    w.f = prefill_ws(p, false, base);
    Carve c;
    c.base = (char *)base;
    c.off = w.f.bytes;
    const size_t nq = (size_t)p.B * p.s_q * p.head_count;
    w.D = (float *)c.take(nq * 4);
    w.dqr = (float *)c.take(nq * p.Dr * 4);
    if (p.tc) {
        w.qn16 = c.take(nq * p.Dn * 2);
        w.do16 = c.take(nq * p.Dv * 2);
        w.dkvt = c.take((size_t)p.hs * (p.Dn + p.Dv) * p.B * p.kv_pad * 2);
        w.chatT = c.take((size_t)p.Dk * p.B * p.kv_pad * 2);
        w.wT = c.take((size_t)p.Dk * p.head_count * (p.Dn + p.Dv) * 2);
    } else {
        w.dK = (float *)c.take((size_t)p.B * p.hs * p.kv_pad * p.Dn * 4);
        w.dV = (float *)c.take((size_t)p.B * p.hs * p.kv_pad * p.Dv * 4);
    }
    w.dkr = (float *)c.take((size_t)p.B * p.hs * p.kv_pad * p.Dr * 4);
    w.dkr_acc = (float *)c.take((size_t)p.B * p.kv_pad * p.Dr * 4);
    w.dchat = (float *)c.take((size_t)p.B * p.kv_pad * p.Dk * 4);
    w.rms_part = (float *)c.take(rms_bwd_parts(p.s_kv) * p.Dk * 4);
    w.bytes = align_up(c.off, 256);
    return w;
}

mla_status bwd_shape(const mla_dims *d, mla_dtype dt, int B, int s_q, int s_kv, int q_offset, int causal,
                     int head_begin, int head_count, int head_shard, Prefill *p) {
    mla_status st = prefill_shape(d, dt, B, s_q, s_kv, q_offset, causal, head_begin, head_count, head_shard, false, p);
    if (st != MLA_OK) return st;
    if (!p->tc) {   // the CUDA-core backward keeps fp32 intermediates
        if (!bwd_simt_supported(p->Dn, p->Dr, p->Dv)) return MLA_ERR_UNSUPPORTED;
        p->tmid = TY_F32;
    }
    return MLA_OK;
}

// The backward on the tensor cores (bf16 at the DeepSeek dimensions): the forward's prep
// and per-shard K / V reconstruction again, the two attention-backward kernels, the
// weight gradients dW = [dK_nope^T ; dV^T] chat (summed over the batch by running the
// GEMM's k over batch and keys) and dchat += dKV W (W^T as the B operand), then the
// rotations' transposes and the RMSNorm backward.
mla_status bwd_tc(const Prefill &p, const mla_dims *d, float scale, const void *q_nope, const void *q_pe,
                  const void *c_kv, const void *k_pe, const void *w_kv_b, const void *rms_w, const void *out,
                  const float *lse, const void *dout, void *dq_nope, void *dq_pe, void *dc_kv, void *dk_pe,
                  float *dw_kv_b, float *drms_w, const BwdWs &w, cudaStream_t st) {
    const long Dh = p.Dn + p.Dv, kvn = p.kv_need, BK = (long)p.B * p.kv_pad;
    const size_t ein = ty_size(p.tin);
    mla_status ms = prefill_prep(p, false, d, q_pe, c_kv, k_pe, w_kv_b, rms_w, w.f, st);
    if (ms != MLA_OK) return ms;
    MLA_TRY(launch_bwd_prep_tc(p.B, p.s_q, p.head_count, q_nope, dout, out, w.qn16, w.do16, w.D, st));
    MLA_TRY(launch_transpose16(BK, p.Dk, w.f.chat, w.chatT, st));                       // chat^T [Dk][B*kv_pad]
    MLA_TRY(launch_transpose16((long)p.head_count * Dh, p.Dk, w.f.w16, w.wT, st));      // W^T [Dk][hc*Dh]
    TcPrefill t{p.B, p.s_q, p.s_kv, p.q_offset, p.causal, p.head_begin, p.head_count, p.hs, p.n_shards,
                p.Dk, p.Dn, p.Dr, p.Dv, p.H, p.kv_need, scale};
    for (int s = 0; s < p.n_shards; ++s) {
        const int h0 = s * p.hs, nh = std::min(p.hs, p.head_count - h0);
        MLA_TRY(tc_reconstruct(t, h0, nh, w.f.chat, w.f.w16, w.f.k, w.f.v, st));
        MLA_TRY(tc_bwd_attn(t, h0, nh, w.f.k, w.f.v, w.f.kpe, w.qn16, w.f.qpe, w.do16, lse, w.D, dq_nope, w.dqr,
                            w.dkvt, w.dkr, st));
        // dW rows of the shard's heads: [nh*Dh][Dk] = dKV^T [nh*Dh][B*kv_pad] x chat^T [Dk][B*kv_pad]^T,
        // the Dk output columns as a batch of 128-column blocks (single-CTA tiles: four times
        // the tiles of one 256-wide problem)
        const int nb = p.Dk / 128;
        TmaOperand A{w.dkvt, BK, (long)nh * Dh, 1, BK * 2, 0, (int)(nh * Dh), 0, 0};
        TmaOperand Bc{w.chatT, BK, 128, nb, BK * 2, 128 * BK * 2, 128, 0, 1};
        MLA_TRY(tc_gemm(A, Bc, (int)(nh * Dh), 128, (int)BK, nb, true,
                        dw_kv_b + (size_t)(p.head_begin + h0) * Dh * p.Dk, p.Dk, 1, 128, 2, st));
        // dchat [B*kv_pad][Dk] += dKV [B*kv_pad][nh*Dh] x W [nh*Dh][Dk], the latent columns as a
        // batch of 128-column blocks (W^T rows 128 c .. 128 c + 127 for block c)
        TmaOperand Am{w.dkvt, BK, (long)nh * Dh, 1, BK * 2, 0, (int)BK, 0, 0};   // m-major: rows are k
        TmaOperand Bw{(const char *)w.wT + (size_t)h0 * Dh * 2, (long)nh * Dh, 128, nb, (long)p.head_count * Dh * 2,
                      (long)128 * p.head_count * Dh * 2, 128, 0, 1};
        MLA_TRY(tc_gemm(Am, Bw, (int)BK, 128, (int)(nh * Dh), nb, true, w.dchat, p.Dk, 1, 128, 2, st, true, s > 0));
        MLA_TRY(launch_head_sum(p.B, nh, p.kv_pad, p.Dr, p.kv_pad, w.dkr, w.dkr_acc, s > 0, st));
    }
    const long nq = (long)p.B * p.s_q * p.head_count;
    MLA_TRY(launch_rope_inv(nq, p.Dr, w.dqr, p.Dr, p.q_offset, p.head_count, p.s_q, 1L << 40, w.f.rtab, dq_pe,
                            p.tin, p.Dr, st));
    for (int b = 0; b < p.B; ++b) {
        MLA_TRY(launch_rope_inv(p.s_kv, p.Dr, w.dkr_acc + (size_t)b * p.kv_pad * p.Dr, p.Dr, 0, 1, 1L << 40, kvn,
                                w.f.rtab, (char *)dk_pe + (size_t)b * p.s_kv * p.Dr * ein, p.tin, p.Dr, st));
        MLA_TRY(launch_rms_bwd_f32dy(p.tin, kvn, p.s_kv, p.Dk, d->rms_eps, (const char *)c_kv + (size_t)b * p.s_kv * p.Dk * ein,
                                     rms_w, w.dchat + (size_t)b * p.kv_pad * p.Dk,
                                     (char *)dc_kv + (size_t)b * p.s_kv * p.Dk * ein, drms_w, b > 0, w.rms_part, st));
    }
    return MLA_OK;
}

// The backward on the CUDA-core kernels: recompute the forward's normalised latent,
// rotated bands and per-shard K / V, then per head shard the attention backward, the
// weight gradients (dW = dKV^T chat, summed over the batch) and the latent gradient
// (dchat += dKV W); finally the rotations' transposes and the RMSNorm backward.
mla_status bwd_simt(const Prefill &p, const mla_dims *d, float scale, const void *q_nope, const void *q_pe,
                    const void *c_kv, const void *k_pe, const void *w_kv_b, const void *rms_w, const void *out,
                    const float *lse, const void *dout, void *dq_nope, void *dq_pe, void *dc_kv, void *dk_pe,
                    float *dw_kv_b, float *drms_w, const BwdWs &w, cudaStream_t st) {
    const long Dh = p.Dn + p.Dv, kvn = p.kv_need;
    const size_t ein = ty_size(p.tin);
    mla_status ms = prefill_prep(p, false, d, q_pe, c_kv, k_pe, w_kv_b, rms_w, w.f, st);
    if (ms != MLA_OK) return ms;
    MLA_TRY(launch_bwd_rowdot(p.tin, p.B, p.s_q, p.head_count, p.Dv, dout, out, w.D, st));
    for (int s = 0; s < p.n_shards; ++s) {
        const int h0 = s * p.hs, nh = std::min(p.hs, p.head_count - h0);
        const long hg = p.head_begin + h0;
        for (int part = 0; part < 2; ++part) {   // this shard's K_nope, V (fp32)
            GemmArgs g{};
            const int Dp = part == 0 ? p.Dn : p.Dv;
            g.M = (int)kvn; g.N = Dp; g.K = p.Dk; g.nzb = p.B; g.nzh = nh;
            g.A = w.f.chat; g.ta = p.tmid; g.a_zb = p.kv_pad * p.Dk; g.a_m = p.Dk; g.a_k = 1;
            g.B = (const char *)w_kv_b + ((hg * Dh + (part ? p.Dn : 0)) * p.Dk) * ein;
            g.tb = p.tin; g.b_zh = Dh * p.Dk; g.b_n = p.Dk; g.b_k = 1;
            g.C = part == 0 ? w.f.k : w.f.v; g.tc = p.tmid; g.c_zh = kvn * Dp; g.c_zb = (long)p.hs * g.c_zh;
            g.c_m = Dp; g.c_n = 1;
            MLA_TRY(launch_gemm_simt(g, st));
        }
        BwdSimtArgs a{};
        a.B = p.B; a.s_q = p.s_q; a.hc = p.head_count; a.h0 = h0; a.nh = nh;
        a.Dn = p.Dn; a.Dr = p.Dr; a.Dv = p.Dv; a.kv = kvn; a.kv_pad = p.kv_pad;
        a.causal = p.causal; a.q_off = p.q_offset; a.scale = scale; a.ty = p.tin;
        a.q_nope = q_nope; a.qr = (const float *)w.f.qpe; a.kr = (const float *)w.f.kpe;
        a.K = (const float *)w.f.k; a.V = (const float *)w.f.v;
        a.k_b = (long)p.hs * kvn * p.Dn; a.k_h = kvn * p.Dn; a.v_b = (long)p.hs * kvn * p.Dv; a.v_h = kvn * p.Dv;
        a.lse = lse; a.D = w.D; a.dout = dout; a.dq_nope = dq_nope; a.dqr = w.dqr;
        a.dK = w.dK; a.dV = w.dV; a.dkr = w.dkr;
        MLA_TRY(launch_attn_bwd_simt(a, st));
        // dW_K(h) = dK^T chat and dW_V(h) = dV^T chat, summed over the batch
        for (int part = 0; part < 2; ++part)
            for (int b = 0; b < p.B; ++b) {
                GemmArgs g{};
                const int Dp = part == 0 ? p.Dn : p.Dv;
                g.M = Dp; g.N = p.Dk; g.K = (int)kvn; g.nzb = 1; g.nzh = nh;
                g.A = (part == 0 ? w.dK : w.dV) + (size_t)b * nh * kvn * Dp; g.ta = TY_F32;
                g.a_zh = kvn * Dp; g.a_m = 1; g.a_k = Dp;
                g.B = (const char *)w.f.chat + (size_t)b * p.kv_pad * p.Dk * 4; g.tb = p.tmid;
                g.b_n = 1; g.b_k = p.Dk;
                g.C = dw_kv_b + (size_t)(hg * Dh + (part ? p.Dn : 0)) * p.Dk; g.tc = TY_F32;
                g.c_zh = Dh * p.Dk; g.c_m = p.Dk; g.c_n = 1;
                g.accumulate = b > 0;
                MLA_TRY(launch_gemm_simt(g, st));
            }
        // dchat += dK W_K(h) + dV W_V(h), head by head (a fixed order)
        for (int hl = 0; hl < nh; ++hl)
            for (int part = 0; part < 2; ++part) {
                GemmArgs g{};
                const int Dp = part == 0 ? p.Dn : p.Dv;
                g.M = (int)kvn; g.N = p.Dk; g.K = Dp; g.nzb = p.B; g.nzh = 1;
                g.A = (part == 0 ? w.dK : w.dV) + (size_t)hl * kvn * Dp; g.ta = TY_F32;
                g.a_zb = (long)nh * kvn * Dp; g.a_m = Dp; g.a_k = 1;
                g.B = (const char *)w_kv_b + (((hg + hl) * Dh + (part ? p.Dn : 0)) * p.Dk) * ein; g.tb = p.tin;
                g.b_n = 1; g.b_k = p.Dk;
                g.C = w.dchat; g.tc = TY_F32; g.c_zb = p.kv_pad * p.Dk; g.c_m = p.Dk; g.c_n = 1;
                g.accumulate = !(s == 0 && hl == 0 && part == 0);
                MLA_TRY(launch_gemm_simt(g, st));
            }
        MLA_TRY(launch_head_sum(p.B, nh, kvn, p.Dr, p.kv_pad, w.dkr, w.dkr_acc, s > 0, st));
    }
    // the rotations' transposes: dq_pe at the query positions, dk_pe at the keys (zeros past kv_need)
    const long nq = (long)p.B * p.s_q * p.head_count;
    MLA_TRY(launch_rope_inv(nq, p.Dr, w.dqr, p.Dr, p.q_offset, p.head_count, p.s_q, 1L << 40, w.f.rtab, dq_pe,
                            p.tin, p.Dr, st));
    for (int b = 0; b < p.B; ++b) {
        MLA_TRY(launch_rope_inv(p.s_kv, p.Dr, w.dkr_acc + (size_t)b * p.kv_pad * p.Dr, p.Dr, 0, 1, 1L << 40, kvn,
                                w.f.rtab, (char *)dk_pe + (size_t)b * p.s_kv * p.Dr * ein, p.tin, p.Dr, st));
        MLA_TRY(launch_rms_bwd_f32dy(p.tin, kvn, p.s_kv, p.Dk, d->rms_eps, (const char *)c_kv + (size_t)b * p.s_kv * p.Dk * ein,
                                     rms_w, w.dchat + (size_t)b * p.kv_pad * p.Dk,
                                     (char *)dc_kv + (size_t)b * p.s_kv * p.Dk * ein, drms_w, b > 0, w.rms_part, st));
    }
    return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_latent_attn_bwd_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                     int causal, int head_count, int head_shard) {
    Prefill p;
    if (bwd_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, 0, head_count, head_shard, &p) != MLA_OK) return 0;
    if (B == 0 || s_q == 0 || head_count == 0) return 0;
    return bwd_ws(p, nullptr).bytes;
}

mla_status mla_latent_attn_bwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                               int causal, int head_begin, int head_count, int head_shard, const void *q_nope,
                               const void *q_pe, const void *c_kv, const void *k_pe, const void *w_kv_b,
                               const void *rms_w, const void *out, const float *lse, const void *dout,
                               void *dq_nope, void *dq_pe, void *dc_kv, void *dk_pe, float *dw_kv_b,
                               float *drms_w, void *workspace, size_t workspace_bytes, void *cuda_stream) {
    Prefill p;
    mla_status st = bwd_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, head_begin, head_count, head_shard, &p);
    if (st != MLA_OK) return st;
    if (B == 0 || s_q == 0 || head_count == 0) return MLA_OK;
    const void *ptrs[] = {q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, dout,
                          dq_nope, dq_pe, dc_kv, dk_pe, dw_kv_b, drms_w, workspace};
    for (const void *q : ptrs)
        if (!q) return MLA_ERR_NULL;
    for (const void *q : ptrs)
        if (!aligned16(q)) return MLA_ERR_ALIGN;
    const BwdWs wsz = bwd_ws(p, nullptr);
    if (workspace_bytes < wsz.bytes) return MLA_ERR_WORKSPACE;
    const size_t es = ty_size(p.tin), nq = (size_t)p.B * p.s_q * p.head_count;
    const size_t nw = (size_t)p.H * (p.Dn + p.Dv) * p.Dk;
    Range in[] = {rng(q_nope, nq * p.Dn * es), rng(q_pe, nq * p.Dr * es), rng(c_kv, (size_t)p.B * p.s_kv * p.Dk * es),
                  rng(k_pe, (size_t)p.B * p.s_kv * p.Dr * es), rng(w_kv_b, nw * es), rng(rms_w, (size_t)p.Dk * es),
                  rng(out, nq * p.Dv * es), rng(lse, nq * 4), rng(dout, nq * p.Dv * es)};
    Range outs[] = {rng(dq_nope, nq * p.Dn * es), rng(dq_pe, nq * p.Dr * es),
                    rng(dc_kv, (size_t)p.B * p.s_kv * p.Dk * es), rng(dk_pe, (size_t)p.B * p.s_kv * p.Dr * es),
                    rng(dw_kv_b, nw * 4), rng(drms_w, (size_t)p.Dk * 4), rng(workspace, wsz.bytes)};
    st = check_alias(in, 9, outs, 7);
    if (st != MLA_OK) return st;
    cudaStream_t cs = (cudaStream_t)cuda_stream;
    const BwdWs w = bwd_ws(p, workspace);
    g_last_path = p.tc ? 2 : 1;
    if (p.tc)
        return bwd_tc(p, dims, scale_of(dims), q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, dout, dq_nope, dq_pe,
                      dc_kv, dk_pe, dw_kv_b, drms_w, w, cs);
    return bwd_simt(p, dims, scale_of(dims), q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, dout, dq_nope, dq_pe,
                    dc_kv, dk_pe, dw_kv_b, drms_w, w, cs);
}

mla_status mla_latent_attn_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                               int causal, int head_begin, int head_count, int head_shard, const void *q_nope,
                               const void *q_pe, const void *c_kv, const void *k_pe, const void *w_kv_b,
                               const void *rms_w, void *out, float *lse, void *workspace, size_t workspace_bytes,
                               void *cuda_stream) {
    return prefill_entry(false, dims, dtype, B, s_q, s_kv, q_offset, causal, head_begin, head_count, head_shard,
                         q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, workspace, workspace_bytes, cuda_stream);
}

mla_status mla_absorbed_attn_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                 int causal, int head_begin, int head_count, int head_shard, const void *q_nope,
                                 const void *q_pe, const void *c_kv, const void *k_pe, const void *w_kv_b,
                                 const void *rms_w, void *out, float *lse, void *workspace, size_t workspace_bytes,
                                 void *cuda_stream) {
    return prefill_entry(true, dims, dtype, B, s_q, s_kv, q_offset, causal, head_begin, head_count, head_shard,
                         q_nope, q_pe, c_kv, k_pe, w_kv_b, rms_w, out, lse, workspace, workspace_bytes, cuda_stream);
}

size_t mla_latent_attn_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                 int causal, int head_count, int head_shard) {
    Prefill p;
    if (prefill_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, 0, head_count, head_shard, false, &p) != MLA_OK)
        return 0;
    if (B == 0 || s_q == 0 || head_count == 0) return 0;
    return prefill_ws(p, false, nullptr).bytes;
}

mla_status mla_latent_attn_fused_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                     int causal, int head_begin, int head_count, const void *q_nope, const void *q_pe,
                                     const void *c_kv, const void *k_pe, const void *w_kv_b, const void *rms_w,
                                     void *out, float *lse, void *workspace, size_t workspace_bytes,
                                     void *cuda_stream) {
    return prefill_entry(false, dims, dtype, B, s_q, s_kv, q_offset, causal, head_begin, head_count, 0, q_nope, q_pe,
                         c_kv, k_pe, w_kv_b, rms_w, out, lse, workspace, workspace_bytes, cuda_stream, true);
}

size_t mla_latent_attn_fused_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                       int causal, int head_count) {
    Prefill p;
    if (prefill_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, 0, head_count, 0, false, &p) != MLA_OK || !p.tc)
        return 0;
    if (B == 0 || s_q == 0 || head_count == 0) return 0;
    return prefill_ws(p, false, nullptr, true).bytes;
}

void mla_set_fused_cluster(int size) { g_fused_cluster = size; }

size_t mla_absorbed_attn_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv, int q_offset,
                                   int causal, int head_count, int head_shard) {
    Prefill p;
    if (prefill_shape(dims, dtype, B, s_q, s_kv, q_offset, causal, 0, head_count, head_shard, true, &p) != MLA_OK)
        return 0;
    if (B == 0 || s_q == 0 || head_count == 0) return 0;
    return prefill_ws(p, true, nullptr).bytes;
}

size_t mla_decode_workspace(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits) {
    Decode p;
    if (decode_shape(dims, dtype, B, kv_len, n_splits, &p) != MLA_OK) return 0;
    if (B == 0) return 0;
    return decode_ws(p, nullptr, true).bytes;
}

size_t mla_tpla_decode_workspace(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits,
                                 int n_shards) {
    Decode p;
    if (decode_shape(dims, dtype, B, kv_len, n_splits, &p, n_shards) != MLA_OK) return 0;
    if (B == 0) return 0;
    return decode_ws(p, nullptr, true).bytes;
}

namespace {
// Split-KV latent decode over g latent shards (g = 1: plain latent decode).  With g > 1
// `lse` is the shard log-sum-exps [g][B][H] and the partials stay in the workspace.
mla_status decode_call(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits, int g,
                       const void *q_nope, const void *q_pe, const void *c_cache, const void *kpe_cache,
                       const void *w_kv_b, void *out, float *lse, float *part_out, float *part_lse, void *workspace,
                       size_t workspace_bytes, void *cuda_stream) {
    Decode p;
    mla_status st = decode_shape(dims, dtype, B, kv_len, n_splits, &p, g);
    if (st != MLA_OK) return st;
    if (B == 0) return MLA_OK;
    const void *ptrs[] = {q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out, lse};
    for (const void *q : ptrs)
        if (!q) return MLA_ERR_NULL;
    if ((part_out == nullptr) != (part_lse == nullptr)) return MLA_ERR_NULL;
    for (const void *q : ptrs)
        if (!aligned16(q)) return MLA_ERR_ALIGN;
    if ((part_out && !aligned16(part_out)) || (part_lse && !aligned16(part_lse))) return MLA_ERR_ALIGN;
    bool own = part_out == nullptr;
    DecodeWs wsz = decode_ws(p, nullptr, true);   // the query always covers the own-partials case
    if (workspace_bytes < wsz.bytes) return MLA_ERR_WORKSPACE;
    if (wsz.bytes && !workspace) return MLA_ERR_NULL;
    if (workspace && !aligned16(workspace)) return MLA_ERR_ALIGN;
    const size_t es = ty_size(p.tin);
    size_t rows = (size_t)p.B * p.H;
    Range in[] = {rng(q_nope, rows * p.Dn * es), rng(q_pe, rows * p.Dr * es),
                  rng(c_cache, (size_t)p.B * p.L * p.Dk * es), rng(kpe_cache, (size_t)p.B * p.L * p.Dr * es),
                  rng(w_kv_b, (size_t)p.H * (p.Dn + p.Dv) * p.Dk * es)};
    Range outs[] = {rng(out, rows * p.Dv * es), rng(lse, rows * p.g * 4), rng(workspace, wsz.bytes),
                    rng(part_out, (size_t)p.n * rows * p.Dk * 4), rng(part_lse, (size_t)p.n * rows * 4)};
    st = check_alias(in, 5, outs, 5);
    if (st != MLA_OK) return st;
    DecodeWs w = decode_ws(p, workspace, true);   // its partials buffer also serves as fp16 scratch
    float *po = own ? w.po : part_out;
    float *pl = own ? w.pl : part_lse;
    cudaStream_t cs = (cudaStream_t)cuda_stream;
    float scale = scale_of(dims);
    g_last_path = p.tc ? 2 : 1;
    if (p.tc) {
        const long rows = (long)p.B * p.H;
        MLA_TRY(launch_rope_rows_at(p.tin, TY_F16, rows, p.Dr, q_pe, p.L - 1, dims->rope_base, w.qpe, cs));
        TcDecode t{p.B, p.L, p.n, p.H, p.Dk, p.Dn, p.Dr, p.Dv, p.chunk, scale, dims->rope_base, p.g};
        return cuda_status(tc_decode(t, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out, lse, po, pl, w.po, !own,
                                     w.qabs, w.qpe, w.olat, w.qx, w.qpx, cs));
    }
    return decode_simt(p, scale, dims, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out, lse, po, pl, w, cs);
}
}  // namespace

mla_status mla_decode_splitkv(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits,
                              const void *q_nope, const void *q_pe, const void *c_cache, const void *kpe_cache,
                              const void *w_kv_b, void *out, float *lse, float *part_out, float *part_lse,
                              void *workspace, size_t workspace_bytes, void *cuda_stream) {
    return decode_call(dims, dtype, B, kv_len, n_splits, 1, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out, lse,
                       part_out, part_lse, workspace, workspace_bytes, cuda_stream);
}

mla_status mla_tpla_decode(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits, int n_shards,
                           const void *q_nope, const void *q_pe, const void *c_cache, const void *kpe_cache,
                           const void *w_kv_b, void *out, float *shard_lse, void *workspace, size_t workspace_bytes,
                           void *cuda_stream) {
    return decode_call(dims, dtype, B, kv_len, n_splits, n_shards, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out,
                       shard_lse, nullptr, nullptr, workspace, workspace_bytes, cuda_stream);
}

size_t mla_rmsnorm_bwd_workspace(mla_dtype dtype, long rows, int d, int n_shards) {
    if (!valid_dtype(dtype) || rows < 0 || d < 1 || n_shards < 1 || d % n_shards) return 0;
    return align_up(rmsnorm_bwd_ws(ty_of(dtype), rows, d, n_shards), 256);
}

mla_status mla_rmsnorm_bwd(mla_dtype dtype, long rows, int d, int n_shards, float eps, const void *x, const void *w,
                           const void *dy, void *dx, float *dw, void *workspace, size_t workspace_bytes,
                           void *cuda_stream) {
    if (!valid_dtype(dtype)) return MLA_ERR_DTYPE;
    if (rows < 0 || d < 1 || n_shards < 1 || d % n_shards || !(eps >= 0.f)) return MLA_ERR_SHAPE;
    if (rows == 0) {   // only dw is written (zeros)
        if (!dw) return MLA_ERR_NULL;
        if (!aligned16(dw)) return MLA_ERR_ALIGN;
        g_last_path = 1;
        return cuda_status(launch_rmsnorm_bwd(ty_of(dtype), 0, d, n_shards, eps, nullptr, nullptr, nullptr, nullptr, dw,
                                              nullptr, (cudaStream_t)cuda_stream));
    }
    if (!x || !w || !dy || !dx || !dw || !workspace) return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(dy) || !aligned16(dx) || !aligned16(dw) || !aligned16(workspace))
        return MLA_ERR_ALIGN;
    const size_t need = mla_rmsnorm_bwd_workspace(dtype, rows, d, n_shards);
    if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
    const size_t es = ty_size(ty_of(dtype));
    Range in[] = {rng(x, (size_t)rows * d * es), rng(w, (size_t)d * es), rng(dy, (size_t)rows * d * es)};
    Range outs[] = {rng(dx, (size_t)rows * d * es), rng(dw, (size_t)d * 4), rng(workspace, need)};
    mla_status st = check_alias(in, 3, outs, 3);
    if (st != MLA_OK) return st;
    g_last_path = 1;
    return cuda_status(launch_rmsnorm_bwd(ty_of(dtype), rows, d, n_shards, eps, x, w, dy, dx, dw, (float *)workspace,
                                          (cudaStream_t)cuda_stream));
}

mla_status mla_rmsnorm(mla_dtype dtype, long rows, int d, int n_shards, float eps, const void *x, const void *w,
                       void *y, void *cuda_stream) {
    if (!valid_dtype(dtype)) return MLA_ERR_DTYPE;
    if (rows < 0 || d < 1 || n_shards < 1 || d % n_shards || !(eps >= 0.f)) return MLA_ERR_SHAPE;
    if (rows == 0) return MLA_OK;
    if (!x || !w || !y) return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return MLA_ERR_ALIGN;
    const size_t es = ty_size(ty_of(dtype));
    Range in[] = {rng(x, (size_t)rows * d * es), rng(w, (size_t)d * es)};
    Range outs[] = {rng(y, (size_t)rows * d * es)};
    mla_status st = check_alias(in, 2, outs, 1);
    if (st != MLA_OK) return st;
    g_last_path = 1;
    return cuda_status(launch_rmsnorm_shards(ty_of(dtype), rows, d, n_shards, eps, x, w, y,
                                             (cudaStream_t)cuda_stream));
}

mla_status mla_lse_combine(mla_dtype out_dtype, int n_splits, int rows, int D, const float *part_out,
                           const float *part_lse, void *out, float *lse, void *cuda_stream) {
    if (!valid_dtype(out_dtype)) return MLA_ERR_DTYPE;
    if (n_splits < 1 || n_splits > 256 || rows < 0 || D < 1) return MLA_ERR_SHAPE;
    if (rows == 0) return MLA_OK;
    if (!part_out || !part_lse || !out || !lse) return MLA_ERR_NULL;
    if (!aligned16(part_out) || !aligned16(part_lse) || !aligned16(out) || !aligned16(lse)) return MLA_ERR_ALIGN;
    const size_t es = ty_size(ty_of(out_dtype));
    Range in[] = {rng(part_out, (size_t)n_splits * rows * D * 4), rng(part_lse, (size_t)n_splits * rows * 4)};
    Range outs[] = {rng(out, (size_t)rows * D * es), rng(lse, (size_t)rows * 4)};
    mla_status st = check_alias(in, 2, outs, 2);
    if (st != MLA_OK) return st;
    g_last_path = 1;
    return cuda_status(launch_lse_combine(ty_of(out_dtype), n_splits, rows, D, part_out, part_lse, out, lse,
                                          (cudaStream_t)cuda_stream));
}

const char *mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_NULL: return "MLA_ERR_NULL: a required pointer is NULL";
        case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE: a size, offset or head range is out of range";
        case MLA_ERR_DTYPE: return "MLA_ERR_DTYPE: unknown dtype";
        case MLA_ERR_ALIGN: return "MLA_ERR_ALIGN: a pointer is not 16-byte aligned";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace smaller than the *_workspace figure";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: no kernel for these dimensions";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call or kernel launch failed";
        case MLA_ERR_DEVICE_TIMEOUT: return "MLA_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
        case MLA_ERR_ALIAS: return "MLA_ERR_ALIAS: an output overlaps an input or another output";
    }
    return "unknown mla_status";
}

mla_status mla_check_device_error(void *cuda_stream) {
    cudaStream_t cs = (cudaStream_t)cuda_stream;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return MLA_ERR_CUDA;
    unsigned int flags = 0;
    if (tc_read_and_clear_error(&flags, cs) != cudaSuccess) return MLA_ERR_CUDA;
    return flags ? MLA_ERR_DEVICE_TIMEOUT : MLA_OK;
}

mla_status mla_selftest_bounded_wait(unsigned limit_us, void *cuda_stream) {
    if (limit_us < 1 || limit_us > 100000) return MLA_ERR_SHAPE;
    return cuda_status(launch_wait_probe((uint64_t)limit_us * 1000u, (cudaStream_t)cuda_stream));
}

int mla_last_path(void) { return g_last_path; }

void mla_set_path_override(int mode) { g_path_override = mode; }

}  // extern "C"
