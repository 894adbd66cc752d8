// mla_internal.h -- host-side declarations shared by the translation units of libmla.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

// Storage codes of a tensor (element type in memory; arithmetic is always fp32).
enum { TY_F16 = 0, TY_BF16 = 1, TY_F32 = 2 };
inline int ty_of(mla_dtype dt) { return dt == MLA_F32 ? TY_F32 : TY_BF16; }
inline size_t ty_size(int ty) { return ty == TY_F32 ? 4 : 2; }

// Launch accounting / optional event timing around every kernel launch (profile.cu).
void prof_begin(const char *name, cudaStream_t st);
void prof_end(const char *name, cudaStream_t st);
struct ProfScope {
    const char *n;
    cudaStream_t s;
    ProfScope(const char *name, cudaStream_t st) : n(name), s(st) { prof_begin(n, s); }
    ~ProfScope() { prof_end(n, s); }
};

// ------------------------------------------------------------------ shared prep ----

// RoPE table: tab[(pos - pos0) * Dr/2 + t] = (cos, sin)(pos * base^(-2t/Dr)) for
// positions [pos0, pos0 + n_pos), angles formed in double precision.
cudaError_t launch_rope_table(long pos0, long n_pos, int Dr, float base, float2 *tab, cudaStream_t st);

// One warp per latent row: chat = RMSNorm(c_kv) * rms_w and kpe = RoPE(k_pe, j) for
// keys j < n_rows of every batch.  c_kv [B, s_kv, Dk], k_pe [B, s_kv, Dr] (storage
// tin) -> chat [B, pad_rows, Dk], kpe [B, pad_rows, Dr] (storage tout); rows
// n_rows..pad_rows-1 are zero-filled.  `tab` covers positions from 0.
cudaError_t launch_latent_prep(int tin, int tout, int B, int s_kv, int n_rows, int pad_rows, int Dk, int Dr,
                               const void *c_kv, const void *k_pe, const void *rms_w, float eps, const float2 *tab,
                               void *chat, void *kpe, cudaStream_t st);

// RoPE on `rows` rows of width Dr; row r sits at position pos0 + (r / pos_div) % pos_mod;
// `tab` starts at position tab_pos0.
// Rows at one position `pos` (the decode query): RoPE with the position's table computed
// inside the launch (one launch instead of launch_rope_table + launch_rope_rows).
cudaError_t launch_rope_rows_at(int tin, int tout, long rows, int Dr, const void *x, long pos, float base, void *y,
                                cudaStream_t st);
cudaError_t launch_rope_rows(int tin, int tout, long rows, int Dr, const void *x, long pos0, long pos_div,
                             long pos_mod, const float2 *tab, long tab_pos0, void *y, cudaStream_t st);

// y[i] = x[i] for i < n, converting storage type.
cudaError_t launch_convert(int tin, const void *x, int tout, void *y, long n, cudaStream_t st);

// Every prep step of the tensor-core explicit prefill in one launch (bf16 in, fp16
// out; Dr == 64, Dk a multiple of 256 up to 1024): the RoPE table for positions
// [0, n_pos), chat = RMSNorm(c_kv) * rms_w and kpe = RoPE(k_pe, j) as in
// launch_latent_prep, an fp16 copy of the n_w bf16 weights w_src -> w16 (n_w a multiple
// of 8), and qpe = RoPE(q_pe) in fp16 for q rows [B][s_q][n_hq] at positions q_offset + i
// (n_pos must cover them).
bool prep_tc_supported(int Dk, int Dr);
cudaError_t launch_prep_tc(int B, int s_kv, int n_rows, int pad_rows, int Dk, long n_pos, float base,
                           const void *c_kv, const void *k_pe, const void *rms_w, float eps, float2 *tab, void *chat,
                           void *kpe, const void *w_src, void *w16, long n_w, const void *q_pe, void *qpe, int s_q,
                           int q_offset, int n_hq, cudaStream_t st);

// ------------------------------------------------------------------- SIMT path ----

// C(m,n) = sum_k A(m,k) B(n,k) for every (zb, zh), arbitrary element strides.
struct GemmArgs {
    int M, N, K, nzb, nzh;
    const void *A; int ta; long a_zb, a_zh, a_m, a_k;
    const void *B; int tb; long b_zb, b_zh, b_n, b_k;
    void *C; int tc; long c_zb, c_zh, c_m, c_n;
    int accumulate;   // 1: C += A B^T (C read in its storage type), 0: C = A B^T
};
cudaError_t launch_gemm_simt(const GemmArgs &g, cudaStream_t st);

// Softmax attention over rows x keys with the scores split in two bands
// (q1.k1 over D1 dims + q2.k2 over D2 dims), values of width Dv.
// Grid: z = (b, h) pairs, rows per pair, keys split into n_splits chunks.
struct AttnArgs {
    int n_b, n_h, n_rows, D1, D2, Dv;
    const void *q1; int tq1; long q1_b, q1_h, q1_r;
    const void *q2; int tq2; long q2_b, q2_h, q2_r;
    const void *k1; int tk1; long k1_b, k1_h, k1_r;
    const void *k2; int tk2; long k2_b, k2_h, k2_r;
    const void *v;  int tv;  long v_b, v_h, v_r;
    long kv_len;
    int n_splits; long chunk;
    int causal; long pos0;          // row r sits at absolute position pos0 + r
    float scale;
    // normalised output and lse, used when part_out == nullptr
    void *out; int to; long o_b, o_h, o_r;
    float *lse; long l_b, l_h, l_r;
    // split partials (fp32), output normalised within the split
    float *part_out; long po_s, po_b, po_h, po_r;
    float *part_lse; long pl_s, pl_b, pl_h, pl_r;
};
cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t st);

// lse-combine: part_out [n][rows][D], part_lse [n][rows] -> out [rows][D] (storage tout), lse [rows]
// The same merge over fp16 partials (n <= 32 splits, D % 128 == 0, D <= 1024), bf16 out.
cudaError_t launch_lse_combine16(int n, long rows, int D, const void *po, const float *pl, void *out, float *lse,
                                 cudaStream_t st);
cudaError_t launch_lse_combine(int tout, int n, long rows, int D, const float *po, const float *pl, void *out,
                               float *lse, cudaStream_t st);

// y = per-shard RMSNorm of x [rows][D]: each of the g shards of D/g columns is scaled by
// its own 1/sqrt(mean square + eps) and multiplied by the matching slice of w [D].
cudaError_t launch_rmsnorm_shards(int ty, long rows, int D, int g, float eps, const void *x, const void *w, void *y,
                                  cudaStream_t st);

// Backward of launch_rmsnorm_shards for an upstream dy: dx (storage ty) and dw (fp32, summed
// over rows).  ws: fp32 scratch of rmsnorm_bwd_ws(...) bytes.
size_t rmsnorm_bwd_ws(int ty, long rows, int D, int g);
cudaError_t launch_rmsnorm_bwd(int ty, long rows, int D, int g, float eps, const void *x, const void *w,
                               const void *dy, void *dx, float *dw, float *ws, cudaStream_t st);

// TPLA decode around the latent decode kernels: qa [B][H][Dk], qp [B][H][Dr] -> qx
// [B][g][H][Dk] (row (b,i,h) zero outside shard i's dims), qpx [B][g][H][Dr] (replicated);
// storage ty.
cudaError_t launch_tpla_expand(int ty, int B, int H, int g, int Dk, int Dr, const void *qa, const void *qp, void *qx,
                               void *qpx, cudaStream_t st);
// Split partials po [n][B][g][H][Dk], pl [n][B][g][H] -> out [B][H][Dk] (shard i's dims from
// rows (b,i,h), storage tout) and the shard log-sum-exps slse [g][B][H].
cudaError_t launch_tpla_combine(int tout, int n, int B, int H, int g, int Dk, const float *po, const float *pl,
                                void *out, float *slse, cudaStream_t st);

// One-thread kernel whose bounded mbarrier wait (limit_ns) runs out by construction and
// records the timeout in the device error word (the self-test of that mechanism).
cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st);

// ------------------------------------------------------------------ backward ----
// D[b][h][i] = dO[b][i][h] . out[b][i][h] (fp32 [B][hc][s_q]).
cudaError_t launch_bwd_rowdot(int ty, int B, int s_q, int hc, int Dv, const void *dout, const void *out, float *D,
                              cudaStream_t st);
// CUDA-core attention backward of one head shard (heads h0 .. h0 + nh of the call):
// dq_nope (storage ty) and the rotated dq (fp32) of every query row, dK / dV / this
// shard's per-head dk_rot (fp32 [B][nh][kv][..]) of every key below kv.  K / V fp32 with
// batch and head strides; qr, kr fp32 (the forward's rotated bands); lse, D fp32.
struct BwdSimtArgs {
    int B, s_q, hc, h0, nh, Dn, Dr, Dv;
    long kv, kv_pad;
    int causal;
    long q_off;
    float scale;
    int ty;
    const void *q_nope;
    const float *qr, *K, *V, *kr, *lse, *D;
    long k_b, k_h, v_b, v_h;
    const void *dout;
    void *dq_nope;
    float *dqr, *dK, *dV, *dkr;
};
bool bwd_simt_supported(int Dn, int Dr, int Dv);
cudaError_t launch_attn_bwd_simt(const BwdSimtArgs &a, cudaStream_t st);
// acc[b][j][:] (+)= sum_hl part[b][hl][j][:] for j < kv (acc row pitch acc_pitch rows).
cudaError_t launch_head_sum(int B, int nh, long kv, int Dr, long acc_pitch, const float *part, float *acc,
                            bool accumulate, cudaStream_t st);
// y = RoPE(x, -pos) (the transpose of the forward rotation), rows at positions
// pos0 + (r / pos_div) % pos_mod, zeros at positions >= pos_end; tab from position 0.
cudaError_t launch_rope_inv(long rows, int Dr, const float *x, long x_pitch, long pos0, long pos_div, long pos_mod,
                            long pos_end, const float2 *tab, void *y, int ty, long y_pitch, cudaStream_t st);
// RMSNorm backward of one batch's latent rows with an fp32 upstream gradient: dx for rows
// < n_rows, zeros for rows [n_rows, s_kv); dw (fp32) set or accumulated in a fixed order.
// part: fp32 scratch of rms_bwd_parts(s_kv) * Dk floats.
size_t rms_bwd_parts(long s_kv);
cudaError_t launch_rms_bwd_f32dy(int ty, long n_rows, long s_kv, int Dk, float eps, const void *x, const void *w,
                                 const float *dy, void *dx, float *dw, bool accumulate, float *part,
                                 cudaStream_t st);

// Reads and clears the bounded-wait error words of the tensor-core kernels.
cudaError_t tc_read_and_clear_error(unsigned int *flags, cudaStream_t st);

}  // namespace mla
