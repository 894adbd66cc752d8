// tc.h -- host interface of the tensor-core (tcgen05 + TMA) kernels of libmla.
#pragma once

#include <cuda_runtime.h>

namespace mla {

struct TcPrefill {
    int B, s_q, s_kv, q_offset, causal, head_begin, head_count, hs, n_shards;
    int Dk, Dn, Dr, Dv, H;
    long kv_need;
    float scale;
};

struct TcDecode {
    int B, L, n, H, Dk, Dn, Dr, Dv;
    long chunk;
    float scale, rope_base;
    int g;   // latent shards (TPLA); 1 for plain latent decode
};

bool tc_explicit_supported(int Dk, int Dn, int Dr, int Dv);
bool tc_absorbed_supported(int Dk, int Dn, int Dr, int Dv);
bool tc_decode_supported(int Dk, int Dn, int Dr, int Dv, int H);

// Explicit prefill after the shared prep (fp16 chat, kpe, qpe already in the
// workspace): per head shard, an fp16 copy of the shard's W_kv_b rows, the K_nope /
// V^T reconstruction GEMMs and the attention kernel.
// qpe: the rotated q_pe in fp16 [B][s_q][head_count][64]; w16: fp16 copy of the
// head_count heads' W_kv_b rows [head_count][Dn+Dv][Dk].
cudaError_t tc_explicit_prefill(const TcPrefill &p, const void *q_nope, const void *w_kv_b, void *out,
                                float *lse, const void *chat, const void *kpe, const void *qpe, void *kws,
                                void *vws, const void *w16, cudaStream_t st);
// Explicit prefill with the K_nope / V^T reconstruction inside the attention kernel
// (tc_fused.cu): no K/V workspace; `cluster` (4 or 8) query tiles of a head share every
// rebuilt key tile.  Inputs as tc_explicit_prefill (w16 holds all head_count heads).
cudaError_t tc_fused_prefill(const TcPrefill &p, const void *q_nope, void *out, float *lse, const void *chat,
                             const void *kpe, const void *qpe, const void *w16, int cluster, cudaStream_t st);
// The K_nope / V^T reconstruction of heads h0 .. h0 + nh of the call into the per-shard
// workspace (kws [B][kv_pad][hs*128], vws [B][hs*128][kv_pad], fp16).
cudaError_t tc_reconstruct(const TcPrefill &p, int h0, int nh, const void *chat, const void *w16, void *kws,
                           void *vws, cudaStream_t st);
// Backward (tc_bwd.cu): q_nope / dO widened to fp16 and D = dO . out; a 16-bit transpose;
// the attention backward of one head shard (dq_nope bf16, rotated dq fp32, [dK_nope^T ;
// dV^T] per head fp16 [nh][256][B][kv_pad], dk_rot per head fp32 [B][nh][kv_pad][64]).
cudaError_t launch_bwd_prep_tc(int B, int s_q, int hc, const void *q_nope, const void *dout, const void *out,
                               void *qn16, void *do16, float *D, cudaStream_t st);
cudaError_t launch_transpose16(long R, long C, const void *x, void *y, cudaStream_t st);
cudaError_t tc_bwd_attn(const TcPrefill &p, int h0, int nh, const void *kws, const void *vws, const void *kpe,
                        const void *qn16, const void *qpe, const void *do16, const float *lse, const float *D,
                        void *dq_nope, float *dqr, void *dkvt, float *dkr, cudaStream_t st);
cudaError_t tc_absorbed_prefill(const TcPrefill &p, const void *q_nope, const void *w_kv_b, void *out,
                                float *lse, const void *chat, const void *kpe, const void *qpe, void *qabs,
                                void *olat, void *w16, cudaStream_t st);
// po / pl: the split partials (the caller's, fp32, when user_po; else the workspace's);
// po16: workspace room for the partials in fp16 (the plain decode with n <= 32 splits merges
// fp16 partials: written so by the kernel, or rounded from the caller's fp32 ones, so the
// output does not depend on whether the caller asked for the partials).
cudaError_t tc_decode(const TcDecode &p, const void *q_nope, const void *q_pe, const void *c_cache,
                      const void *kpe_cache, const void *w_kv_b, void *out, float *lse, float *po, float *pl,
                      void *po16, bool user_po, void *qabs, void *qpe, void *olat, void *qx, void *qpx,
                      cudaStream_t st);

}  // namespace mla
