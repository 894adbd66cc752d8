/*
 * mla.h -- C ABI of libmla: multi-head latent attention (MLA) computed from the
 * compressed latent, on one GB300 GPU (sm_103a).
 *
 * What the library computes (pages cited by title and section):
 *  - "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
 *    (arXiv 2607.17644), "What carries the argument" and Fig. 2: the per-rank
 *    compute of LAGA -- RMSNorm of the gathered latent c_KV, per-head K_nope/V
 *    rebuilt locally through W_kv_b one head shard at a time (the paper's section
 *    3.3 "H_r slice of W_kv_b(latent)"), decoupled RoPE on q_pe and on the k_pe
 *    band shared by all heads, causal softmax attention, output plus log-sum-exp.
 *    The absorbed form (q_absorbed = W_kv_b^T q_nope, latent-space attention,
 *    un-absorb) is the companion path of the same figure.
 *  - "TPLA: Tensor Parallel Latent Attention ..." (arXiv 2508.15881), "What
 *    carries the argument": the latent normalisation is an RMSNorm; "The reading":
 *    the latent cut into shards, each attended with all heads and its own softmax,
 *    outputs summed (mla_tpla_decode, with the per-shard norm of mla_rmsnorm).
 *  - "Helix Parallelism ..." (arXiv 2507.07120), "What carries the argument" and
 *    "Assumptions" (paper section 2.1.1): split-KV partial outputs and their
 *    log-sum-exp scalars are rescaled and summed into the exact softmax output.
 *
 * Conventions for every entry point:
 *  - All tensors are dense, row-major, contiguous, in device memory (except where
 *    stated), and every pointer must be 16-byte aligned.  The caller owns all
 *    memory; the library never allocates device memory.  Scratch memory is the
 *    caller's `workspace` (size from the matching *_workspace query).
 *  - `mla_dtype` selects the storage type of every floating-point tensor except
 *    the log-sum-exp and the split partials, which are always fp32.  Arithmetic is
 *    fp32 (bf16 tensor-core products accumulate in fp32).
 *  - Calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy default
 *    stream) and do no host synchronisation, except mla_check_device_error.
 *  - Inputs are never written.  Outputs and the workspace may not overlap any
 *    input or each other (MLA_ERR_ALIAS).
 *  - On any error status nothing has been launched, except MLA_ERR_CUDA, which
 *    reports a failed launch or failed CUDA runtime call.
 *  - Precision of the bf16 tensor-core kernels: their score operands (normalised
 *    latent, rotated RoPE bands, K_nope, q_abs) and P are fp16, so every such value
 *    must lie inside fp16's range (|x| < 65504), and a log-sum-exp carries an absolute
 *    error of up to about 2^-11 of the largest |lse| of the call (measured 5.7e-4 at
 *    unit-scale inputs, whose |lse| stays below ~8; 0.1 at scores near 500).  Callers
 *    whose scores go well beyond that range and who need a tighter log-sum-exp select
 *    the CUDA-core kernels, which keep fp32 intermediates, with
 *    mla_set_path_override(1).
 *  - Positions: query row i of a prefill call sits at absolute position q_offset+i,
 *    key j at position j; a decode query sits at kv_len-1.  RoPE pairs (t, t+d/2)
 *    with angle pos * rope_base^(-2t/d_rope).  Causal: key j visible iff
 *    j <= q_offset + i.  LSE is the natural log of the softmax normaliser (scale
 *    included); a row that sees no key gives lse = -inf and output 0.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_NULL = -1,           /* a required pointer is NULL                       */
    MLA_ERR_SHAPE = -2,          /* a size, offset or head range is out of range      */
    MLA_ERR_DTYPE = -3,          /* unknown mla_dtype                                 */
    MLA_ERR_ALIGN = -4,          /* a pointer is not 16-byte aligned                  */
    MLA_ERR_WORKSPACE = -5,      /* workspace_bytes below the *_workspace figure      */
    MLA_ERR_UNSUPPORTED = -6,    /* dimensions this build has no kernel for           */
    MLA_ERR_CUDA = -7,           /* a CUDA runtime call or kernel launch failed       */
    MLA_ERR_DEVICE_TIMEOUT = -8, /* a bounded device-side wait gave up (see below)    */
    MLA_ERR_ALIAS = -9           /* an output/workspace overlaps an input or another  */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/* Per-model dimensions and constants. */
typedef struct {
    int n_heads;         /* H: query heads of the model                         */
    int d_kv;            /* latent width of c_KV (512 for DeepSeek-V3)          */
    int d_nope;          /* per-head non-rotary q/k width (128)                 */
    int d_rope;          /* decoupled RoPE band width (64), even                */
    int d_v;             /* per-head value width (128)                          */
    float rope_base;     /* RoPE base (10000)                                   */
    float rms_eps;       /* RMSNorm epsilon inside the square root (1e-6)       */
    float softmax_scale; /* <= 0 selects 1/sqrt(d_nope + d_rope)                */
} mla_dims;

/*
 * Prefill, explicit / LAGA per-rank compute.
 * Queries are rows [q_offset, q_offset+s_q) of a sequence whose full latent of
 * s_kv tokens is given (a simulated sequence-parallel rank when q_offset > 0).
 * Heads [head_begin, head_begin+head_count) are computed; per-head K_nope/V are
 * rebuilt head_shard heads at a time (0 = all at once) into the workspace, so the K/V
 * part of the workspace grows with head_shard, not with head_count; the rest (the
 * normalised latent, the rotated RoPE bands of the keys and of every query row and
 * head, the RoPE table and, on the tensor-core path, an fp16 copy of the call's
 * W_kv_b rows) grows with the call's tokens and heads.
 *   q_nope [B, s_q, head_count, d_nope]     q_pe [B, s_q, head_count, d_rope] (not rotated)
 *   c_kv   [B, s_kv, d_kv]                  k_pe [B, s_kv, d_rope] (not rotated)
 *   w_kv_b [n_heads*(d_nope+d_v), d_kv]: head h owns rows h*(d_nope+d_v) ..,
 *          first d_nope rows -> K_nope, next d_v rows -> V
 *   rms_w  [d_kv]
 *   out    [B, s_q, head_count, d_v]        lse (fp32) [B, head_count, s_q]
 * Causal calls need q_offset + s_q <= s_kv.  B, s_q or head_count of 0 is a no-op.
 */
mla_status mla_latent_attn_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                               int q_offset, int causal, int head_begin, int head_count,
                               int head_shard, const void *q_nope, const void *q_pe,
                               const void *c_kv, const void *k_pe, const void *w_kv_b,
                               const void *rms_w, void *out, float *lse, void *workspace,
                               size_t workspace_bytes, void *cuda_stream);

/*
 * Prefill, absorbed form (same arguments, layouts and result as
 * mla_latent_attn_fwd): q_abs = W_K(h)^T q_nope (d_kv wide) and the latent
 * accumulator o_lat (d_kv wide) are materialised per head shard in the
 * workspace, then out = W_V(h) o_lat.  This is the companion path whose larger
 * activation footprint the LAGA page measures.
 */
mla_status mla_absorbed_attn_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                                 int q_offset, int causal, int head_begin, int head_count,
                                 int head_shard, const void *q_nope, const void *q_pe,
                                 const void *c_kv, const void *k_pe, const void *w_kv_b,
                                 const void *rms_w, void *out, float *lse, void *workspace,
                                 size_t workspace_bytes, void *cuda_stream);

/*
 * Prefill, explicit form with the per-head up-projection fused into the attention
 * kernel (LAGA page, "Where Pith is reading between the lines": the fused
 * up-projection that completes LAGA).  Same arguments, layouts and result as
 * mla_latent_attn_fwd, without head_shard: K_nope and V are rebuilt from the
 * normalised latent 64 keys at a time inside the attention kernel, each rebuilt tile
 * shared through distributed shared memory by a cluster of 4 or 8 query tiles of its
 * head, and never written to device memory.  The workspace
 * (mla_latent_attn_fused_workspace) holds only the normalised latent, the rotated RoPE
 * bands, the RoPE table and an fp16 copy of the call's W_kv_b rows.  Each key tile is
 * rebuilt once per cluster rather than once per call, so the call does more tensor
 * work than mla_latent_attn_fwd in exchange for no K/V intermediates.
 * Needs bf16 and d_kv = 512, d_nope = d_v = 128, d_rope = 64 (MLA_ERR_UNSUPPORTED
 * otherwise, nothing launched).
 */
mla_status mla_latent_attn_fused_fwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                                     int q_offset, int causal, int head_begin, int head_count,
                                     const void *q_nope, const void *q_pe, const void *c_kv,
                                     const void *k_pe, const void *w_kv_b, const void *rms_w, void *out,
                                     float *lse, void *workspace, size_t workspace_bytes,
                                     void *cuda_stream);

/*
 * Backward of mla_latent_attn_fwd (LAGA page, "What carries the argument": the method's
 * equivalence claim covers gradients).  The chain rule through the forward's own steps:
 * softmax, scores, the RoPE rotations (whose transposes rotate by the opposite angle),
 * the per-head reconstruction through W_kv_b, the latent RMSNorm.  Inputs: the forward's
 * inputs and arguments, its out and lse, and an upstream gradient dout of out
 * [B, s_q, head_count, d_v] (dtype); lse is not differentiated.  Outputs:
 *   dq_nope, dq_pe     like q_nope, q_pe (dtype)
 *   dc_kv, dk_pe       like c_kv, k_pe (dtype): summed over the call's heads; rows of keys
 *                      that no query of the call sees are zero
 *   dw_kv_b (fp32)     like w_kv_b: only the rows of heads [head_begin, head_begin +
 *                      head_count) are written, the others are left as they are
 *   drms_w (fp32)      [d_kv]
 * A call over one query shard (q_offset > 0) writes that shard's contributions: the
 * gradients of c_kv, k_pe, w_kv_b and rms_w of the shards of a sequence add up to those
 * of one call over the whole sequence.  K/V are recomputed head_shard heads at a time.
 * Every band (d_nope, d_rope, d_v) up to 256 wide; B, s_q or head_count of 0 is a no-op.
 * Workspace: mla_latent_attn_bwd_workspace.
 */
mla_status mla_latent_attn_bwd(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                               int q_offset, int causal, int head_begin, int head_count,
                               int head_shard, const void *q_nope, const void *q_pe,
                               const void *c_kv, const void *k_pe, const void *w_kv_b,
                               const void *rms_w, const void *out, const float *lse,
                               const void *dout, void *dq_nope, void *dq_pe, void *dc_kv,
                               void *dk_pe, float *dw_kv_b, float *drms_w, void *workspace,
                               size_t workspace_bytes, void *cuda_stream);
size_t mla_latent_attn_bwd_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q,
                                     int s_kv, int q_offset, int causal, int head_count,
                                     int head_shard);

/*
 * Decode over a latent cache: one query per sequence at position kv_len-1, all
 * n_heads heads, absorbed-form scores, keys split into n_splits contiguous chunks
 * of ceil(kv_len/n_splits) (the last may be short or empty), partials merged by the
 * log-sum-exp rescale.  The cache holds already-normalised c_KV and already-rotated
 * k_pe (what a prefill writes); q_pe is given un-rotated.
 *   q_nope [B, H, d_nope]   q_pe [B, H, d_rope]   c_cache [B, kv_len, d_kv]
 *   kpe_cache [B, kv_len, d_rope]   w_kv_b as above   out [B, H, d_v]   lse (fp32) [B, H]
 *   part_out (fp32, optional) [n_splits, B, H, d_kv]: per-split latent output,
 *            normalised within the split;  part_lse (fp32, optional) [n_splits, B, H].
 *   Pass both NULL to keep the partials in the workspace.
 * 1 <= n_splits <= 256.  kv_len >= 1.
 */
mla_status mla_decode_splitkv(const mla_dims *dims, mla_dtype dtype, int B, int kv_len,
                              int n_splits, const void *q_nope, const void *q_pe,
                              const void *c_cache, const void *kpe_cache, const void *w_kv_b,
                              void *out, float *lse, float *part_out, float *part_lse,
                              void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * TPLA decode (TPLA page, "The reading" and "What carries the argument"): the latent
 * is cut into n_shards equal shards of d_kv/n_shards dims; every shard attends with all
 * n_heads heads over its own dims plus the whole RoPE band, with its own softmax, and
 * the shards' up-projected outputs are summed (what an all-reduce over tensor-parallel
 * ranks would add).  Readings: no orthogonal reparameterisation of the latent, the
 * score scale of mla_dims unchanged, the local softmaxes not rescaled.
 *   c_cache [B, kv_len, d_kv]: each shard RMS-normalised on its own, as
 *            mla_rmsnorm(..., n_shards, ...) writes it; kpe_cache already rotated.
 *   q_nope, q_pe, kpe_cache, w_kv_b, out: as mla_decode_splitkv.
 *   shard_lse (fp32) [n_shards, B, H]: each shard's log-sum-exp over its scores.
 * n_shards = 1 computes exactly mla_decode_splitkv (shard_lse = its lse).
 * 1 <= n_shards <= 16 and n_shards divides d_kv; other sizes as mla_decode_splitkv.
 * Split partials always stay in the workspace (mla_tpla_decode_workspace).
 * The tensor-core path needs bf16, the DeepSeek dimensions and n_heads * n_shards a
 * multiple of 128; anything else runs on the SIMT kernels.
 */
mla_status mla_tpla_decode(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits,
                           int n_shards, const void *q_nope, const void *q_pe, const void *c_cache,
                           const void *kpe_cache, const void *w_kv_b, void *out, float *shard_lse,
                           void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * RMSNorm of `rows` rows of x [rows, d] into y, each row cut into n_shards shards of
 * d/n_shards columns normalised on their own (LAGA page, step 1 of the forward for
 * n_shards = 1; TPLA page, "The reading", for the per-shard latent norm):
 *   y[r][i*ds + t] = x[r][i*ds + t] / sqrt(mean_t' x[r][i*ds + t']^2 + eps) * w[i*ds + t]
 * w [d] in the same dtype; fp32 arithmetic.  1 <= n_shards, n_shards divides d, eps >= 0.
 * This is the cache write of a TPLA decode (the latent of every new token).
 */
mla_status mla_rmsnorm(mla_dtype dtype, long rows, int d, int n_shards, float eps, const void *x,
                       const void *w, void *y, void *cuda_stream);

/*
 * Backward of mla_rmsnorm for an upstream gradient dy [rows, d] (the first piece of the
 * backward pass; LAGA page, "What carries the argument": its equivalence claim covers
 * gradients).  Per shard of ds = d/n_shards columns with r = sqrt(mean x^2 + eps):
 *   dx_k = dy_k w_k / r - x_k (sum over the shard of dy w x) / (ds r^3)   (dtype, [rows, d])
 *   dw_k = sum over rows of dy_k x_k / r                                  (fp32, [d])
 * dw is summed in a fixed order (the same bits on every run).  Scratch: the caller's
 * workspace of mla_rmsnorm_bwd_workspace bytes.  rows = 0 sets dw to zero and reads
 * nothing else (x, w, dy, dx and the workspace may then be NULL).
 */
mla_status mla_rmsnorm_bwd(mla_dtype dtype, long rows, int d, int n_shards, float eps,
                           const void *x, const void *w, const void *dy, void *dx, float *dw,
                           void *workspace, size_t workspace_bytes, void *cuda_stream);
size_t mla_rmsnorm_bwd_workspace(mla_dtype dtype, long rows, int d, int n_shards);

/*
 * Log-sum-exp merge (Helix / Flash-Decoding combine):
 *   lse[r] = log sum_s exp(part_lse[s][r]);  out[r][:] = sum_s exp(part_lse[s][r]-lse[r]) part_out[s][r][:]
 * part_out fp32 [n_splits, rows, D], part_lse fp32 [n_splits, rows] -> out (out_dtype)
 * [rows, D], lse fp32 [rows].  Splits with part_lse = -inf carry no weight.
 * 1 <= n_splits <= 256.
 */
mla_status mla_lse_combine(mla_dtype out_dtype, int n_splits, int rows, int D,
                           const float *part_out, const float *part_lse, void *out, float *lse,
                           void *cuda_stream);

/* Workspace bytes the matching call needs (0 on invalid arguments). */
size_t mla_latent_attn_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                                 int q_offset, int causal, int head_count, int head_shard);
size_t mla_absorbed_attn_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                                   int q_offset, int causal, int head_count, int head_shard);
size_t mla_latent_attn_fused_workspace(const mla_dims *dims, mla_dtype dtype, int B, int s_q, int s_kv,
                                       int q_offset, int causal, int head_count);
size_t mla_decode_workspace(const mla_dims *dims, mla_dtype dtype, int B, int kv_len, int n_splits);
size_t mla_tpla_decode_workspace(const mla_dims *dims, mla_dtype dtype, int B, int kv_len,
                                 int n_splits, int n_shards);

/* Static description of a status code. */
const char *mla_status_string(mla_status status);

/*
 * Synchronises `cuda_stream`, then reads and clears the device-side error word.
 * Kernels that spin on an mbarrier bound every wait by an iteration limit; when a
 * limit is hit the kernel records it in that word and leaves without trapping.
 * Returns MLA_ERR_DEVICE_TIMEOUT if any did since the last check, MLA_ERR_CUDA if
 * the stream reports an error, MLA_OK otherwise.
 */
mla_status mla_check_device_error(void *cuda_stream);

/*
 * Self-test of the bounded device wait behind MLA_ERR_DEVICE_TIMEOUT (the pages have
 * no counterpart).  Launches one tiny kernel on `cuda_stream` in which one thread waits,
 * with the library's bounded mbarrier wait and a limit of limit_us microseconds, on an
 * mbarrier that no thread ever arrives at; no copy, MMA or tensor-memory allocation is
 * in flight.  The wait runs out (within about limit_us plus up to 64 ms of polling),
 * records the timeout in the device error word and the kernel returns, so the context
 * stays usable.  The next mla_check_device_error on that stream then returns
 * MLA_ERR_DEVICE_TIMEOUT (and clears the word).  1 <= limit_us <= 100000, else
 * MLA_ERR_SHAPE with nothing launched.
 */
mla_status mla_selftest_bounded_wait(unsigned limit_us, void *cuda_stream);

/*
 * Which kernel family the last call on this host thread used, for tests and the
 * benchmark: 0 = none yet, 1 = SIMT (CUDA cores, any dimensions, fp32 or bf16),
 * 2 = tensor cores (tcgen05 + TMA, bf16 at the DeepSeek dimensions), 3 = the fused
 * tensor-core prefill of mla_latent_attn_fused_fwd.
 */
int mla_last_path(void);

/* Overrides the path choice on this host thread: 0 = automatic (default),
 * 1 = force the SIMT kernels.  Used by tests to compare the two families. */
void mla_set_path_override(int mode);

/* Query tiles per cluster of the fused prefill on this host thread: 4 or 8; anything
 * else = chosen per call (8 when the call has at least 8 query tiles).  For tests and
 * tuning. */
void mla_set_fused_cluster(int size);

/*
 * Split-KV decode that allocates nothing.  The pages have no counterpart: this is
 * a library convenience for callers that cannot allocate device memory, such as
 * code that runs while a stream is being captured into a CUDA graph (where
 * cudaMalloc is refused), or a host runtime that owns every byte of device memory
 * through its own pool and gives its plugins no allocator.
 * It computes exactly what mla_decode_splitkv computes (same arguments and layouts,
 * partials kept internally), using as its scratch a fixed array of
 * MLA_NOALLOC_SCRATCH_BYTES bytes that the library defines in device memory; every
 * GPU that loads the library holds that array until the process exits.
 *  - A call needing more scratch than the array holds (see mla_decode_workspace)
 *    returns MLA_ERR_WORKSPACE and launches nothing.
 *  - A call outside stream capture looks up the array's device address in the current
 *    context (so calls after a cudaDeviceReset find the new one) and remembers it per
 *    device; a call made while cuda_stream is capturing uses the remembered address.
 *    Make one call on the device before capturing, and capture again after a reset.
 *  - Every call shares the one array and leaves its contents behind.  Nothing in it
 *    needs to start at zero: each call writes all the scratch it reads.  Calls
 *    that overlap on the GPU (other streams, other host threads) race on it;
 *    serialise them.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
mla_status mla_decode_splitkv_noalloc(const mla_dims *dims, mla_dtype dtype, int B, int kv_len,
                                      int n_splits, const void *q_nope, const void *q_pe,
                                      const void *c_cache, const void *kpe_cache,
                                      const void *w_kv_b, void *out, float *lse,
                                      void *cuda_stream);

/*
 * Measurement hooks (not part of the computation).
 * mla_launch_count: launches this library has made since load, all threads, counted
 *   per launch step: one per kernel on the forward and decode paths; a few backward
 *   steps that launch a fixed pair of kernels (a row pass and its fixed-order sum)
 *   count once.
 * mla_profile_enable(1): from now on every launch is bracketed by a pair of CUDA
 *   events recorded on the launching stream (the caller's stream), grouped by
 *   kernel name; mla_profile_enable(0) stops recording and drops what was recorded.
 * mla_profile_kernel: synchronises the recorded events of kernel `name` and returns
 *   the number of launches and their summed device time in milliseconds (0 launches
 *   for an unknown name).  Names: "prep", "latent_prep", "rope_table", "rope_rows",
 *   "convert", "gemm_simt", "attn_simt", "lse_combine", "tc_gemm", "tc_attn",
 *   "tc_latent_attn", "tc_decode_attn", "transpose", "rmsnorm", "rmsnorm_bwd", "tpla_expand",
 *   "tpla_combine", "wait_probe", "tc_fused_attn", "bwd_rowdot",
 *   "attn_bwd_simt", "bwd_rows", "bwd_prep", "tc_bwd_dkv", "tc_bwd_dq".
 * mla_profile_reset: forgets recorded events, keeps recording on/off as it was.
 * Launches from several host threads are recorded safely; call enable, reset and the
 * queries between computations, not while another thread's calls are in flight.
 */
unsigned long long mla_launch_count(void);
void mla_profile_enable(int on);
int mla_profile_kernel(const char *name, long long *launches, double *total_ms);
void mla_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
