// tc_latent.cu -- latent-space (absorbed-form) attention on the sm_103a tensor cores for
// the absorbed prefill, and the host side of the split-KV decode (whose attention kernel
// is in tc_decode.cu).
//
// Method: "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
// (arXiv 2607.17644), Fig. 2 absorbed dataflow and "Core claim" (the absorb trick is
// the decode form): scores s_rj = scale * (q_abs_r . c_j + RoPE(q_pe_r) . RoPE(k_pe_j)),
// latent accumulator o_r = sum_j softmax_j(s_rj) c_j; and "Helix Parallelism ..."
// (arXiv 2507.07120), "What carries the argument": each key split yields a partial
// output plus its log-sum-exp, merged later by the rescale-and-sum.
//
// Shape of the problem: one work unit = 128 queries of one head against the keys they
// see.  Its fp32 accumulator (128 x 512) fills the whole of one SM's TMEM, and Q
// (128 x 576) does not fit in shared memory next to the key stages.  So a unit runs
// on a cluster of two CTAs that split the 512 latent dimensions:
//   * CTA r holds Q's dims [256r, 256r+256) in TMEM (rank 0 also the 64-dim RoPE
//     band) and streams the same dims of each 64-key tile through a TMA ring;
//   * each CTA computes a partial score tile over its dims (tcgen05, A from TMEM),
//     the two partials are swapped through distributed shared memory and summed in a
//     fixed order, so both CTAs hold the identical score tile and run the identical
//     online softmax;
//   * each CTA accumulates its own half of the latent output, O_r += P . C_r, with P
//     from TMEM and the key tile itself as the (MN-major) B operand.
// The prefill prep writes the latent, q_abs and the rotated q_pe in fp16 (11-bit
// significand), so every score stays within ~3e-4 of exact.
//
// Warps (256 threads): 0 TMA producer, 1 MMA issuer + TMEM owner, 2-5 softmax (one
// row per thread), 6-7 idle.  The partial-score swap is one 32 KB bulk copy
// (cp.async.bulk, shared::cta -> shared::cluster) per tile and direction, completing
// as transaction bytes on the receiver's mbarrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_latent_err = 0;

namespace {

using namespace tc;

constexpr int ROWS = 128, NK = 64, ST = 4;
constexpr uint32_t BOX = NK * 128;               // 64 keys x 64 dims (16-bit): 8 KB
constexpr uint32_t STAGE_BYTES = 5 * BOX;        // 4 latent boxes (+ RoPE box on rank 0)
constexpr uint32_t XBUF_BYTES = ROWS * NK * 4;   // one tile of partial scores (send or receive)
constexpr uint32_t SMEM_BYTES = ST * STAGE_BYTES + 2 * XBUF_BYTES + 1024 + 512;
// TMEM columns: accumulators at multiples of their width (O 256, S 64), the A operands
// (P: 64 keys fp16 = 32 columns; Q: up to 320 dims fp16 = 160 columns) after them.
constexpr uint32_t T_O = 0, T_S = 256, T_P = 320, T_Q = 352;
constexpr float RESCALE_LOG2 = 8.0f;

struct LatK {
    int s_q, q_offset, kv_need, causal, n_qtiles, nh, nb, head_off;
    const __half *qa;   // q_abs rows (fp16, 512 wide)
    long qa_b, qa_h, qa_r;
    const __half *qp;   // rotated q_pe rows (fp16, 64 wide)
    long qp_b, qp_h, qp_r;
    float scale_log2;
    __nv_bfloat16 *ol;  // o_lat [b][i][hl][512]
    long ol_b, ol_h, ol_r;
    float *lse;         // lse [b][head][i]
    long l_b, l_h;
    uint32_t idesc_s0, idesc_s1, idesc_pv;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Work unit of a cluster: which rows, which keys, where Q lives and where results go.
struct Unit {
    int b, hl, q0;   // sequence, head within the shard, first query row
    long kb, ke;     // key range [kb, ke)
    int nt;          // 64-key tiles
};

__device__ __forceinline__ Unit unit_of(const LatK &p, int u) {
    Unit w{};
    // (head, batch) pairs fastest, query tiles from the latest (heaviest under the
    // causal mask) down: the first waves take the heaviest tiles of every head
    const int hb = u % (p.nh * p.nb);
    const int qt = p.n_qtiles - 1 - u / (p.nh * p.nb);
    w.hl = hb % p.nh;
    w.b = hb / p.nh;
    w.q0 = qt * ROWS;
    w.kb = 0;
    w.ke = p.causal ? min((long)p.kv_need, (long)p.q_offset + w.q0 + ROWS) : (long)p.kv_need;
    w.nt = w.ke > w.kb ? (int)((w.ke - w.kb + NK - 1) / NK) : 0;
    return w;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    tc_latent_kernel(const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap mR, LatK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *stages = smem;
    // [row][64] partial scores, 16-byte slots of a row rotated by the row index
    float *xbuf = (float *)(stages + ST * STAGE_BYTES);          // received from the peer
    float *sendbuf = (float *)((uint8_t *)xbuf + XBUF_BYTES);    // this CTA's, to the peer
    uint64_t *bars = (uint64_t *)((uint8_t *)sendbuf + XBUF_BYTES);
    uint64_t *k_full = bars, *k_empty = bars + ST;
    uint64_t *q_ready = bars + 3 * ST, *s_full = q_ready + 1, *s_free = q_ready + 2, *p_full = q_ready + 3;
    uint64_t *o_done = q_ready + 4, *o_final = q_ready + 5, *x_full = q_ready + 6, *x_empty = q_ready + 7;
    uint32_t *tslot = (uint32_t *)(q_ready + 8);
    volatile int *abort = (volatile int *)(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const Unit w = unit_of(p, blockIdx.x >> 1);
    const int nt = w.nt;

    if (tid == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        mbar_init(q_ready, 4);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(o_final, 1);
        mbar_init(x_full, 1);      // local expect_tx + the peer's bulk copy
        mbar_init(x_empty, 4);     // one arrival per softmax warp of the peer CTA
        *abort = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(x_full, XBUF_BYTES);   // arm the first tile's receive
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrive
    tc_fence_after();
    const uint32_t tmem = *tslot;

    const int n_box = rank == 0 ? 5 : 4;             // latent boxes of this CTA (+ RoPE band on rank 0)
    const uint32_t stage_tx = (uint32_t)n_box * BOX;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nt > 0) {
            tma_prefetch_desc(&mC);
            tma_prefetch_desc(&mR);
            for (int j = 0; j < nt; ++j) {
                const int s = j % ST;
                if (j >= ST && !mbar_wait(&k_empty[s], ((j / ST) - 1) & 1, abort, &g_tc_latent_err)) break;
                uint8_t *dst = stages + s * STAGE_BYTES;
                const int key0 = (int)(w.kb + (long)j * NK);
                mbar_arrive_expect_tx(&k_full[s], stage_tx);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    tma_load_3d(dst + i * BOX, &mC, &k_full[s], 256 * (int)rank + 64 * i, key0, w.b);
                if (rank == 0) tma_load_3d(dst + 4 * BOX, &mR, &k_full[s], 0, key0, w.b);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (warp-uniform loop; one elected lane issues)
        if (nt > 0) {
            bool ok = __all_sync(0xffffffffu, mbar_wait(q_ready, 0, abort, &g_tc_latent_err));
            const int nks = rank == 0 ? 20 : 16;          // 16-dim k-steps of the partial score
            const uint32_t idesc_s = rank == 0 ? p.idesc_s0 : p.idesc_s1;
            auto issue_pv = [&](int t) -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait(p_full, t & 1, abort, &g_tc_latent_err))) return false;
                tc_fence_after();
                const uint8_t *tile = stages + (t % ST) * STAGE_BYTES;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 16 keys per step; B = 256 dims x 16 keys, MN-major
                        mma_ts(tmem + T_O, tmem + T_P + kk * 8, sdesc_mnmajor(tile + kk * 2048, BOX), p.idesc_pv,
                               (t | kk) != 0);
                    mma_commit(&k_empty[t % ST]);
                    mma_commit(o_done);
                }
                __syncwarp();
                return true;
            };
            for (int j = 0; j < nt && ok; ++j) {
                const int s = j % ST;
                bool go = __all_sync(0xffffffffu, mbar_wait(&k_full[s], (j / ST) & 1, abort, &g_tc_latent_err));
                if (go && j > 0) go = __all_sync(0xffffffffu, mbar_wait(s_free, (j - 1) & 1, abort, &g_tc_latent_err));
                if (!go) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *tile = stages + s * STAGE_BYTES;
                if (elect_one()) {
                    for (int kk = 0; kk < nks; ++kk)
                        mma_ts(tmem + T_S, tmem + T_Q + kk * 8, sdesc_kmajor(tile + (kk >> 2) * BOX) + 2 * (kk & 3),
                               idesc_s, kk != 0);
                    mma_commit(s_full);
                }
                __syncwarp();
                if (j > 0 && !issue_pv(j - 1)) ok = false;
            }
            if (ok) issue_pv(nt - 1);
            if (elect_one()) mma_commit(o_final);
            __syncwarp();
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------- softmax warps
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
        const int i = w.q0 + row;   // query row
        const bool valid = i < p.s_q;
        const long pos = (long)p.q_offset + i;
        // ---- this row of Q into TMEM: latent dims [256 rank, +256), rank 0 also the RoPE band
        {
            const __half *qa = p.qa + w.b * p.qa_b + (long)w.hl * p.qa_h + (long)i * p.qa_r;
            const __half *qp = p.qp + w.b * p.qp_b + (long)(p.head_off + w.hl) * p.qp_h + (long)i * p.qp_r;
            const uint4 *src = (const uint4 *)(qa + 256 * rank);
            for (int c = 0; c < (rank == 0 ? 5 : 4); ++c) {
                const uint4 *sp = c < 4 ? src + c * 8 : (const uint4 *)qp;
                uint32_t r32[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    uint4 x = valid ? sp[v] : make_uint4(0, 0, 0, 0);
                    r32[4 * v] = x.x;
                    r32[4 * v + 1] = x.y;
                    r32[4 * v + 2] = x.z;
                    r32[4 * v + 3] = x.w;
                }
                tmem_st32(lb + T_Q + c * 32, r32);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        const uint32_t peer_recv = map_peer(smem_u32(xbuf), peer);
        const uint32_t peer_x_full = map_peer(smem_u32(x_full), peer);
        const uint32_t peer_x_empty = map_peer(smem_u32(x_empty), peer);
        const bool elected = warp == 2 && lane == 0;
        float *my_send = sendbuf + row * 64;
        const float *my_row = xbuf + row * 64;
        float m = -INFINITY, l = 0.f;
        // A failed wait clears `ok` (warp-uniform) but never leaves the loop early: every
        // softmax thread passes the same named barriers, so an abort cannot strand one.
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(s_full, j & 1, abort, &g_tc_latent_err));
            tc_fence_after();
            uint32_t sr[2][32];
            if (ok) {
                tmem_ld32(lb + T_S, sr[0]);
                tmem_ld32(lb + T_S + 32, sr[1]);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) sr[0][e] = sr[1][e] = 0u;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            // ---- swap partial scores with the peer CTA: stage, then one bulk copy
            named_bar_sync(1, 128);   // the previous copy has finished reading the send buffer
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int slot = (c + row) & 15;
                const uint32_t *q = &sr[c >> 3][(c & 7) * 4];
                *(float4 *)(my_send + slot * 4) =
                    make_float4(__uint_as_float(q[0]), __uint_as_float(q[1]), __uint_as_float(q[2]),
                                __uint_as_float(q[3]));
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (elected) {
                bool go = ok;
                if (go && j > 0) go = mbar_wait_cluster(x_empty, (j - 1) & 1, abort, &g_tc_latent_err);
                if (go) {
                    bulk_copy_to_peer(peer_recv, sendbuf, XBUF_BYTES, peer_x_full);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                ok = go;
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait_cluster(x_full, j & 1, abort, &g_tc_latent_err));
            float x[64];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int slot = (c + row) & 15;
                const float4 o4 = *(const float4 *)(my_row + slot * 4);
                const float ov[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mine = __uint_as_float(sr[c >> 3][(c & 7) * 4 + e]);
                    // rank 0's partial first on both CTAs: identical sums, identical softmax
                    x[c * 4 + e] = (rank == 0 ? mine + ov[e] : ov[e] + mine) * p.scale_log2;
                }
            }
            __syncwarp();   // every lane has read its row of the received partial
            if (lane == 0) {
                if (warp == 2 && j + 1 < nt) mbar_arrive_expect_tx(x_full, XBUF_BYTES);   // arm the next receive
                mbar_arrive_peer(peer_x_empty);
            }
            const long key0 = w.kb + (long)j * NK;
            const bool masked = key0 + NK > w.ke || (p.causal && key0 + NK - 1 > (long)p.q_offset + w.q0);
            if (masked) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const long key = key0 + c;
                    if (key >= w.ke || (p.causal && key > pos)) x[c] = -INFINITY;
                }
            }
            // independent accumulators: the reductions are latency chains otherwise
            float mx[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
            for (int c = 8; c < 64; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
            const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float m_new = fmaxf(m, mt);
            const bool need = m_new > m + RESCALE_LOG2;
            bool pv_done = false;
            if (__any_sync(0xffffffffu, need)) {
                const float m_use = need ? m_new : m;
                const float alpha = (m == -INFINITY) ? 0.f : ex2(m - m_use);
                if (j > 0) {
                    ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, (j - 1) & 1, abort, &g_tc_latent_err));
                    pv_done = true;
                }
                if (j > 0 && ok) {
                    tc_fence_after();
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[32];
                        tmem_ld32(lb + T_O + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(lb + T_O + c * 32, o);
                    }
                    tmem_st_wait();
                }
                l *= alpha;
                m = m_use;
            }
            const float m_eff = (m == -INFINITY) ? 0.f : m;
            float ra[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float p0 = ex2(x[2 * e] - m_eff), p1 = ex2(x[2 * e + 1] - m_eff);
                ra[e & 7] += p0 + p1;
                pk[e] = pack_f16(p0, p1);
            }
            const float rs = ((ra[0] + ra[1]) + (ra[2] + ra[3])) + ((ra[4] + ra[5]) + (ra[6] + ra[7]));
            if (j > 0 && !pv_done)   // P of the previous tile must have been consumed
                ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, (j - 1) & 1, abort, &g_tc_latent_err));
            tc_fence_after();
            if (ok) {
                tmem_st32(lb + T_P, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            l += rs;
        }
        // ---- epilogue: this CTA's half of the normalised latent output (+ lse on rank 0)
        if (ok && nt > 0) ok = mbar_wait(o_final, 0, abort, &g_tc_latent_err);
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        for (int c = 0; c < 8; ++c) {
            uint32_t o[32];
            if (nt > 0) {
                tmem_ld32(lb + T_O + c * 32, o);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (!ok || !valid) continue;
            uint4 *dst = (uint4 *)(p.ol + w.b * p.ol_b + (long)w.hl * p.ol_h + (long)i * p.ol_r + 256 * rank + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint32_t q[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    q[e] = pack_bf16(__uint_as_float(o[8 * v + 2 * e]) * inv, __uint_as_float(o[8 * v + 2 * e + 1]) * inv);
                dst[v] = make_uint4(q[0], q[1], q[2], q[3]);
            }
        }
        if (ok && valid && rank == 0) p.lse[w.b * p.l_b + (long)(p.head_off + w.hl) * p.l_h + i] = lse;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the peer may still be arriving on this CTA's barriers until here
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

// Launches the latent attention over `units` work units (two CTAs each).
// cache: [B][rows][512] fp16 (+ kpe [B][rows][64] fp16).
cudaError_t launch_latent_attn(const void *cache, const void *kpe, long cache_rows, int B, LatK &p, long units,
                               cudaStream_t st) {
    if (units == 0) return cudaSuccess;
    CUtensorMap mC, mR;
    cudaError_t e;
    {
        unsigned long long d[3] = {512, (unsigned long long)cache_rows, (unsigned long long)B};
        unsigned long long s[2] = {1024, (unsigned long long)cache_rows * 1024};
        unsigned box[3] = {64, NK, 1};
        if ((e = make_tma_map(&mC, cache, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {64, (unsigned long long)cache_rows, (unsigned long long)B};
        unsigned long long s[2] = {128, (unsigned long long)cache_rows * 128};
        unsigned box[3] = {64, NK, 1};
        if ((e = make_tma_map(&mR, kpe, 3, d, s, box)) != cudaSuccess) return e;
    }
    p.idesc_s0 = idesc_f16(128, NK, true);
    p.idesc_s1 = idesc_f16(128, NK, true);
    p.idesc_pv = idesc_f16(128, 256, true, true);
    dim3 grid((unsigned)(2 * units)), block(256);
    ProfScope ps("tc_latent_attn", st);
    e = cudaFuncSetAttribute(tc_latent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e == cudaSuccess) tc_latent_kernel<<<grid, block, SMEM_BYTES, st>>>(mC, mR, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_latent_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_latent_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_latent_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

namespace {

// dst[hl][k][d] = W[hl * Dh + d][k] for d < Dn, k < Dk: the K_nope rows of each head's
// block of W_kv_b, transposed so the absorb product can read them K-major.
__global__ void transpose_wk_kernel(const __nv_bfloat16 *W, int Dh, int Dn, int Dk, __nv_bfloat16 *dst) {
    __shared__ __nv_bfloat16 t[32][33];
    const int hl = blockIdx.z, k0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
    const __nv_bfloat16 *src = W + (long)hl * Dh * Dk;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int d = d0 + r, k = k0 + threadIdx.x;
        t[r][threadIdx.x] = (d < Dn && k < Dk) ? src[(long)d * Dk + k] : __float2bfloat16(0.f);
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int k = k0 + r, d = d0 + threadIdx.x;
        if (k < Dk && d < Dn) dst[((long)hl * Dk + k) * Dn + d] = t[threadIdx.x][r];
    }
}

cudaError_t transpose_wk(const void *w_kv_b, long h0, int nh, int Dh, int Dn, int Dk, void *dst, cudaStream_t st) {
    dim3 grid((Dk + 31) / 32, (Dn + 31) / 32, nh), block(32, 8);
    ProfScope ps("transpose", st);
    transpose_wk_kernel<<<grid, block, 0, st>>>((const __nv_bfloat16 *)w_kv_b + h0 * Dh * Dk, Dh, Dn, Dk,
                                                (__nv_bfloat16 *)dst);
    return cudaGetLastError();
}

// A GEMM operand whose rows per z-slice are `rows` can feed a tile of `tile` rows
// when one box covers whole z-slices or lies inside one.
bool tileable(long rows, int tile) { return rows >= tile || tile % rows == 0; }
int tile_n(long N) { return N >= 256 ? 256 : (N >= 128 ? 128 : 64); }

}  // namespace

bool tc_absorbed_supported(int Dk, int Dn, int Dr, int Dv) {
    return Dk == 512 && Dr == 64 && Dn % 64 == 0 && Dn <= 256 && Dv == 128;
}

bool tc_decode_supported(int Dk, int Dn, int Dr, int Dv, int H) {
    return Dk == 512 && Dr == 64 && Dn % 64 == 0 && Dn <= 256 && Dv == 128 && H % 128 == 0;
}

cudaError_t tc_decode(const TcDecode &p, const void *q_nope, const void *q_pe, const void *c_cache,
                      const void *kpe_cache, const void *w_kv_b, void *out, float *lse, float *po, float *pl,
                      void *po16, bool user_po, void *qabs, void *qpe, void *olat, void *qx, void *qpx,
                      cudaStream_t st) {
    (void)q_pe;   // rotated into qpe (fp16) by the caller
    const long Dh = p.Dn + p.Dv, rows = (long)p.B * p.H;
    cudaError_t e;
    // q_nope is the absorb product's N operand and o_lat the un-absorb product's M operand
    const bool tc_small_gemms = tileable(p.B, tile_n(p.B)) && tileable(p.B, 128);
    // 1. q_abs[b][h][k] = sum_d q_nope[b][h][d] W_K(h)[d][k]  (fp16 out, fp32 accumulate)
    if (tc_small_gemms) {
        // A = W_K(h) read in place, m-major: rows d < Dn of head h's block, k contiguous
        TmaOperand A{w_kv_b, p.Dk, p.Dn, p.H, (long)p.Dk * 2, Dh * p.Dk * 2, p.Dk, 0, 1};
        TmaOperand Bq{q_nope, p.Dn, p.B, p.H, (long)p.H * p.Dn * 2, (long)p.Dn * 2, p.B, 0, 1};
        e = tc_gemm(A, Bq, p.Dk, p.B, p.Dn, p.H, false, qabs, 1, (long)p.H * p.Dk, p.Dk, 0, st, true);
    } else {
        GemmArgs g{};
        g.M = p.B; g.N = p.Dk; g.K = p.Dn; g.nzb = 1; g.nzh = p.H;
        g.A = q_nope; g.ta = TY_BF16; g.a_zh = p.Dn; g.a_m = (long)p.H * p.Dn; g.a_k = 1;
        g.B = w_kv_b; g.tb = TY_BF16; g.b_zh = Dh * p.Dk; g.b_n = 1; g.b_k = p.Dk;
        g.C = qabs; g.tc = TY_F16; g.c_zh = p.Dk; g.c_m = (long)p.H * p.Dk; g.c_n = 1;
        e = launch_gemm_simt(g, st);
    }
    if (e != cudaSuccess) return e;
    if (p.g > 1) {
        // TPLA: g query rows per head, row (b, i, h) zero outside latent shard i
        if ((e = launch_tpla_expand(TY_F16, p.B, p.H, p.g, p.Dk, p.Dr, qabs, qpe, qx, qpx, st)) != cudaSuccess)
            return e;
        // 2. the decode kernel over g*H query rows; at g = 2 with whole 128-head blocks per
        //    shard each unit reads and multiplies only its shard's latent dims
        const int shard_rows = p.g == 2 && p.H % 128 == 0 ? p.H : 0;
        e = launch_decode_attn(qx, qpx, c_cache, kpe_cache, p.B, p.L, p.H * p.g, p.n, p.chunk, p.scale, po, pl, st,
                               shard_rows);
        if (e != cudaSuccess) return e;
        // 3. each shard's merge over its own dims -> o_lat (bf16), shard lse [g][B][H]
        e = launch_tpla_combine(TY_BF16, p.n, p.B, p.H, p.g, p.Dk, po, pl, olat, lse, st);
    } else {
        // 2. per (sequence, split, 128 heads): partial latent output and its lse; 3. the
        //    log-sum-exp merge of the splits -> o_lat (bf16) and lse.  Up to 32 splits the
        //    merge reads fp16 partials (half the bytes of fp32 to write and to read back).
        const bool f16 = p.n <= 32;
        const bool direct16 = f16 && !user_po;
        e = launch_decode_attn(qabs, qpe, c_cache, kpe_cache, p.B, p.L, p.H, p.n, p.chunk, p.scale,
                               direct16 ? (float *)po16 : po, pl, st, 0, direct16);
        if (e != cudaSuccess) return e;
        if (f16 && user_po) e = launch_convert(TY_F32, po, TY_F16, po16, (long)p.n * rows * p.Dk, st);
        if (e != cudaSuccess) return e;
        e = f16 ? launch_lse_combine16(p.n, rows, p.Dk, po16, pl, olat, lse, st)
                : launch_lse_combine(TY_BF16, p.n, rows, p.Dk, po, pl, olat, lse, st);
    }
    if (e != cudaSuccess) return e;
    // 4. out[b][h][d] = sum_k o_lat[b][h][k] W_V(h)[d][k]: rows b (M), columns d (N), so
    //    each output row is written contiguously (a 128-row tile holds B = 64 valid rows)
    if (tc_small_gemms) {
        TmaOperand Ao{olat, p.Dk, p.B, p.H, (long)p.H * p.Dk * 2, (long)p.Dk * 2, p.B, 0, 1};
        TmaOperand Bw{(const char *)w_kv_b + (long)p.Dn * p.Dk * 2, p.Dk, p.Dv, p.H, (long)p.Dk * 2,
                      Dh * p.Dk * 2, p.Dv, 0, 1};
        return tc_gemm(Ao, Bw, p.B, p.Dv, p.Dk, p.H, false, out, (long)p.H * p.Dv, 1, p.Dv, 1, st);
    }
    GemmArgs u{};
    u.M = p.B; u.N = p.Dv; u.K = p.Dk; u.nzb = 1; u.nzh = p.H;
    u.A = olat; u.ta = TY_BF16; u.a_zh = p.Dk; u.a_m = (long)p.H * p.Dk; u.a_k = 1;
    u.B = (const char *)w_kv_b + (long)p.Dn * p.Dk * 2; u.tb = TY_BF16; u.b_zh = Dh * p.Dk; u.b_n = p.Dk; u.b_k = 1;
    u.C = out; u.tc = TY_BF16; u.c_zh = p.Dv; u.c_m = (long)p.H * p.Dv; u.c_n = 1;
    return launch_gemm_simt(u, st);
}

cudaError_t tc_absorbed_prefill(const TcPrefill &p, const void *q_nope, const void *w_kv_b, void *out, float *lse,
                                const void *chat, const void *kpe, const void *qpe, void *qabs, void *olat,
                                void *w16, cudaStream_t st) {
    const long Dh = p.Dn + p.Dv, kv_pad = (p.kv_need + 127) / 128 * 128;
    const long HL = p.head_count;
    cudaError_t e;
    for (int s = 0; s < p.n_shards; ++s) {
        const int h0 = s * p.hs, nh = std::min(p.hs, p.head_count - h0);
        const long hg = p.head_begin + h0;
        if ((e = transpose_wk(w_kv_b, hg, nh, (int)Dh, p.Dn, p.Dk, w16, st)) != cudaSuccess) return e;
        for (int b = 0; b < p.B; ++b) {
            // q_abs[b][i][hl][k] = sum_d q_nope[b][i][h0+hl][d] W_K(hg+hl)[d][k]
            TmaOperand A{(const char *)q_nope + ((long)b * p.s_q * HL + h0) * p.Dn * 2, p.Dn, p.s_q, nh,
                         HL * p.Dn * 2, (long)p.Dn * 2, p.s_q, 0, 1};
            TmaOperand Bw{w16, p.Dn, p.Dk, nh, (long)p.Dn * 2, (long)p.Dk * p.Dn * 2, p.Dk, 0, 1};
            e = tc_gemm(A, Bw, p.s_q, p.Dk, p.Dn, nh, false, (char *)qabs + (long)b * p.s_q * p.hs * p.Dk * 2,
                        (long)p.hs * p.Dk, 1, p.Dk, 0, st);
            if (e != cudaSuccess) return e;
        }
        LatK k{};
        k.s_q = p.s_q;
        k.q_offset = p.q_offset;
        k.kv_need = (int)p.kv_need;
        k.causal = p.causal;
        k.n_qtiles = (p.s_q + ROWS - 1) / ROWS;
        k.nh = nh;
        k.nb = p.B;
        k.head_off = h0;
        k.qa = (const __half *)qabs;
        k.qa_b = (long)p.s_q * p.hs * p.Dk;
        k.qa_h = p.Dk;
        k.qa_r = (long)p.hs * p.Dk;
        k.qp = (const __half *)qpe;
        k.qp_b = (long)p.s_q * HL * p.Dr;
        k.qp_h = p.Dr;
        k.qp_r = HL * p.Dr;
        k.scale_log2 = p.scale * 1.4426950408889634f;
        k.ol = (__nv_bfloat16 *)olat;
        k.ol_b = (long)p.s_q * p.hs * p.Dk;
        k.ol_h = p.Dk;
        k.ol_r = (long)p.hs * p.Dk;
        k.lse = lse;
        k.l_b = HL * p.s_q;
        k.l_h = p.s_q;
        e = launch_latent_attn(chat, kpe, kv_pad, p.B, k, (long)p.B * nh * k.n_qtiles, st);
        if (e != cudaSuccess) return e;
        for (int b = 0; b < p.B; ++b) {
            // out[b][i][h0+hl][d] = sum_k o_lat[b][i][hl][k] W_V(hg+hl)[d][k]
            TmaOperand A{(const char *)olat + (long)b * p.s_q * p.hs * p.Dk * 2, p.Dk, p.s_q, nh,
                         (long)p.hs * p.Dk * 2, (long)p.Dk * 2, p.s_q, 0, 1};
            TmaOperand Bw{(const char *)w_kv_b + (hg * Dh + p.Dn) * p.Dk * 2, p.Dk, p.Dv, nh, (long)p.Dk * 2,
                          Dh * p.Dk * 2, p.Dv, 0, 1};
            e = tc_gemm(A, Bw, p.s_q, p.Dv, p.Dk, nh, false,
                        (char *)out + ((long)b * p.s_q * HL + h0) * p.Dv * 2, HL * p.Dv, 1, p.Dv, 1, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t tc_read_and_clear_error(unsigned int *flags, cudaStream_t st) {
    cudaError_t e = tc_gemm_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_attn_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_latent_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_decode_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_fused_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_bwd_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = simt_read_and_clear_error(flags, st);
    return e;
}

}  // namespace mla
