// tc_decode.cu -- split-KV latent decode on the sm_103a tensor cores.
//
// Method: "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
// (arXiv 2607.17644), Fig. 2 absorbed dataflow and "Core claim" (the absorbed form is
// the decode form): s_hj = scale * (q_abs_h . c_j + RoPE(q_pe_h) . RoPE(k_pe_j)),
// o_h = sum_j softmax_j(s_hj) c_j over the latent cache; "Helix Parallelism ..."
// (arXiv 2507.07120), "What carries the argument": each key split yields a partial
// output and its log-sum-exp, merged afterwards by the rescale-and-sum.
//
// One work unit = the 128 heads of one sequence against one key split.  Its fp32
// accumulator (128 heads x 512 latent dims) fills the whole tensor memory of an SM,
// so a unit runs on a cluster of two CTAs with different jobs:
//   rank 0 (scores): Q in bf16 in TMEM; each 80-key tile of the bf16 cache (latent +
//     RoPE band) arrives through a two-deep TMA ring whose stages fill and drain in
//     three groups of three 64-dim boxes (a group of tile t + 2 loads as soon as tile t's
//     MMAs have read it, which keeps the SM's TMA unit busy); S = Q.K^T
//     on the tensor core (A from TMEM; an N = 80 MMA costs what an N = 64 one does),
//     double-buffered in TMEM, issued by two warps that take alternate tiles, each
//     running its loop warp-uniformly and issuing from one elected lane; eight warps run the online
//     softmax (two threads per head, swapping row maxima through shared memory) and
//     stage P in bf16 (already in the MMA operand layout) in one of two staging slots;
//     a copier warp moves it and the per-head rescale factors into rank 1's shared
//     memory with two bulk copies;
//   rank 1 (accumulator): O (128 x 512 fp32) in all 512 TMEM columns; streams the same
//     tiles' latent rows (L2 hits: an idle warp here prefetches rank 0's next tiles
//     into L2, away from rank 0's TMA unit)
//     and issues O += P.C with both operands in shared memory; four
//     warps rescale rows of O when rank 0 reports a grown row maximum, and write the
//     normalised partial output and the split's log-sum-exp at the end.
// P only flows from rank 0 to rank 1, through two slots, so rank 0 runs ahead and the
// cross-CTA latency stays off the critical path.
//
// Precision.  The tensor core takes bf16 against the bf16 cache, but a score's rounding
// error lands directly in the log-sum-exp of a split with few keys (q_abs rounded to
// bf16: ~1.4e-3 per score on N(0,1) data, in fp16: ~1.7e-4).  So q_abs arrives in fp16
// and is split q = q_hi + q_lo with q_hi = bf16(q):
//   * RoPE band: both halves go through the tensor core (8 more MMAs per tile), so that
//     part of every score is as exact as fp16 q_pe;
//   * latent band: the MMA uses q_hi only.  The missing term delta_j = scale * q_lo . c_j
//     shifts a split's log-sum-exp by sum_j w_j delta_j + O(delta^2), and
//     sum_j w_j delta_j = scale * q_lo . (sum_j w_j c_j) = scale * q_lo . o, the split's
//     own normalised output, which rank 1 holds at the end: it adds that term (the
//     second-order remainder, half the w-variance of delta, is ~1e-6).  The output
//     itself moves by sum_j w_j (delta_j - mean delta) c_j, ~1e-3 of |c| at most.
// P multiplies the cache on rank 1 in bf16: its rounding only perturbs the weights of an
// average (relative 2^-9), and the row sums use the unrounded fp32 probabilities.
//
// TPLA (two latent shards, each with its own softmax): a unit whose heads all belong to
// shard i loads only that shard's four latent boxes and the RoPE box per key tile (in
// two groups of three and two boxes), issues the shard's 16 latent score MMAs and the 8
// RoPE ones, runs P.C at N = 256 over the shard's dims, and writes those dims only.
//
// Warps (384 threads per CTA): rank 0 -- 0 TMA producer, 1 and 11 MMA issuers (1 also
// owns TMEM), 2-9 softmax (two threads per head), 10 copier; rank 1 -- 0 TMA producer,
// 1 MMA issuer and TMEM owner, 2-5 rescale, 2-9 epilogue, 10 L2 prefetch, 11 idle.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_decode_err = 0;

namespace {

using namespace tc;

constexpr int ROWS = 128, NK = 80, NTHREADS = 384;
constexpr int KST = 2;     // rank 0: key-tile stages (one per S buffer)
constexpr int KGRP = 3;    // rank 0: a stage fills and drains in three groups of three boxes
constexpr int VST = 2;     // rank 1: latent-tile stages
constexpr int NPB = 2;     // rank 1: P slots (= rank 0's staging slots)
constexpr int PF1 = 4;     // key tiles prefetched into L2 ahead of rank 1's latent loads
constexpr uint32_t KBOX = NK * 128;         // 80 keys x 64 dims, bf16: 10 KB
constexpr uint32_t KSTAGE = 9 * KBOX;       // boxes 0-7 latent dims, box 8 the RoPE band
constexpr uint32_t VSTAGE = 8 * KBOX;       // 512 latent dims
// One P transfer.  P [128 heads][80 keys] bf16 as the K-major A operand of P.C: keys
// 0-63 in a 128-byte-swizzled block (128 B per head), keys 64-79 in a 32-byte-swizzled
// block (32 B per head).  Then the per-head extras: rescale factor, 1/l and
// m + log2(l) (meaningful on the last tile), and one "some head rescaled" word per lane
// quarter.
constexpr uint32_t P_BLK1 = 16384, P_BYTES = 16384 + 4096;
constexpr uint32_t X_ALPHA = 0, X_INVL = 512, X_LSE = 1024, X_FLAG = 1536, X_BYTES = X_FLAG + 16;
constexpr uint32_t XOFF = P_BYTES;           // extras within a rank-1 slot
constexpr uint32_t XSLOT = 22528;            // rank-1 slot stride (1024-aligned)
// rank 0: K stages, two P staging slots, their extras, the two halves' row maxima
// (double-buffered); rank 1: latent stages, then the P slots.  The barriers sit after
// both layouts, at the same offset in both CTAs (the peer addresses them by offset).
constexpr uint32_t OFF_STG = KST * KSTAGE, OFF_EXT = OFF_STG + NPB * P_BYTES, EXT_STRIDE = 1664;
constexpr uint32_t OFF_RED = OFF_EXT + NPB * EXT_STRIDE;
constexpr uint32_t OFF_PB = VST * VSTAGE, OFF_RED1 = OFF_PB + NPB * XSLOT;   // rank 1: the epilogue's dot halves
// rank 1's epilogue, in the latent stages once the last MMAs are done: eight 4 KB output
// staging buffers, then the q_abs block (eight 16 KB boxes)
constexpr uint32_t QB_OFF = 8 * 4096;
static_assert(QB_OFF + 8 * 16384 <= OFF_PB, "epilogue staging fits the latent stages");
constexpr uint32_t END0 = OFF_RED + 2 * 2 * ROWS * 4, END1 = OFF_RED1 + 2 * ROWS * 4;
constexpr uint32_t OFF_BAR = END0 > END1 ? END0 : END1;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;
// rank 0 TMEM columns: S buffers; bf16 q_hi of the latent band (256 columns); the RoPE
// band's q_hi and q_lo (32 columns each)
constexpr uint32_t T_S = 0, T_Q = 2 * NK, T_QP = T_Q + 256, T_QL = T_QP + 32;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr unsigned FULL = 0xffffffffu;

static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(KSTAGE % 1024 == 0 && OFF_STG % 1024 == 0 && P_BYTES % 1024 == 0 && OFF_PB % 1024 == 0 &&
                  XSLOT % 1024 == 0,
              "swizzle atoms aligned");
static_assert(XOFF + X_BYTES <= XSLOT && X_BYTES <= EXT_STRIDE && OFF_EXT % 16 == 0, "P transfer layout");
static_assert(T_QL + 32 <= 512, "TMEM budget of rank 0");
static_assert(NK == 80, "P layout: one 64-key block and one 16-key block");

struct DecK {
    int n_splits, row_tiles;
    long chunk, kv_len;                 // keys per split, cache length
    const __half *qa;                   // q_abs rows [b][h][512]
    long qa_b, qa_r;
    const __half *qp;                   // rotated q_pe rows [b][h][64]
    long qp_b, qp_r;
    const __nv_bfloat16 *cache, *kpe;   // [B][kv_len][512], [B][kv_len][64] (for the L2 prefetch)
    float scale_log2;
    float *po, *pl;                     // partials [split][b][h][512], [split][b][h]
    int po16;                           // the partial outputs in fp16 (else fp32)
    long po_s, po_b, pl_s, pl_b;
    uint32_t idesc_s, idesc_pv;
    // TPLA with two latent shards: rows [b][i][h] of g = 2 shards x shard_rows heads
    // (shard_rows a multiple of 128, so a unit's heads all belong to shard r0 /
    // shard_rows); 0 = plain decode over all 512 dims
    int shard_rows;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Unit {
    int b, split, r0;   // sequence, key split, first head
    int shard;          // TPLA latent shard of the unit's rows (dims 256 shard ..), -1 = all dims
    long kb, ke;        // key range [kb, ke)
    int nt;             // key tiles
};

__device__ __forceinline__ Unit unit_of(const DecK &p, int u) {
    Unit w{};
    w.r0 = (u % p.row_tiles) * ROWS;
    u /= p.row_tiles;
    w.split = u % p.n_splits;
    w.b = u / p.n_splits;
    w.kb = min((long)w.split * p.chunk, p.kv_len);
    w.ke = min(w.kb + p.chunk, p.kv_len);
    w.nt = w.ke > w.kb ? (int)((w.ke - w.kb + NK - 1) / NK) : 0;
    w.shard = p.shard_rows ? w.r0 / p.shard_rows : -1;
    return w;
}

// After an abandoned wait: give TMA loads that were already issued time to land
// before the CTA's shared memory is released (bounded: 100 microseconds).
__device__ void settle() {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 100000ull) {
    }
}

// SHD: the TPLA two-shard units (a template parameter so that the plain decode's issue
// loops carry no shard branches).
template <bool SHD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap mC, const __grid_constant__ CUtensorMap mR,
                     const __grid_constant__ CUtensorMap mP, const __grid_constant__ CUtensorMap mQa,
                     const __grid_constant__ CUtensorMap mQp, DecK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + OFF_BAR);
    // rank 0: s_free = S buffer drained by the softmax warps; grp_full / grp_empty
    // [stage][group] = three boxes of a stage landed / read by the MMAs; staged = the softmax warps
    // have staged the tile's P; stg_free = the copy to rank 1 has read the staging slot
    uint64_t *s_free = bars, *stg_free = bars + 2, *s_full = bars + 6, *staged = bars + 8;
    uint64_t *grp_full = bars + 32, *grp_empty = bars + 32 + KST * KGRP;   // [stage][group]
    uint64_t *q_ready = bars + 10, *q_full = bars + 30;   // Q in TMEM / Q staged in the K stages
    uint64_t *qb_full = bars + 31;   // rank 1: the q_abs block staged for the epilogue
    float *red = (float *)(smem + OFF_RED);   // rank 0: [tile parity][half][row] row maxima
    // both: P slot t % NPB consumed by the P.C MMAs of tile t (one multicast commit
    // completes it in both CTAs)
    uint64_t *p_empty = bars + 11;
    // rank 1
    uint64_t *p_full = bars + 14, *pc_ready = bars + 17, *v_full = bars + 20, *v_empty = bars + 24;
    uint64_t *o_final = bars + 28;
    uint32_t *tslot = (uint32_t *)(bars + 29);
    volatile int *abort = (volatile int *)(tslot + 1);
    volatile int *prog = (volatile int *)(bars + 27);   // rank 1: latent tiles whose loads are issued
    unsigned *err = &g_tc_decode_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const Unit w = unit_of(p, blockIdx.x >> 1);
    const int nt = w.nt;
    constexpr bool shd = SHD;
    const int box0 = shd ? 4 * w.shard : 0;   // first latent box of the unit's dims
    constexpr int ngrp = shd ? 2 : KGRP;      // box groups per key stage

    if (tid == 0) {
        if (rank == 0) {
            for (int s = 0; s < KST; ++s) {
                mbar_init(&s_free[s], 8);   // one arrival per softmax warp
                mbar_init(&stg_free[s], 1);
                mbar_init(&s_full[s], 1);
                mbar_init(&staged[s], 8);
            }
            for (int i = 0; i < KST * KGRP; ++i) {
                mbar_init(&grp_full[i], 1);
                mbar_init(&grp_empty[i], 1);
            }
            mbar_init(q_ready, 8);
            mbar_init(q_full, 1);
        } else {
            for (int s = 0; s < NPB; ++s) {
                mbar_init(&p_full[s], 1);   // this CTA's expect_tx + the bytes of rank 0's stores
                mbar_init(&pc_ready[s], 4);
            }
            for (int s = 0; s < VST; ++s) {
                mbar_init(&v_full[s], 1);
                mbar_init(&v_empty[s], 1);
            }
            mbar_init(o_final, 1);
            mbar_init(qb_full, 1);
        }
        for (int s = 0; s < NPB; ++s) mbar_init(&p_empty[s], 1);
        *abort = 0;
        *prog = 0;
        fence_mbar_init();
        if (rank == 0) {   // both S buffers start free: the softmax warps' arrivals for tiles 0 and 1
            for (int s = 0; s < KST; ++s)
                for (int i = 0; i < 8; ++i) mbar_arrive(&s_free[s]);
        } else {           // every P slot armed for its first transfer
            for (int s = 0; s < NPB; ++s) mbar_arrive_expect_tx(&p_full[s], P_BYTES + X_BYTES);
        }
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrival
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (rank == 0) {
        if (warp == 0) {
            // ---------------------------------------------------------------- TMA producer
            if (lane == 0 && nt > 0) {
                tma_prefetch_desc(&mC);
                tma_prefetch_desc(&mR);
                // the unit's Q block (128 heads: q_abs in eight 64-dim boxes, the rotated
                // q_pe in one) staged in the K stages; the softmax threads move it to TMEM
                tma_prefetch_desc(&mQa);
                tma_prefetch_desc(&mQp);
                const int qrow = w.b * p.row_tiles * ROWS + w.r0;
                mbar_arrive_expect_tx(q_full, 9 * 128 * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i) tma_load_2d(smem + i * 16384, &mQa, q_full, 64 * i, qrow);
                tma_load_2d(smem + 8 * 16384, &mQp, q_full, 0, qrow);
                // the stages hold Q until it is in TMEM
                bool go = mbar_wait(q_ready, 0, abort, err);
                for (int t = 0; t < nt && go; ++t) {
                    const int s = t & 1;
                    const uint32_t ph = ((t >> 1) - 1) & 1;   // phase of tile t - 2 in this stage
                    uint8_t *dst = smem + s * KSTAGE;
                    const int key0 = (int)(w.kb + (long)t * NK);
                    for (int g = 0; g < ngrp && go; ++g) {   // a group refills once tile t - 2 has read it
                        uint64_t *full = &grp_full[s * KGRP + g];
                        if (t >= KST && !mbar_wait(&grp_empty[s * KGRP + g], ph, abort, err)) go = false;
                        if (!go) break;
                        if (!shd) {
                            mbar_arrive_expect_tx(full, 3 * KBOX);
                            for (int i = 3 * g; i < 3 * g + 3; ++i) {
                                if (i < 8) tma_load_3d(dst + i * KBOX, &mC, full, 64 * i, key0, w.b);
                                else tma_load_3d(dst + 8 * KBOX, &mR, full, 0, key0, w.b);
                            }
                        } else {   // the shard's boxes 0-3 (group 0: three, group 1: one + RoPE)
                            mbar_arrive_expect_tx(full, (g == 0 ? 3 : 2) * KBOX);
                            for (int j = 3 * g; j < 3 * g + 3 && j < 5; ++j) {
                                const int i = box0 + j;   // same slot as in the full layout
                                if (j < 4) tma_load_3d(dst + i * KBOX, &mC, full, 64 * i, key0, w.b);
                                else tma_load_3d(dst + 8 * KBOX, &mR, full, 0, key0, w.b);
                            }
                        }
                    }
                    if (!go) break;
                }
            }
        } else if (warp == 1 || warp == 11) {
            // --------------------- S = Q.K^T issuers: warp 1 even tiles, warp 11 odd tiles
            // The whole warp runs the loop and one elected lane issues: with warp-uniform
            // control flow the operands stay in uniform registers and an MMA issues in
            // about two thirds of the time a lane-divergent issuer takes.
            if (nt > 0) {
                bool ok = __all_sync(FULL, mbar_wait(q_ready, 0, abort, err));
                for (int t = warp == 1 ? 0 : 1; t < nt && ok; t += 2) {
                    const int s = t & 1;
                    const uint32_t ph = (t >> 1) & 1;
                    // S buffer s drained by the softmax, then the stage group by group
                    if (!__all_sync(FULL, mbar_wait(&s_free[s], ph, abort, err))) break;
                    const uint64_t d0 = sdesc_kmajor(smem + s * KSTAGE);
                    const uint32_t dt = tmem + T_S + s * NK, at = tmem + T_Q;
                    bool go = true;
#pragma unroll
                    for (int g = 0; g < KGRP; ++g) {
                        if (g >= ngrp) break;
                        go = go && __all_sync(FULL, mbar_wait(&grp_full[s * KGRP + g], ph, abort, err));
                        if (!go) break;
                        tc_fence_after();
                        if (elect_one()) {
                            if (!shd) {
#pragma unroll
                                for (int kk = 12 * g; kk < 12 * g + 12 && kk < 32; ++kk)   // latent band, q_hi only
                                    mma_ts(dt, at + kk * 8, d0 + (uint64_t)((kk >> 2) * (KBOX >> 4) + 2 * (kk & 3)),
                                           p.idesc_s, kk != 0);
                            } else {   // the shard's latent boxes of this group
#pragma unroll
                                for (int j = 3 * g; j < 3 * g + 3 && j < 4; ++j)
#pragma unroll
                                    for (int q = 0; q < 4; ++q) {
                                        const int kk = 4 * (box0 + j) + q;
                                        mma_ts(dt, at + kk * 8, d0 + (uint64_t)((box0 + j) * (KBOX >> 4) + 2 * q),
                                               p.idesc_s, (j | q) != 0);
                                    }
                            }
                            if (g == ngrp - 1) {
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk)   // RoPE band: q_hi then q_lo against the same box
                                    mma_ts(dt, tmem + (kk < 4 ? T_QP : T_QL) + (kk & 3) * 8,
                                           d0 + (uint64_t)(8 * (KBOX >> 4) + 2 * (kk & 3)), p.idesc_s, 1);
                            }
                            mma_commit(&grp_empty[s * KGRP + g]);
                            if (g == ngrp - 1) mma_commit(&s_full[s]);
                        }
                        __syncwarp();
                    }
                    if (!go) break;
                }
            }
        } else if (warp >= 2 && warp < 10) {
            // ---------------------------------------------------------- softmax warps
            // two threads per head: warps 2-5 take keys 0-39 of a tile, warps 6-9 keys 40-79
            const int quad = warp & 3, row = quad * 32 + lane, h = (warp - 2) >> 2;
            const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
            if (nt > 0) {
                // this head's Q into TMEM from the staged block: bf16(q_abs) (steps 0-15),
                // then the RoPE band's bf16 halves (steps 16-17), 32 fp16 values per step; a
                // step is half a 128-byte row of a box (16-byte chunk j at j ^ (row mod 8));
                // the head's two threads take nine steps each
                const bool staged_q = __all_sync(FULL, mbar_wait(q_full, 0, abort, err));
                for (int c = 9 * h; c < 9 * h + 9 && staged_q; ++c) {
                    const uint8_t *box = smem + (c < 16 ? (c >> 1) : 8) * 16384 + row * 128;
                    const int half = c < 16 ? (c & 1) : c - 16;
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 x = *(const uint4 *)(box + (((half * 4 + v) ^ (row & 7)) << 4));
                        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[e]));
                            const uint32_t hb = pack_bf16(f.x, f.y);
                            hi[4 * v + e] = hb;
                            lo[4 * v + e] =
                                pack_bf16(f.x - __uint_as_float(hb << 16), f.y - __uint_as_float(hb & 0xffff0000u));
                        }
                    }
                    if (c < 16) {
                        tmem_st16(lb + T_Q + c * 16, hi);
                    } else {
                        tmem_st16(lb + T_QP + (c - 16) * 16, hi);
                        tmem_st16(lb + T_QL + (c - 16) * 16, lo);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(q_ready);
            }
            const float c = p.scale_log2;
            constexpr int HK = NK / 2;   // keys per thread
            float m = -INFINITY, l = 0.f;   // running maximum (scaled, log2 units), this half's sum
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const int s = t & 1;
                ok = __all_sync(FULL, ok && mbar_wait(&s_full[s], (t >> 1) & 1, abort, err));
                tc_fence_after();
                uint32_t sa[32], sb[8];
                if (ok) {   // half 0: columns 0-31, 32-39; half 1: columns 40-47, 48-79
                    const uint32_t base = lb + T_S + s * NK + h * HK;
                    if (h == 0) {
                        tmem_ld32(base, sa);
                        tmem_ld8(base + 32, sb);
                    } else {
                        tmem_ld8(base, sb);
                        tmem_ld32(base + 8, sa);
                    }
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) sa[e] = 0u;
#pragma unroll
                    for (int e = 0; e < 8; ++e) sb[e] = 0u;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[s]);   // S buffer s may take tile t + 2
                float x[HK];   // this thread's keys, in key order
#pragma unroll
                for (int e = 0; e < HK; ++e)
                    x[e] = __uint_as_float(h == 0 ? (e < 32 ? sa[e] : sb[e - 32]) : (e < 8 ? sb[e] : sa[e - 8]));
                const long key0 = w.kb + (long)t * NK + h * HK;
                if (key0 + HK > w.ke) {
#pragma unroll
                    for (int e = 0; e < HK; ++e)
                        if (key0 + e >= w.ke) x[e] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
                for (int e = 8; e < HK; ++e) mx[e & 7] = fmaxf(mx[e & 7], x[e]);
                float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                // the row maximum of the tile: this half's and the partner thread's
                red[(s * 2 + h) * ROWS + row] = mt;
                named_bar_sync(1, 256);
                mt = fmaxf(mt, red[(s * 2 + (h ^ 1)) * ROWS + row]) * c;
                // the accumulator is rescaled only when the row maximum grows by > 2^8
                // (both threads of a row take the same decision from the same numbers)
                const bool need = mt > m + RESCALE_LOG2;
                float alpha = 1.f;
                if (need) {
                    alpha = m == -INFINITY ? 0.f : ex2(m - mt);
                    m = mt;
                }
                l *= alpha;
                const float m_eff = m == -INFINITY ? 0.f : m;
                float ra[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint32_t pk[HK / 2];
#pragma unroll
                for (int e = 0; e < HK / 2; ++e) {
                    const float p0 = ex2(fmaf(x[2 * e], c, -m_eff)), p1 = ex2(fmaf(x[2 * e + 1], c, -m_eff));
                    ra[e & 7] += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                l += ((ra[0] + ra[1]) + (ra[2] + ra[3])) + ((ra[4] + ra[5]) + (ra[6] + ra[7]));
                const bool rescaled = __any_sync(FULL, need && t > 0);
                uint8_t *ext = smem + OFF_EXT + s * EXT_STRIDE;
                if (t == nt - 1) {   // the row's sum: this half's plus the partner's (the other
                                     // parity's slots: both threads are past their last reads)
                    red[((s ^ 1) * 2 + h) * ROWS + row] = l;
                    named_bar_sync(1, 256);
                    const float lt = l + red[((s ^ 1) * 2 + (h ^ 1)) * ROWS + row];
                    if (h == 0) {
                        ((float *)(ext + X_INVL))[row] = lt > 0.f ? 1.f / lt : 0.f;
                        ((float *)(ext + X_LSE))[row] = lt > 0.f ? m + log2f(lt) : -INFINITY;
                    }
                }
                // staging slot s: its copy of tile t - 2 has read it
                if (t >= 2) ok = __all_sync(FULL, ok && mbar_wait(&stg_free[s], ((t >> 1) - 1) & 1, abort, err));
                // 16-byte chunk j holds keys 8j .. 8j+7 of the tile
                uint8_t *stg = smem + OFF_STG + s * P_BYTES;
#pragma unroll
                for (int q = 0; q < HK / 8; ++q) {
                    const int j = h * (HK / 8) + q;
                    uint8_t *dst = j < 8 ? stg + row * 128 + ((j ^ (row & 7)) << 4)
                                         : stg + P_BLK1 + row * 32 + (((j - 8) ^ ((row >> 2) & 1)) << 4);
                    *(uint4 *)dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
                if (h == 0) {
                    ((float *)(ext + X_ALPHA))[row] = alpha;
                    if (lane == 0) ((uint32_t *)(ext + X_FLAG))[quad] = rescaled ? 1u : 0u;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&staged[s]);
            }
        } else if (warp == 10) {
            // ------------------------------- copier: staged P and extras -> rank 1
            if (lane == 0 && nt > 0) {
                const uint32_t peer_slot0 = map_peer(smem_u32(smem + OFF_PB), 1);
                const uint32_t peer_full0 = map_peer(smem_u32(p_full), 1);   // armed by rank 1 itself
                for (int t = 0; t < nt; ++t) {
                    const int s = t & 1, pb = t % NPB;
                    if (!mbar_wait(&staged[s], (t >> 1) & 1, abort, err)) break;
                    // P slot pb of rank 1 is free once its P.C MMAs of tile t - NPB are done
                    if (t >= NPB && !mbar_wait_cluster(&p_empty[pb], ((t / NPB) - 1) & 1, abort, err)) break;
                    const uint32_t dst = peer_slot0 + pb * XSLOT, bar = peer_full0 + pb * 8;
                    bulk_copy_to_peer(dst, smem + OFF_STG + s * P_BYTES, P_BYTES, bar);
                    bulk_copy_to_peer(dst + XOFF, smem + OFF_EXT + s * EXT_STRIDE, X_BYTES, bar);
                    bulk_commit();
                    bulk_wait_read<0>();   // the staging has been read
                    mbar_arrive(&stg_free[s]);
                }
                bulk_wait_all();   // nothing in flight into the peer at exit
            }
        }
    } else {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer (latent rows)
            if (lane == 0 && nt > 0) {
                tma_prefetch_desc(&mC);
                for (int t = 0; t < nt; ++t) {
                    const int s = t % VST;
                    if (t >= VST && !mbar_wait(&v_empty[s], ((t / VST) - 1) & 1, abort, err)) break;
                    uint8_t *dst = smem + s * VSTAGE;
                    const int key0 = (int)(w.kb + (long)t * NK);
                    constexpr int nbx = shd ? 4 : 8;   // the unit's latent boxes, into slots 0 ..
                    mbar_arrive_expect_tx(&v_full[s], nbx * KBOX);
#pragma unroll
                    for (int i = 0; i < nbx; ++i)
                        tma_load_3d(dst + i * KBOX, &mC, &v_full[s], 64 * (box0 + i), key0, w.b);
                    *prog = t + 1;   // paces the prefetching warp
                    if (t == (nt > 3 ? nt - 3 : 0)) {   // the epilogue's q_abs rows (128 KB) into L2
                        const __half *q0 = p.qa + w.b * p.qa_b + (long)w.r0 * p.qa_r;
                        for (int k = 0; k < 8; ++k) l2_prefetch(q0 + k * 16 * 512, 16 * 1024);
                    }
                }
                // once the last P.C MMAs are done the latent stages are free: the unit's
                // q_abs block goes there for the epilogue (eight 64-dim boxes of 128 rows)
                if (mbar_wait(o_final, 0, abort, err)) {
                    tma_prefetch_desc(&mQa);
                    const int qrow = w.b * p.row_tiles * ROWS + w.r0;
                    mbar_arrive_expect_tx(qb_full, 8 * 128 * 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i) tma_load_2d(smem + QB_OFF + i * 16384, &mQa, qb_full, 64 * i, qrow);
                }
            }
        } else if (warp == 10) {
            // ------------------------------- L2 prefetch of the key tiles rank 0 loads next
            // Issued from this CTA, whose TMA unit has room: a thread issuing bulk
            // prefetches waits behind them, and in rank 0's producer that wait held back
            // every stage refill.  This CTA's latent loads trail rank 0's key loads by
            // about two tiles; tile t + PF1 is prefetched once tile t's rows load here.
            if (lane == 0 && nt > 0) {
                auto prefetch = [&](int t) {
                    const long key0 = w.kb + (long)t * NK;
                    const int rows = (int)min((long)NK, p.kv_len - key0);
                    const long row = (long)w.b * p.kv_len + key0;
                    for (int r = 0; r < rows; r += 16)
                        l2_prefetch(p.cache + (row + r) * 512, (uint32_t)min(16, rows - r) * 1024u);
                    l2_prefetch(p.kpe + row * 64, (uint32_t)rows * 128u);
                };
                for (int t = 0; t < nt && t < PF1; ++t) prefetch(t);
                const uint64_t t0 = global_ns();
                for (int t = PF1; t < nt; ++t) {
                    bool ok = true;
                    while (*prog < t - PF1 + 1) {   // the latent loads of tile t - PF1 are issued
                        if (*abort || global_ns() - t0 > WAIT_NS) {
                            ok = false;
                            break;
                        }
                        __nanosleep(128);
                    }
                    if (!ok) break;
                    prefetch(t);
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------- O += P.C issuer
            // (warp-uniform loop, one elected lane issues, as for the score MMAs)
            if (nt > 0) {
                bool ok = true;
                for (int t = 0; t < nt; ++t) {
                    const int s = t % VST, pb = t % NPB;
                    ok = __all_sync(FULL, mbar_wait(&v_full[s], (t / VST) & 1, abort, err));
                    ok = ok && __all_sync(FULL, mbar_wait(&pc_ready[pb], (t / NPB) & 1, abort, err));
                    if (!ok) break;
                    tc_fence_after();
                    const uint8_t *slot = smem + OFF_PB + pb * XSLOT;
                    const uint64_t pa0 = sdesc_kmajor(slot), pa1 = sdesc_kmajor_sw32(slot + P_BLK1);
                    const uint64_t vb = sdesc_mnmajor(smem + s * VSTAGE, KBOX);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < NK / 16; ++kk) {   // 16 keys per step; N = 256 latent dims per MMA
                            const uint64_t pa = kk < 4 ? pa0 + (uint64_t)(2 * kk) : pa1;
                            const uint32_t acc = (t | kk) != 0;
                            mma_ss(tmem, pa, vb + (uint64_t)(kk * (2048 >> 4)), p.idesc_pv, acc);
                            if (!shd)
                                mma_ss(tmem + 256, pa, vb + (uint64_t)((4 * KBOX + kk * 2048) >> 4), p.idesc_pv, acc);
                        }
                        mma_commit(&v_empty[s]);
                        mma_commit_mc(&p_empty[pb], 3);   // slot pb consumed: tells rank 0 and this CTA
                    }
                    __syncwarp();
                }
                if (elect_one()) mma_commit(o_final);
                __syncwarp();
            }
        } else if (warp >= 2 && warp < 10) {
            // ------------------------ row rescale (warps 2-5) + epilogue (warps 2-9)
            const int quad = warp & 3, row = quad * 32 + lane, g = (warp - 2) >> 2;
            const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
            float inv_l = 0.f, lse2 = -INFINITY;   // 1/l and m + log2(l) from rank 0's last transfer
            bool ok = true;
            for (int t = 0; t < nt && ok && g == 0; ++t) {
                const int pb = t % NPB;
                ok = __all_sync(FULL, mbar_wait_cluster(&p_full[pb], (t / NPB) & 1, abort, err));
                if (!ok) break;
                if (warp == 2 && lane == 0 && t + NPB < nt)   // arm the slot for tile t + NPB
                    mbar_arrive_expect_tx(&p_full[pb], P_BYTES + X_BYTES);
                const uint8_t *xs = smem + OFF_PB + pb * XSLOT + XOFF;
                const uint32_t *fl = (const uint32_t *)(xs + X_FLAG);
                if ((fl[0] | fl[1] | fl[2] | fl[3]) != 0u) {   // the same answer in every thread
                    // O must hold tile t - 1's product before it is rescaled.  Slot q's
                    // previous phase is waited for first, so the parity test is never
                    // two phases behind.
                    const int q = (t - 1) % NPB, k = (t - 1) / NPB;
                    bool gw = k == 0 || mbar_wait(&p_empty[q], (k - 1) & 1, abort, err);
                    gw = gw && mbar_wait(&p_empty[q], k & 1, abort, err);
                    ok = __all_sync(FULL, gw);
                    if (!ok) break;
                    tc_fence_after();
                    const float a = ((const float *)(xs + X_ALPHA))[row];
                    if (__any_sync(FULL, a != 1.f)) {
                        for (int cc = 0; cc < (shd ? 8 : 16); ++cc) {
                            uint32_t o[32];
                            tmem_ld32(lb + cc * 32, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                            tmem_st32(lb + cc * 32, o);
                        }
                        tmem_st_wait();
                    }
                    tc_fence_before();
                }
                if (t == nt - 1) {
                    inv_l = ((const float *)(xs + X_INVL))[row];
                    lse2 = ((const float *)(xs + X_LSE))[row];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&pc_ready[pb]);
            }
            // ---- epilogue: the normalised partial output of this split (warps 2-5 latent
            // dims 0-255, warps 6-9 dims 256-511) and its log-sum-exp with the first-order
            // term of the latent q_lo added.  The q_abs row is loaded before the wait.
            // 1/l of the row from the warps that received the transfers
            float *red1 = (float *)(smem + OFF_RED1);
            if (g == 0) red1[ROWS + row] = inv_l;
            named_bar_sync(2, 256);
            if (g == 1) inv_l = red1[ROWS + row];
            if (ok && nt > 0) ok = mbar_wait(o_final, 0, abort, err);
            if (ok && nt > 0) ok = mbar_wait(qb_full, 0, abort, err);
            ok = __all_sync(FULL, ok);
            tc_fence_after();
            float dot[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
                // 32 x 32 fp32 blocks staged per warp in the (now idle) latent stages, 128-byte
                // swizzled (chunk j of a row at j ^ (row mod 8)), written by TMA tile stores
                uint8_t *buf = smem + (warp - 2) * 4096;
                const int prow = (int)(((long)w.split * p.po_s + w.b * p.po_b) / 512) + w.r0 + quad * 32;
                if (lane == 0) tma_prefetch_desc(&mP);
                // kept rolled: the body's code is fetched once (the cache stream leaves no code in L2)
                // this warp's columns: TMEM column tc0 + 32 cc holds latent dim od0 + 32 cc
                constexpr int ncc = shd ? 4 : 8;
                const int tc0 = shd ? 128 * g : 256 * g, od0 = 256 * (shd ? w.shard : 0) + tc0;
#pragma unroll 1
                for (int cc = 0; cc < ncc; ++cc) {
                    uint32_t o[32];
                    if (nt > 0) {
                        tmem_ld32(lb + tc0 + cc * 32, o);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    float ov[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __uint_as_float(o[e]) * inv_l;
                    if (!p.po16) {
                        if (cc >= 1) {   // the previous chunk's store has read the buffer
                            if (lane == 0) bulk_wait_read<0>();
                            __syncwarp();
                        }
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *(float4 *)(buf + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                                make_float4(ov[4 * v], ov[4 * v + 1], ov[4 * v + 2], ov[4 * v + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {   // columns in fp16 units of the map: 2 per fp32 value
                            tma_store_2d(&mP, buf, (od0 + 32 * cc) * 2, prow);
                            bulk_commit();
                        }
                    } else {
                        // fp16: two chunks fill one 128-byte row (chunk cc in its half cc & 1),
                        // one TMA tile store per pair
                        const int h = cc & 1;
                        if (cc >= 2 && h == 0) {   // the previous pair's store has read the buffer
                            if (lane == 0) bulk_wait_read<0>();
                            __syncwarp();
                        }
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            *(uint4 *)(buf + lane * 128 + (((4 * h + v) ^ (lane & 7)) << 4)) =
                                make_uint4(pack_f16(ov[8 * v], ov[8 * v + 1]), pack_f16(ov[8 * v + 2], ov[8 * v + 3]),
                                           pack_f16(ov[8 * v + 4], ov[8 * v + 5]), pack_f16(ov[8 * v + 6], ov[8 * v + 7]));
                        if (h == 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&mP, buf, od0 + 32 * (cc - 1), prow);
                                bulk_commit();
                            }
                        }
                    }
                    // dims od0 + 32 cc .. +31: half (od / 32) & 1 of the row of box od / 64
                    const int od = od0 + 32 * cc;
                    const uint8_t *qrow_s = smem + QB_OFF + (od >> 6) * 16384 + row * 128;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {   // q_lo = q - bf16(q), rounded as rank 0 rounded q_hi
                        const uint4 x = *(const uint4 *)(qrow_s + (((((od >> 5) & 1) * 4 + v) ^ (row & 7)) << 4));
                        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[e]));
                            const uint32_t hb = pack_bf16(f.x, f.y);
                            dot[e] = fmaf(f.x - __uint_as_float(hb << 16), ov[8 * v + 2 * e], dot[e]);
                            dot[e] = fmaf(f.y - __uint_as_float(hb & 0xffff0000u), ov[8 * v + 2 * e + 1], dot[e]);
                        }
                    }
                }
            }
            if (lane == 0) bulk_wait_all();   // the partial output is written before exit
            // the two halves' dot products meet in shared memory
            if (g == 1) red1[row] = (dot[0] + dot[1]) + (dot[2] + dot[3]);
            named_bar_sync(3, 256);
            if (g == 0 && ok) {
                const float corr = ((dot[0] + dot[1]) + (dot[2] + dot[3]) + red1[row]) * p.scale_log2;
                p.pl[w.split * p.pl_s + w.b * p.pl_b + w.r0 + row] =
                    nt > 0 && lse2 > -INFINITY ? (lse2 + corr) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
    if (tid == 0 && *abort) settle();
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the peer may still address this CTA's barriers and slots until here
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

// Partial latent outputs and log-sum-exps of every (sequence, key split, 128 heads).
// qa: q_abs [B][H][512] fp16; qp: rotated q_pe [B][H][64] fp16; cache [B][L][512],
// kpe [B][L][64] bf16; po [n][B][H][512] fp32, pl [n][B][H].
cudaError_t launch_decode_attn(const void *qa, const void *qp, const void *cache, const void *kpe, int B, long L,
                               int H, int n_splits, long chunk, float scale, float *po, float *pl, cudaStream_t st,
                               int shard_rows, bool po16) {
    if (po16 && shard_rows) return cudaErrorInvalidValue;   // the two-shard units write fp32 only
    const long units = (long)B * n_splits * (H / ROWS);
    if (units == 0) return cudaSuccess;
    if (shard_rows && (shard_rows % ROWS != 0 || H != 2 * shard_rows)) return cudaErrorInvalidValue;
    CUtensorMap mC, mR, mP, mQa, mQp;
    cudaError_t e;
    {   // q_abs [B * H][512] and the rotated q_pe [B * H][64], fp16, boxes of 128 rows
        unsigned long long d[2] = {512, (unsigned long long)B * H}, s[1] = {1024};
        unsigned box[2] = {64, 128};
        if ((e = make_tma_map(&mQa, qa, 2, d, s, box)) != cudaSuccess) return e;
        unsigned long long dp[2] = {64, (unsigned long long)B * H}, sp[1] = {128};
        if ((e = make_tma_map(&mQp, qp, 2, dp, sp, box)) != cudaSuccess) return e;
    }
    if (!po16) {   // the fp32 partial output as rows of 1024 16-bit units (2 KB), boxes of 32 x 32 fp32
        unsigned long long d[2] = {1024, (unsigned long long)n_splits * B * H};
        unsigned long long s[1] = {2048};
        unsigned box[2] = {64, 32};
        if ((e = make_tma_map(&mP, po, 2, d, s, box)) != cudaSuccess) return e;
    } else {       // fp16 partials: rows of 512 (1 KB), boxes of 32 rows x 64
        unsigned long long d[2] = {512, (unsigned long long)n_splits * B * H};
        unsigned long long s[1] = {1024};
        unsigned box[2] = {64, 32};
        if ((e = make_tma_map(&mP, po, 2, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {512, (unsigned long long)L, (unsigned long long)B};
        unsigned long long s[2] = {1024, (unsigned long long)L * 1024};
        unsigned box[3] = {64, NK, 1};
        if ((e = make_tma_map(&mC, cache, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {64, (unsigned long long)L, (unsigned long long)B};
        unsigned long long s[2] = {128, (unsigned long long)L * 128};
        unsigned box[3] = {64, NK, 1};
        if ((e = make_tma_map(&mR, kpe, 3, d, s, box)) != cudaSuccess) return e;
    }
    DecK p{};
    p.n_splits = n_splits;
    p.row_tiles = H / ROWS;
    p.chunk = chunk;
    p.kv_len = L;
    p.qa = (const __half *)qa;
    p.qa_b = (long)H * 512;
    p.qa_r = 512;
    p.qp = (const __half *)qp;
    p.qp_b = (long)H * 64;
    p.qp_r = 64;
    p.cache = (const __nv_bfloat16 *)cache;
    p.kpe = (const __nv_bfloat16 *)kpe;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.po = po;
    p.pl = pl;
    p.po_s = (long)B * H * 512;
    p.po_b = (long)H * 512;
    p.pl_s = (long)B * H;
    p.pl_b = H;
    p.idesc_s = idesc_f16(128, NK, false);
    p.idesc_pv = idesc_f16(128, 256, false, true);
    p.shard_rows = shard_rows;
    p.po16 = po16 ? 1 : 0;
    ProfScope ps("tc_decode_attn", st);
    auto kern = shard_rows ? tc_decode_kernel<true> : tc_decode_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e == cudaSuccess)
        kern<<<dim3((unsigned)(2 * units)), dim3(NTHREADS), SMEM_BYTES, st>>>(mC, mR, mP, mQa, mQp, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_decode_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_decode_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_decode_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

}  // namespace mla
