// tc_fused.cu -- explicit-form (LAGA per-rank) MLA prefill with the K_nope / V
// up-projection inside the attention kernel: no K/V workspace.
//
// Method ("A Training-Memory Regression in MLA Sequence Parallelism ... LAGA",
// arXiv 2607.17644, "What carries the argument" and Fig. 2): per head h,
// K_nope = chat W_K(h)^T and V = chat W_V(h)^T from the normalised latent, then
//   s_ij = scale * (q_nope_i . K_nope_j + RoPE(q_pe_i) . RoPE(k_pe_j)),
// softmax over the visible keys (j <= q_offset + i), output plus log-sum-exp.  The
// page names an up-projection fused into the attention kernel as the natural
// completion of LAGA ("Where Pith is reading between the lines"); this is that kernel.
//
// Sharing.  Rebuilding a 64-key tile of one head costs 2 x 64 x 512 x 256 FLOP, about
// 3.6 times one 128-query tile's attention over it, so every rebuilt tile is shared:
// a thread-block cluster of CL CTAs holds CL consecutive 128-query tiles of one head
// (and batch).  Key tile T is rebuilt by CTA T mod CL, written as fp16 into its own
// ring slot and bulk-copied through distributed shared memory into the same slot of
// every other CTA of the cluster; each CTA then attends its query tile over it.  Every
// slot barrier is armed (its expected bytes registered) before any byte can land on
// it: a CTA arms its slot for tile T once its own MMAs have released the slot's
// previous tile, then signals the tile's owner, which copies only after all CL CTAs
// have signalled.  The K/V never leave the chip.
//
// Per CTA (one query tile, 17 warps):
//   warp 0     slot producer: the unit's Q (TMA, staged in the reconstruction ring);
//              per key tile, once the slot is free here: arms the slot's barriers, loads
//              the rotated k_pe tile, tells the tile's owner the slot is ready.
//   warp 1     score MMAs S = Q K^T (M = 128, N = 64 keys, K = 192: 8 MMAs over the
//              K_nope^T tile as an MN-major operand, 4 over the k_pe tile), Q in TMEM.
//   warp 2     P.V MMAs O += P V (N = 144: the V^T tile + a row of ones gives the row
//              sums in O column 128), P read from TMEM where the softmax wrote it.
//   warp 3     reconstruction loader: latent and W_K / W_V chunks of 64 dims (TMA).
//   warp 16    reconstruction MMAs: K_nope^T = W_K chat^T and V^T = W_V chat^T
//              (M = 128, N = 64 keys, K = 512) into TMEM, for the CTA's own tiles.
//   warps 4-7  drain: thread = row of K_nope^T / V^T, TMEM -> fp16 -> own slot, then
//              bulk copies to the cluster's other CTAs.
//   warps 8-15 softmax, two threads per query row (32 keys each): online softmax in
//              the log2 domain, O rescaled only when a row maximum grows by > 2^8;
//              epilogue O / l and lse.
// Operand precision as the two-kernel tensor-core path: fp16 latent, weights, rotated
// bands, K_nope, V^T and P (11-bit significand), fp32 accumulation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_fused_err = 0;

namespace {

using namespace tc;

constexpr int BQ = 128, BKV = 64;
constexpr int NSLOT = 3;                    // K/V ring slots
constexpr int RST = 2;                      // reconstruction operand stages
constexpr uint32_t KT_BYTES = 128 * 128;    // K_nope^T: 128 d_nope rows x 64 keys, fp16
constexpr uint32_t KR_BYTES = 64 * 128;     // rotated k_pe: 64 keys x 64 dims, fp16
constexpr uint32_t K_SLOT = KT_BYTES + KR_BYTES;
constexpr uint32_t VT_BYTES = 128 * 128;    // V^T: 128 d_v rows x 64 keys, fp16
constexpr uint32_t ONES = 16 * 128;         // 16 constant rows after V^T: row 0 ones, the rest zeros
constexpr uint32_t V_SLOT = VT_BYTES + ONES;
constexpr uint32_t RC_BYTES = 64 * 128;     // latent chunk: 64 keys x 64 dims
constexpr uint32_t RW_BYTES = 128 * 128;    // weight chunk: 128 rows x 64 dims
constexpr uint32_t R_STAGE = RC_BYTES + 2 * RW_BYTES;
constexpr uint32_t QBOX = 128 * 128;        // a staged Q box: 128 rows x 128 bytes
constexpr uint32_t OFF_K = 0, OFF_V = OFF_K + NSLOT * K_SLOT, OFF_R = OFF_V + NSLOT * V_SLOT;
constexpr uint32_t OFF_BAR = OFF_R + RST * R_STAGE;
constexpr uint32_t OFF_RED = OFF_BAR + 512;
constexpr uint32_t SMEM_BYTES = OFF_RED + 2 * 2 * BQ * 4 + 1024;
static_assert(3 * QBOX <= RST * R_STAGE, "the Q staging fits in the reconstruction ring");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// TMEM columns: S buffers 0-63 and 64-127; O 128-271 (d_v 0-127, row sum 256, zeros);
// Q (192 fp16 = 96 columns) 272-367; reconstruction K_nope^T 384-447, V^T 448-511
constexpr uint32_t T_O = 128, T_L = T_O + 128, T_Q = 272, T_RK = 384, T_RV = 448;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int NWARPS = 17;

struct FusedK {
    int s_q, kv_need, q_offset, causal;
    int head_off;       // first query/output head of the call within q_nope / out
    int nh, nb, groups; // heads, batch, query-tile groups of CL tiles
    float scale_log2;
    __nv_bfloat16 *out;
    long out_b, out_i, out_h;
    int out_v8;
    float *lse;
    long lse_b, lse_h;
    uint32_t idesc_smn, idesc_sk, idesc_pv, idesc_r;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Key tiles (of BKV) that the 128-query tile starting at row q0 attends to.
__device__ __forceinline__ int tiles_of(const FusedK &p, int q0) {
    if (q0 >= p.s_q) return 0;
    const int kv_end = p.causal ? min(p.kv_need, p.q_offset + q0 + BQ) : p.kv_need;
    return (kv_end + BKV - 1) / BKV;
}

__device__ void settle() {   // let copies into this CTA land before it leaves after an abort
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 100000ull) {
    }
}

template <int CL>
__global__ void __launch_bounds__(32 * NWARPS, 1)
    tc_fused_kernel(const __grid_constant__ CUtensorMap mQn, const __grid_constant__ CUtensorMap mQr,
                    const __grid_constant__ CUtensorMap mKr, const __grid_constant__ CUtensorMap mC,
                    const __grid_constant__ CUtensorMap mW, FusedK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + OFF_BAR);
    // slot barriers (same offsets in every CTA: peers complete k_full / v_full with their
    // copies and arrive on armed).  k_full / v_full: two arrivals (this CTA's slot producer
    // twice, or once plus the drain for a tile this CTA rebuilds) and the bytes;
    // k_free / v_free: this CTA's MMAs have read the slot; armed: every CTA of the cluster
    // has armed its slot for the next tile this CTA rebuilds into it.
    uint64_t *k_full = bars, *k_free = bars + 3, *v_full = bars + 6, *v_free = bars + 9, *armed = bars + 29;
    uint64_t *s_full = bars + 12, *p_full = bars + 14, *pv_done = bars + 16;
    uint64_t *o_done = bars + 18, *o_final = bars + 19, *qs_full = bars + 20, *q_ready = bars + 21;
    uint64_t *r_full = bars + 22, *r_empty = bars + 24, *racc_full = bars + 26, *racc_free = bars + 27;
    uint64_t *drained = bars + 28;   // the four drain warps have written a rebuilt tile
    uint32_t *tslot = (uint32_t *)(bars + 32);
    volatile int *abort = (volatile int *)(tslot + 1);
    float (*red)[2][BQ] = (float (*)[2][BQ])(smem + OFF_RED);   // [tile parity][half][row] maxima
    unsigned *err = &g_tc_fused_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank();
    // cluster -> (query-tile group, heaviest first; head; batch)
    const int cl = blockIdx.x / CL;
    const int nhb = p.nh * p.nb;
    const int grp = p.groups - 1 - cl / nhb;
    const int hl = (cl % nhb) % p.nh, b = (cl % nhb) / p.nh;
    const int hq = p.head_off + hl;
    const int q0 = (grp * CL + rank) * BQ;
    const int nt = tiles_of(p, q0);                 // tiles this CTA attends
    int nt_max = 0;                                 // tiles the cluster walks (same in every CTA)
#pragma unroll
    for (int r = 0; r < CL; ++r) nt_max = max(nt_max, tiles_of(p, (grp * CL + r) * BQ));

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&k_full[s], 2);
            mbar_init(&k_free[s], 1);
            mbar_init(&v_full[s], 2);
            mbar_init(&v_free[s], 1);
            mbar_init(&armed[s], CL);   // one arrival per CTA of the cluster
        }
        mbar_init(drained, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 8);
            mbar_init(&pv_done[i], 1);
            mbar_init(&r_full[i], 1);
            mbar_init(&r_empty[i], 1);
        }
        mbar_init(o_done, 1);
        mbar_init(o_final, 1);
        mbar_init(qs_full, 1);
        mbar_init(q_ready, 8);
        mbar_init(racc_full, 1);
        mbar_init(racc_free, 4);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    // the constant rows after every V^T tile: row 0 fp16 ones, rows 1-15 zeros (a constant
    // row is unchanged by the 128-byte swizzle)
    for (int i = tid; i < NSLOT * (int)(ONES / 16); i += blockDim.x) {
        const int s = i / (ONES / 16), off = i % (ONES / 16);
        const uint32_t v = off < 8 ? 0x3c003c00u : 0u;
        *(uint4 *)(smem + OFF_V + s * V_SLOT + VT_BYTES + off * 16) = make_uint4(v, v, v, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // every CTA's barriers exist before any cross-CTA arrival
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------ slot producer
        if (lane == 0) {
            tma_prefetch_desc(&mQn);
            tma_prefetch_desc(&mQr);
            tma_prefetch_desc(&mKr);
            uint8_t *qs = smem + OFF_R;   // Q staged where the reconstruction ring will run
            mbar_arrive_expect_tx(qs_full, 3 * QBOX);
            tma_load_4d(qs, &mQn, qs_full, 0, hq, q0, b);
            tma_load_4d(qs + QBOX, &mQn, qs_full, 64, hq, q0, b);
            tma_load_4d(qs + 2 * QBOX, &mQr, qs_full, 0, hq, q0, b);
            bool ok = true;
            for (int T = 0; T < nt_max && ok; ++T) {
                const int s = T % NSLOT, n = T / NSLOT;
                const bool own = (T % CL) == rank;
                // this CTA's MMAs have read tile T - NSLOT out of slot s
                if (T >= NSLOT)
                    ok = mbar_wait(&k_free[s], (n - 1) & 1, abort, err) && mbar_wait(&v_free[s], (n - 1) & 1, abort, err);
                if (!ok) break;
                // arm slot s for tile T before anything can land in it
                if (own) {   // the drain supplies K_nope^T and V^T and the second arrivals
                    mbar_arrive_expect_tx(&k_full[s], KR_BYTES);
                    mbar_arrive(&v_full[s]);
                } else {     // the owner's copies supply K_nope^T and V^T
                    mbar_arrive_expect_tx(&k_full[s], KR_BYTES + KT_BYTES);
                    mbar_arrive(&k_full[s]);
                    mbar_arrive_expect_tx(&v_full[s], VT_BYTES);
                    mbar_arrive(&v_full[s]);
                }
                tma_load_3d(smem + OFF_K + s * K_SLOT + KT_BYTES, &mKr, &k_full[s], 0, T * BKV, b);
                // tell the tile's owner (possibly this CTA) that slot s is ready for it
                mbar_arrive_peer(map_peer(smem_u32(&armed[s]), (uint32_t)(T % CL)));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ score MMAs
        bool ok = __all_sync(0xffffffffu, mbar_wait(q_ready, 0, abort, err));
        for (int T = 0; T < nt_max && ok; ++T) {
            const int s = T % NSLOT;
            ok = __all_sync(0xffffffffu, mbar_wait(&k_full[s], (T / NSLOT) & 1, abort, err));
            // S buffer T & 1 last held P_{T-2}: its P.V must be done
            if (ok && T < nt && T >= 2)
                ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[T & 1], ((T - 2) >> 1) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                if (T < nt) {
                    const uint32_t d = tmem + (T & 1) * BKV;
                    const uint8_t *ks = smem + OFF_K + s * K_SLOT;
                    const uint64_t dkt = sdesc_mnmajor(ks, KT_BYTES);   // keys along N, d_nope along K
                    const uint64_t dkr = sdesc_kmajor(ks + KT_BYTES);
#pragma unroll
                    for (int k = 0; k < 8; ++k)   // 16 d_nope rows = 2048 bytes per step
                        mma_ts(d, tmem + T_Q + k * 8, dkt + (uint64_t)(k * (2048 >> 4)), p.idesc_smn, k != 0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ts(d, tmem + T_Q + 64 + k * 8, dkr + 2 * k, p.idesc_sk, 1);
                    mma_commit(&s_full[T & 1]);
                }
                mma_commit(&k_free[s]);   // this CTA is done with slot s's K part
            }
            __syncwarp();
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ P.V MMAs
        bool ok = true;
        for (int T = 0; T < nt_max && ok; ++T) {
            const int s = T % NSLOT;
            if (T < nt) ok = __all_sync(0xffffffffu, mbar_wait(&p_full[T & 1], (T >> 1) & 1, abort, err));
            ok = ok && __all_sync(0xffffffffu, mbar_wait(&v_full[s], (T / NSLOT) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                if (T < nt) {
                    const uint32_t pa = tmem + (T & 1) * BKV;
                    const uint64_t dv = sdesc_kmajor(smem + OFF_V + s * V_SLOT);   // 144 rows: V^T + constants
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ts(tmem + T_O, pa + k * 8, dv + 2 * k, p.idesc_pv, (T | k) != 0);
                }
                mma_commit(&v_free[s]);
                if (T < nt) {
                    mma_commit(&pv_done[T & 1]);
                    mma_commit(o_done);
                    if (T == nt - 1) mma_commit(o_final);
                }
            }
            __syncwarp();
        }
    } else if (warp == 3) {
        // ------------------------------------------------ reconstruction loader
        if (lane == 0) {
            tma_prefetch_desc(&mC);
            tma_prefetch_desc(&mW);
            // the Q staging in this ring has been moved into TMEM
            bool ok = mbar_wait(q_ready, 0, abort, err);
            int it = 0;
            for (int T = rank; T < nt_max && ok; T += CL) {
                for (int kc = 0; kc < 8; ++kc, ++it) {
                    const int st = it % RST;
                    if (it >= RST && !mbar_wait(&r_empty[st], ((it / RST) - 1) & 1, abort, err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *rs = smem + OFF_R + st * R_STAGE;
                    mbar_arrive_expect_tx(&r_full[st], R_STAGE);
                    tma_load_3d(rs, &mC, &r_full[st], kc * 64, T * BKV, b);
                    tma_load_3d(rs + RC_BYTES, &mW, &r_full[st], kc * 64, 0, hq);
                    tma_load_3d(rs + RC_BYTES + RW_BYTES, &mW, &r_full[st], kc * 64, 128, hq);
                }
            }
        }
    } else if (warp == 16) {
        // ------------------------------------------------ reconstruction MMAs
        bool ok = true;
        int it = 0, k = 0;
        for (int T = rank; T < nt_max && ok; T += CL, ++k) {
            // the drain has read the previous tile out of the accumulators
            if (k > 0) ok = __all_sync(0xffffffffu, mbar_wait(racc_free, (k - 1) & 1, abort, err));
            for (int kc = 0; kc < 8 && ok; ++kc, ++it) {
                const int st = it % RST;
                ok = __all_sync(0xffffffffu, mbar_wait(&r_full[st], (it / RST) & 1, abort, err));
                if (!ok) break;
                tc_fence_after();
                const uint8_t *rs = smem + OFF_R + st * R_STAGE;
                const uint64_t dc = sdesc_kmajor(rs);
                const uint64_t dwk = sdesc_kmajor(rs + RC_BYTES), dwv = sdesc_kmajor(rs + RC_BYTES + RW_BYTES);
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        mma_ss(tmem + T_RK, dwk + 2 * j, dc + 2 * j, p.idesc_r, (kc | j) != 0);
                        mma_ss(tmem + T_RV, dwv + 2 * j, dc + 2 * j, p.idesc_r, (kc | j) != 0);
                    }
                    mma_commit(&r_empty[st]);
                    if (kc == 7) mma_commit(racc_full);
                }
                __syncwarp();
            }
        }
    } else if (warp >= 4 && warp <= 7) {
        // ------------------------------------------------------------ drain
        const int quad = warp & 3, row = quad * 32 + lane;   // d_nope / d_v row
        const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        int k = 0;
        int uses[NSLOT] = {0, 0, 0};   // this CTA's rebuilt tiles so far per slot (armed phases)
        for (int T = rank; T < nt_max && ok; T += CL, ++k) {
            const int s = T % NSLOT;
            ok = __all_sync(0xffffffffu, mbar_wait(racc_full, k & 1, abort, err));
            // slot s is free and armed in every CTA of the cluster (this one included)
            ok = ok && __all_sync(0xffffffffu, mbar_wait_cluster(&armed[s], uses[s] & 1, abort, err));
            ++uses[s];
            if (!ok) break;
            tc_fence_after();
            // K_nope^T then V^T, 32 keys at a time: keys 8c .. 8c+7 -> 16-byte chunk c of
            // the row, stored at chunk c ^ (row & 7) (128-byte swizzle)
#pragma unroll 1
            for (int part = 0; part < 4; ++part) {
                uint32_t a[32];
                tmem_ld32(lb + (part < 2 ? T_RK : T_RV) + 32 * (part & 1), a);
                tmem_ld_wait();
                if (part == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(racc_free);   // the next own tile may accumulate
                }
                uint8_t *dst = part < 2 ? smem + OFF_K + s * K_SLOT + row * 128 : smem + OFF_V + s * V_SLOT + row * 128;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = 4 * (part & 1) + cc;
                    *(uint4 *)(dst + ((c ^ (row & 7)) << 4)) =
                        make_uint4(pack_f16(__uint_as_float(a[8 * cc]), __uint_as_float(a[8 * cc + 1])),
                                   pack_f16(__uint_as_float(a[8 * cc + 2]), __uint_as_float(a[8 * cc + 3])),
                                   pack_f16(__uint_as_float(a[8 * cc + 4]), __uint_as_float(a[8 * cc + 5])),
                                   pack_f16(__uint_as_float(a[8 * cc + 6]), __uint_as_float(a[8 * cc + 7])));
                }
            }
            fence_proxy_async_smem();   // the tensor core and the bulk copies read these rows
            __syncwarp();
            if (lane == 0) mbar_arrive(drained);
            if (warp == 4) {
                // all four warps' rows are written: copy the tile into the other CTAs' slot
                // s and complete this CTA's own slot
                ok = __all_sync(0xffffffffu, mbar_wait(drained, k & 1, abort, err));
                if (ok && lane == 0) {
                    uint8_t *kts = smem + OFF_K + s * K_SLOT, *vts = smem + OFF_V + s * V_SLOT;
#pragma unroll 1
                    for (int r = 0; r < CL; ++r) {
                        if (r == rank) continue;
                        bulk_copy_to_peer(map_peer(smem_u32(kts), r), kts, KT_BYTES,
                                          map_peer(smem_u32(&k_full[s]), r));
                        bulk_copy_to_peer(map_peer(smem_u32(vts), r), vts, VT_BYTES,
                                          map_peer(smem_u32(&v_full[s]), r));
                    }
                    bulk_commit();
                    mbar_arrive(&k_full[s]);
                    mbar_arrive(&v_full[s]);
                    bulk_wait_read<0>();   // the slot is not rewritten before its copies have read it
                }
                __syncwarp();
            }
        }
        if (warp == 4 && lane == 0) bulk_wait_all();   // every copy into the peers has landed
    } else {
        // ------------------------------------------------------------ softmax (warps 8-15)
        const int quad = warp & 3, h = (warp - 8) >> 2;   // half h: keys [32h, 32h + 32) of a tile
        const int row = quad * 32 + lane;
        const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        // ---- Q from the staging into TMEM: half h widens q_nope dims [64h, 64h + 64) to fp16
        // (columns 32h ...) and copies the rotated q_pe dims [32h, 32h + 32) (columns 64 + 16h
        // ...); chunk c of row r of a staged box sits at chunk c ^ (r & 7)
        {
            ok = __all_sync(0xffffffffu, mbar_wait(qs_full, 0, abort, err));
            const uint8_t *qs = smem + OFF_R;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t qn[16];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = 4 * part + cc;
                    const uint4 v = *(const uint4 *)(qs + h * QBOX + row * 128 + ((c ^ (row & 7)) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        qn[4 * cc + i] = pack_f16(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xffff0000u));
                }
                tmem_st16(lb + T_Q + 32 * h + 16 * part, qn);
            }
            uint32_t qp[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = *(const uint4 *)(qs + 2 * QBOX + row * 128 + (((4 * h + c) ^ (row & 7)) << 4));
                qp[4 * c] = v.x, qp[4 * c + 1] = v.y, qp[4 * c + 2] = v.z, qp[4 * c + 3] = v.w;
            }
            tmem_st16(lb + T_Q + 64 + 16 * h, qp);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        const int pos = p.q_offset + q0 + row;
        float m = -INFINITY;
        for (int T = 0; T < nt; ++T) {
            const int sb = T & 1;
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&s_full[sb], (T >> 1) & 1, abort, err));
            tc_fence_after();
            uint32_t sr[32];
            if (ok) {
                tmem_ld32(lb + sb * BKV + h * 32, sr);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) sr[i] = 0u;
            }
            const int j0 = T * BKV + h * 32;
            const bool masked = (j0 + 32 > p.kv_need) || (p.causal && j0 + 31 > p.q_offset + q0);
            float x[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(sr[c]);
            if (masked) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int key = j0 + c;
                    if (key >= p.kv_need || (p.causal && key > pos)) x[c] = -INFINITY;
                }
            }
            float mx[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) mx[a] = x[a];
#pragma unroll
            for (int c = 4; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], x[c]);
            red[sb][h][row] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            // both halves have read their S columns before either writes P over them
            named_bar_sync(1, 256);
            const float mt = fmaxf(red[sb][0][row], red[sb][1][row]) * p.scale_log2;
            const float m_new = fmaxf(m, mt);
            const bool need = m_new > m + RESCALE_LOG2;   // also true on the first finite maximum
            if (__any_sync(0xffffffffu, need)) {
                const float m_use = need ? m_new : m;
                const float alpha = (m == -INFINITY) ? 0.f : ex2(m - m_use);
                // before its first P.V, O holds nothing of this unit (accumulate off)
                if (T > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, (T - 1) & 1, abort, err));
                if (T > 0 && ok) {
                    tc_fence_after();
                    // (rare: a row maximum grew by more than 2^8) eight columns at a time, so
                    // that the live scores keep their registers
#pragma unroll 1
                    for (int part = 0; part < 8; ++part) {
                        uint32_t o[8];
                        tmem_ld8(lb + T_O + 64 * h + 8 * part, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st8(lb + T_O + 64 * h + 8 * part, o);
                    }
                    if (h == 0) {   // the row sum is rescaled with the row (warp-uniform)
                        const uint32_t lv = tmem_ld1(lb + T_L);
                        tmem_ld_wait();
                        tmem_st1(lb + T_L, __float_as_uint(__uint_as_float(lv) * alpha));
                    }
                    tmem_st_wait();
                }
                m = m_use;
            }
            const float nm = (m == -INFINITY) ? 0.f : -m;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack_f16(ex2(fmaf(x[2 * i], p.scale_log2, nm)), ex2(fmaf(x[2 * i + 1], p.scale_log2, nm)));
            if (ok) {
                tmem_st16(lb + sb * BKV + h * 16, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        // ---- epilogue: the row sum is O's column 128; each half stores 64 columns
        if (nt > 0) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(o_final, 0, abort, err));
            tc_fence_after();
            const int qi = q0 + row;
            float l = 0.f;
            if (ok) {
                const uint32_t lv = tmem_ld1(lb + T_L);
                tmem_ld_wait();
                l = __uint_as_float(lv);
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool store = ok && qi < p.s_q;
            uint32_t *dst = (uint32_t *)(p.out + b * p.out_b + (long)qi * p.out_i + (long)hq * p.out_h + h * 64);
            // 32 columns at a time; the TMEM loads are warp-wide (.sync.aligned), so every
            // lane takes them, and only the rows inside the call store
#pragma unroll 1
            for (int part = 0; part < 2 && ok; ++part) {
                uint32_t o[32], wv[16];
                tmem_ld32(lb + T_O + 64 * h + 32 * part, o);
                tmem_ld_wait();
                if (store) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        wv[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                    uint32_t *d2 = dst + 16 * part;
                    if (p.out_v8) {
                        st_global_v8(d2, wv);
                        st_global_v8(d2 + 8, wv + 8);
                    } else {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            ((uint4 *)d2)[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                    }
                }
            }
            if (store) {
                if (h == 0)
                    p.lse[b * p.lse_b + (long)hq * p.lse_h + qi] =
                        l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
    if (tid == 0 && *abort) settle();
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // peers may address this CTA's slots and barriers until here
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int CL>
cudaError_t launch_fused(const CUtensorMap *maps, const FusedK &a, int n_clusters, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(tc_fused_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_clusters * CL));
    cfg.blockDim = dim3(32 * NWARPS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_fused_kernel<CL>, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

}  // namespace

cudaError_t tc_fused_prefill(const TcPrefill &p, const void *q_nope, void *out, float *lse, const void *chat,
                             const void *kpe, const void *qpe, const void *w16, int cluster, cudaStream_t st) {
    if (cluster != 4 && cluster != 8) return cudaErrorInvalidValue;
    const long kv_pad = (p.kv_need + 127) / 128 * 128;
    cudaError_t e;
    CUtensorMap maps[5];   // q_nope, rotated q_pe, rotated k_pe, latent, fp16 weights
    {
        unsigned long long d[4] = {(unsigned long long)p.Dn, (unsigned long long)p.head_count,
                                   (unsigned long long)p.s_q, (unsigned long long)p.B};
        unsigned long long s[3] = {(unsigned long long)p.Dn * 2, (unsigned long long)p.head_count * p.Dn * 2,
                                   (unsigned long long)p.s_q * p.head_count * p.Dn * 2};
        unsigned box[4] = {64, 1, 128, 1};
        if ((e = make_tma_map(&maps[0], q_nope, 4, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[4] = {(unsigned long long)p.Dr, (unsigned long long)p.head_count,
                                   (unsigned long long)p.s_q, (unsigned long long)p.B};
        unsigned long long s[3] = {(unsigned long long)p.Dr * 2, (unsigned long long)p.head_count * p.Dr * 2,
                                   (unsigned long long)p.s_q * p.head_count * p.Dr * 2};
        unsigned box[4] = {64, 1, 128, 1};
        if ((e = make_tma_map(&maps[1], qpe, 4, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {(unsigned long long)p.Dr, (unsigned long long)kv_pad, (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)p.Dr * 2, (unsigned long long)kv_pad * p.Dr * 2};
        unsigned box[3] = {64, (unsigned)BKV, 1};
        if ((e = make_tma_map(&maps[2], kpe, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {(unsigned long long)p.Dk, (unsigned long long)kv_pad, (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)p.Dk * 2, (unsigned long long)kv_pad * p.Dk * 2};
        unsigned box[3] = {64, (unsigned)BKV, 1};
        if ((e = make_tma_map(&maps[3], chat, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        const long Dh = p.Dn + p.Dv;
        unsigned long long d[3] = {(unsigned long long)p.Dk, (unsigned long long)Dh,
                                   (unsigned long long)p.head_count};
        unsigned long long s[2] = {(unsigned long long)p.Dk * 2, (unsigned long long)Dh * p.Dk * 2};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&maps[4], w16, 3, d, s, box)) != cudaSuccess) return e;
    }
    FusedK a{};
    a.s_q = p.s_q;
    a.kv_need = (int)p.kv_need;
    a.q_offset = p.q_offset;
    a.causal = p.causal;
    a.head_off = 0;
    a.nh = p.head_count;
    a.nb = p.B;
    const int n_qt = (p.s_q + BQ - 1) / BQ;
    a.groups = (n_qt + cluster - 1) / cluster;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.out = (__nv_bfloat16 *)out;
    a.out_b = (long)p.s_q * p.head_count * p.Dv;
    a.out_i = (long)p.head_count * p.Dv;
    a.out_h = p.Dv;
    a.out_v8 = ((uintptr_t)out % 32) == 0;
    a.lse = lse;
    a.lse_b = (long)p.head_count * p.s_q;
    a.lse_h = p.s_q;
    a.idesc_smn = idesc_f16(128, BKV, true, true);   // B = K_nope^T, keys contiguous (MN-major)
    a.idesc_sk = idesc_f16(128, BKV, true);          // B = k_pe, K-major
    a.idesc_pv = idesc_f16(128, 144, true);          // 128 d_v columns + the row-sum block
    a.idesc_r = idesc_f16(128, BKV, true);           // A = weight rows, B = latent rows, both K-major
    const int n_clusters = a.groups * p.head_count * p.B;
    if (n_clusters == 0) return cudaSuccess;
    ProfScope ps("tc_fused_attn", st);
    e = cluster == 8 ? launch_fused<8>(maps, a, n_clusters, st) : launch_fused<4>(maps, a, n_clusters, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t tc_fused_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_fused_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_fused_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

}  // namespace mla
