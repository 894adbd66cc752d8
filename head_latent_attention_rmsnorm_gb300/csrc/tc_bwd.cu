// tc_bwd.cu -- the explicit prefill's backward pass on the sm_103a tensor cores (bf16
// calls at d_nope = d_v = 128, d_rope = 64, d_kv = 512).
//
// Method ("A Training-Memory Regression in MLA Sequence Parallelism ... LAGA", arXiv
// 2607.17644, "What carries the argument": the sequence-parallel method gives the same
// gradients as the baseline).  The chain rule through the forward's steps for an
// upstream gradient dO (the log-sum-exp is not differentiated):
//   P = exp(S - lse),  dP = dO V^T,  dS = P (dP - D) scale,  D_i = dO_i . o_i
//   dQ = dS K (the rotated band's part rotated back later),  dK = dS^T Q,  dV = P^T dO
// Two kernels, both recomputing S from the forward's K_nope / V^T reconstruction:
//  * tc_bwd_dkv_kernel: one CTA per (128-key tile, head); walks the 64-query tiles that
//    see its keys.  S^T = K Q^T and dP^T = V dO^T (keys on TMEM lanes), the softmax
//    warps form P^T and dS^T in place as fp16, then dV += P^T dO and dK += dS^T Q
//    (dK 192 wide: d_nope plus the rotated band, whose per-head sums are added over the
//    heads afterwards).  Output: [dK_nope^T ; dV^T] per head (fp16, key-contiguous, the
//    operand layout of the weight-gradient GEMM) and the band's dk_rot per head (fp32).
//  * tc_bwd_dq_kernel: one CTA per (128-query tile, head); walks its visible 128-key
//    tiles.  S = Q K^T and dP = dO V^T (queries on TMEM lanes), dS in place as fp16, then
//    dQ += dS K with K read as an MN-major operand.  Output: dq_nope (bf16) and the
//    rotated band's dq (fp32).
// Operands are fp16 (Q, dO and the reconstruction converted by the prep launch), P and dS
// are fp16, accumulation is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_bwd_err = 0;

namespace {

using namespace tc;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ void settle() {   // let copies into this CTA land before it leaves after an abort
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 100000ull) {
    }
}

// ------------------------------------------------------------------------ prep ----
// Row (b, i, h): q_nope and dO widened to fp16 copies, D = dO . out.  Warp per row,
// 128-wide rows, 8-byte pieces.
__global__ void bwd_prep_tc_kernel(long rows, int hc, int s_q, const __nv_bfloat16 *q_nope,
                                   const __nv_bfloat16 *dout, const __nv_bfloat16 *out, __half *qn16, __half *do16,
                                   float *D) {
    const long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    const long o = r * 128 + lane * 4;
    const uint2 qv = *(const uint2 *)(q_nope + o), dv = *(const uint2 *)(dout + o), ov = *(const uint2 *)(out + o);
    const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qv.x));
    const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qv.y));
    const float2 d0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&dv.x));
    const float2 d1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&dv.y));
    const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ov.x));
    const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ov.y));
    *(uint2 *)(qn16 + o) = make_uint2(pack_f16(q0.x, q0.y), pack_f16(q1.x, q1.y));
    *(uint2 *)(do16 + o) = make_uint2(pack_f16(d0.x, d0.y), pack_f16(d1.x, d1.y));
    float a = fmaf(d0.x, o0.x, fmaf(d0.y, o0.y, fmaf(d1.x, o1.x, d1.y * o1.y)));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) a += __shfl_xor_sync(0xffffffffu, a, s);
    const long h = r % hc, bi = r / hc, i = bi % s_q, b = bi / s_q;
    if (lane == 0) D[(b * hc + h) * s_q + i] = a;
}

// y[c][r] = x[r][c] for 16-bit matrices, 32 x 32 tiles through shared memory.
__global__ void transpose16_kernel(long R, long C, const uint16_t *x, uint16_t *y) {
    __shared__ uint16_t t[32][33];
    const long r0 = (long)blockIdx.y * 32, c0 = (long)blockIdx.x * 32;
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    for (int k = ty; k < 32; k += blockDim.x / 32)
        if (r0 + k < R && c0 + tx < C) t[k][tx] = x[(r0 + k) * C + c0 + tx];
    __syncthreads();
    for (int k = ty; k < 32; k += blockDim.x / 32)
        if (c0 + k < C && r0 + tx < R) y[(c0 + k) * R + r0 + tx] = t[tx][k];
}

// The same transpose with 16-byte global accesses (R and C multiples of 8, rows 16-byte
// aligned): 64 x 64 tiles; a row pitch of 65 elements in shared memory keeps the column
// gathers of eight consecutive rows on distinct banks.
__global__ void __launch_bounds__(256) transpose16_vec_kernel(long R, long C, const uint4 *x, uint4 *y) {
    __shared__ uint16_t t[64][65];
    const long r0 = (long)blockIdx.y * 64, c0 = (long)blockIdx.x * 64;
    const int ch = threadIdx.x % 8, rr = threadIdx.x / 8;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = rr + 32 * i;
        if (r0 + row < R && c0 + ch * 8 < C) {
            const uint4 v = x[((r0 + row) * C + c0) / 8 + ch];
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                t[row][ch * 8 + 2 * e] = (uint16_t)(u[e] & 0xffffu);
                t[row][ch * 8 + 2 * e + 1] = (uint16_t)(u[e] >> 16);
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int orow = rr + 32 * i;   // output row = input column c0 + orow
        if (c0 + orow < C && r0 + ch * 8 < R) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                u[e] = (uint32_t)t[ch * 8 + 2 * e][orow] | ((uint32_t)t[ch * 8 + 2 * e + 1][orow] << 16);
            y[((c0 + orow) * R + r0) / 8 + ch] = make_uint4(u[0], u[1], u[2], u[3]);
        }
    }
}

// ------------------------------------------------------------ key-stationary ----
constexpr uint32_t KBOX = 128 * 128;   // 128 rows x 64 fp16
constexpr uint32_t QBOX64 = 64 * 128;  // 64 rows x 64 fp16
constexpr uint32_t B_OFF_K = 0, B_OFF_V = 3 * KBOX, B_OFF_Q = B_OFF_V + 2 * KBOX;
constexpr uint32_t B_STAGE = 5 * QBOX64;   // Q (q_nope lo, hi, rotated q_pe) + dO (lo, hi)
constexpr int B_QST = 3;                     // Q / dO stages: a tile's loads start two tiles ahead of its use
constexpr uint32_t B_OFF_LD = B_OFF_Q + B_QST * B_STAGE;   // [2][2][64] lse (log2 domain) and D of a q tile
constexpr uint32_t B_OFF_BAR = B_OFF_LD + 2 * 2 * 64 * 4;
constexpr uint32_t B_SMEM = B_OFF_BAR + 256 + 1024;
// TMEM: S^T double-buffered 0-63 and 64-127 (P^T then goes in its first 32 columns as fp16
// and dS^T in the other 32), dP^T 128-191, dV 192-319, dK (d_nope 128 + band 64) 320-511.
// With dS^T beside P^T, the dP^T columns are free as soon as the softmax has read them,
// so the next tile's dP^T overlaps this tile's softmax instead of waiting for its dK.
constexpr uint32_t B_ST = 0, B_DPT = 128, B_DV = 192, B_DK = 320;

struct DkvK {
    int s_q, kv_need, q_offset, causal, hc, h0, nh, n_kt;
    float scale, scale_log2;
    const float *lse, *D;           // [B][hc][s_q]
    __half *dkvt;                   // [nh][256][B][kv_pad]
    long kv_pad;
    int B;
    float *dkr;                     // [B][nh][kv_pad][64]
    uint32_t idesc_st, idesc_dpt, idesc_dv, idesc_dk;
};

__global__ void __launch_bounds__(384, 1)
    tc_bwd_dkv_kernel(const __grid_constant__ CUtensorMap mKn, const __grid_constant__ CUtensorMap mKr,
                      const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mQn,
                      const __grid_constant__ CUtensorMap mQr, const __grid_constant__ CUtensorMap mDo, DkvK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + B_OFF_BAR);
    // st_full / pt_free [buffer]: S^T landed / P^T and dS^T read by the dV and dK MMAs;
    // dpt_full / dpt_free: dP^T landed / read by the softmax warps; ps_full: the softmax
    // warps wrote P^T and dS^T
    uint64_t *kv_full = bars, *qd_full = bars + 1, *qd_empty = bars + 1 + B_QST, *st_full = bars + 1 + 2 * B_QST;
    uint64_t *dpt_full = st_full + 2, *ps_full = dpt_full + 1, *pt_free = ps_full + 1, *dpt_free = pt_free + 2;
    uint64_t *acc_done = dpt_free + 1;
    uint32_t *tslot = (uint32_t *)(acc_done + 2);
    volatile int *abort = (volatile int *)(tslot + 1);
    float *ld = (float *)(smem + B_OFF_LD);
    unsigned *err = &g_tc_bwd_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (key tile, head, batch), key tiles fastest
    const int kt = blockIdx.x % p.n_kt, hb = blockIdx.x / p.n_kt;
    const int hl = hb % p.nh, b = hb / p.nh, hq = p.h0 + hl;
    const int k0 = kt * 128;
    const int n_qt = (p.s_q + 63) / 64;
    int qt0 = 0;
    if (p.causal) qt0 = max(0, k0 - p.q_offset) / 64;
    if (k0 >= p.kv_need) qt0 = n_qt;   // keys past kv_need: seen by nobody
    const int nqt = max(0, n_qt - qt0);

    if (tid == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < B_QST; ++i) {
            mbar_init(&qd_full[i], 1);
            mbar_init(&qd_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&pt_free[i], 1);
        }
        mbar_init(dpt_full, 1);
        mbar_init(dpt_free, 1);
        mbar_init(ps_full, 8);
        mbar_init(acc_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && nqt > 0) {
            mbar_arrive_expect_tx(kv_full, 5 * KBOX);
            tma_load_3d(smem + B_OFF_K, &mKn, kv_full, hl * 128, k0, b);
            tma_load_3d(smem + B_OFF_K + KBOX, &mKn, kv_full, hl * 128 + 64, k0, b);
            tma_load_3d(smem + B_OFF_K + 2 * KBOX, &mKr, kv_full, 0, k0, b);
            tma_load_3d(smem + B_OFF_V, &mV, kv_full, k0, hl * 128, b);
            tma_load_3d(smem + B_OFF_V + KBOX, &mV, kv_full, k0 + 64, hl * 128, b);
            for (int t = 0; t < nqt; ++t) {
                const int qs = t % B_QST;
                if (t >= B_QST && !mbar_wait(&qd_empty[qs], ((t / B_QST) - 1) & 1, abort, err)) break;
                uint8_t *q = smem + B_OFF_Q + qs * B_STAGE;
                const int q0 = (qt0 + t) * 64;
                mbar_arrive_expect_tx(&qd_full[qs], B_STAGE);
                tma_load_4d(q, &mQn, &qd_full[qs], 0, hq, q0, b);
                tma_load_4d(q + QBOX64, &mQn, &qd_full[qs], 64, hq, q0, b);
                tma_load_4d(q + 2 * QBOX64, &mQr, &qd_full[qs], 0, hq, q0, b);
                tma_load_4d(q + 3 * QBOX64, &mDo, &qd_full[qs], 0, hq, q0, b);
                tma_load_4d(q + 4 * QBOX64, &mDo, &qd_full[qs], 64, hq, q0, b);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ S^T = K Q^T, dP^T = V dO^T
        // S^T of tile t + 1 goes into the other buffer as soon as dP^T of tile t is issued,
        // so it overlaps the softmax of tile t
        bool ok = nqt > 0 && __all_sync(0xffffffffu, mbar_wait(kv_full, 0, abort, err));
        for (int t = 0; t < nqt && ok; ++t) {
            const int st = t & 1;
            const int qs = t % B_QST;
            ok = __all_sync(0xffffffffu, mbar_wait(&qd_full[qs], (t / B_QST) & 1, abort, err));
            // the dV MMAs of tile t - 2 have read P^T out of this buffer
            if (ok && t >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&pt_free[st], ((t - 2) >> 1) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            const uint8_t *q = smem + B_OFF_Q + (t % B_QST) * B_STAGE;
            if (elect_one()) {
#pragma unroll
                for (int kb = 0; kb < 3; ++kb) {
                    const uint64_t da = sdesc_kmajor(smem + B_OFF_K + kb * KBOX), db = sdesc_kmajor(q + kb * QBOX64);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_ss(tmem + B_ST + st * 64, da + 2 * k4, db + 2 * k4, p.idesc_st, (kb | k4) != 0);
                }
                mma_commit(&st_full[st]);
            }
            __syncwarp();
            // the softmax warps have read dP^T of tile t - 1
            if (t >= 1) ok = __all_sync(0xffffffffu, mbar_wait(dpt_free, (t - 1) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                // A = V (keys x d_v) read from V^T as an MN-major operand: two 64-key blocks
                const uint64_t dv = sdesc_mnmajor(smem + B_OFF_V, KBOX);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ss(tmem + B_DPT, dv + (uint64_t)(k * (2048 >> 4)), sdesc_kmajor(q + (3 + (k >> 2)) * QBOX64) + 2 * (k & 3),
                           p.idesc_dpt, k != 0);
                mma_commit(dpt_full);
            }
            __syncwarp();
        }
    } else if (warp == 2) {
        // --------------------------------------------- dV += P^T dO, dK += dS^T Q
        bool ok = true;
        for (int t = 0; t < nqt && ok; ++t) {
            const int st = t & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(ps_full, t & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            const uint8_t *q = smem + B_OFF_Q + (t % B_QST) * B_STAGE;
            if (elect_one()) {
                const uint64_t bdo = sdesc_mnmajor(q + 3 * QBOX64, QBOX64);   // dO^T: two 64-dim blocks
                const uint64_t bq = sdesc_mnmajor(q, QBOX64);                 // Q^T: three 64-dim blocks
#pragma unroll
                for (int k = 0; k < 4; ++k)   // 16 queries per step
                    mma_ts(tmem + B_DV, tmem + B_ST + st * 64 + k * 8, bdo + (uint64_t)(k * (2048 >> 4)), p.idesc_dv,
                           (t | k) != 0);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ts(tmem + B_DK, tmem + B_ST + st * 64 + 32 + k * 8, bq + (uint64_t)(k * (2048 >> 4)), p.idesc_dk,
                           (t | k) != 0);
                mma_commit(&pt_free[st]);
                mma_commit(&qd_empty[t % B_QST]);
                if (t == nqt - 1) mma_commit(acc_done);
            }
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ---------------------------------------- P^T and dS^T (warps 4-11), epilogue
        // thread = key row (TMEM lane), half h = queries [32h, 32h + 32) of a 64-query tile
        const int quad = warp & 3, h = (warp - 4) >> 2, row = quad * 32 + lane;
        const int j = k0 + row;
        const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        // lse (scaled to log2) and D of query tile tt's queries: half 0's thread `row` holds
        // the value of query row & 63 (lse for rows 0-63, D for 64-127).  Loaded a tile ahead
        // (the global load's latency had sat at the top of every tile)
        auto lse_d = [&](int tt) -> float {
            const int i = (qt0 + tt) * 64 + (row & 63);
            const long li = ((long)b * p.hc + hq) * p.s_q + i;
            return i < p.s_q ? (row < 64 ? p.lse[li] * 1.4426950408889634f : p.D[li]) : 0.f;
        };
        float ld_next = (h == 0 && nqt > 0) ? lse_d(0) : 0.f;
        for (int t = 0; t < nqt; ++t) {
            const int q0 = (qt0 + t) * 64;
            // this tile's lse and D into shared memory
            float *lt = ld + (t & 1) * 128;
            if (h == 0) {
                lt[row] = ld_next;
                if (t + 1 < nqt) ld_next = lse_d(t + 1);
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&st_full[t & 1], (t >> 1) & 1, abort, err));
            ok = __all_sync(0xffffffffu, ok && mbar_wait(dpt_full, t & 1, abort, err));
            tc_fence_after();
            const uint32_t sbuf = B_ST + (t & 1) * 64;
            uint32_t sr[32], dr[32];
            if (ok) {
                tmem_ld32(lb + sbuf + 32 * h, sr);
                tmem_ld32(lb + B_DPT + 32 * h, dr);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) sr[c] = dr[c] = 0u;
            }
            // every thread has read its S^T and dP^T columns (and the lse / D rows are in
            // place) before any writes P^T / dS^T over them; dP^T may then take the next tile
            tc_fence_before();
            named_bar_sync(1, 256);
            if (warp == 4 && lane == 0) mbar_arrive(dpt_free);
            // The visibility test only where the warp's 32 keys can miss some of the half-tile's
            // queries (warp-uniform), in a loop of its own: a test inside one loop serialises
            // the exponentials.  lse and D are the same for every lane: 16-byte shared loads.
            const int kmax = k0 + quad * 32 + 31;
            const bool interior = kmax < p.kv_need && (!p.causal || kmax <= p.q_offset + q0 + 32 * h) &&
                                  q0 + 32 * h + 32 <= p.s_q;
            uint32_t pk[16], dk[16];
            if (interior) {
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 l4 = *(const float4 *)(lt + 32 * h + c), d4 = *(const float4 *)(lt + 64 + 32 * h + c);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                    float pv[4], dsv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pv[e] = ex2(fmaf(__uint_as_float(sr[c + e]), p.scale_log2, -lv[e]));
                        dsv[e] = pv[e] * (__uint_as_float(dr[c + e]) - dv4[e]) * p.scale;
                    }
                    pk[c / 2] = pack_f16(pv[0], pv[1]);
                    pk[c / 2 + 1] = pack_f16(pv[2], pv[3]);
                    dk[c / 2] = pack_f16(dsv[0], dsv[1]);
                    dk[c / 2 + 1] = pack_f16(dsv[2], dsv[3]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float pv[2], dsv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int qi = 32 * h + c + e, i = q0 + qi;
                        const bool vis = i < p.s_q && j < p.kv_need && (!p.causal || j <= p.q_offset + i);
                        const float pr = vis ? ex2(fmaf(__uint_as_float(sr[c + e]), p.scale_log2, -lt[qi])) : 0.f;
                        pv[e] = pr;
                        dsv[e] = pr * (__uint_as_float(dr[c + e]) - lt[64 + qi]) * p.scale;
                    }
                    pk[c / 2] = pack_f16(pv[0], pv[1]);
                    dk[c / 2] = pack_f16(dsv[0], dsv[1]);
                }
            }
            if (ok) {
                tmem_st16(lb + sbuf + 16 * h, pk);
                tmem_st16(lb + sbuf + 32 + 16 * h, dk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ps_full);
        }
        // ---- epilogue: half 0 writes dV^T and the band's dk_rot, half 1 dK_nope^T
        if (nqt > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(acc_done, 0, abort, err));
        tc_fence_after();
        const long e_stride = (long)p.B * p.kv_pad;                          // between rows of dKV^T
        __half *dst = p.dkvt + ((long)hl * 256 * p.B + b) * p.kv_pad + j;    // row 0 of this key
#pragma unroll 1
        for (int part = 0; part < 4 + (h == 0 ? 2 : 0); ++part) {
            // half 0: dV columns 0-127 (parts 0-3), dk_rot 0-63 (parts 4-5); half 1: dK_nope 0-127
            uint32_t r[32];
            const uint32_t col = h == 0 ? (part < 4 ? B_DV + 32 * part : B_DK + 128 + 32 * (part - 4)) : B_DK + 32 * part;
            if (ok && nqt > 0) {
                tmem_ld32(lb + col, r);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] = 0u;
            }
            if (h == 0 && part >= 4) {
                float *o = p.dkr + (((long)b * p.nh + hl) * p.kv_pad + j) * 64 + 32 * (part - 4);
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *(float4 *)(o + c) = make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                                     __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
            } else {
                const int e0 = (h == 0 ? 128 : 0) + 32 * part;   // row of [dK_nope^T ; dV^T]
#pragma unroll
                for (int c = 0; c < 32; ++c) dst[(long)(e0 + c) * e_stride] = __float2half_rn(__uint_as_float(r[c]));
            }
        }
    }
    if (tid == 0 && *abort) settle();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------- query-stationary ----
constexpr uint32_t A_OFF_Q = 0, A_OFF_DO = 3 * KBOX, A_OFF_K = A_OFF_DO + 2 * KBOX;   // Q, dO, K ring (2 x 3 boxes)
constexpr uint32_t A_OFF_V = A_OFF_K + 6 * KBOX;                                      // V^T stage (2 boxes)
constexpr uint32_t A_OFF_BAR = A_OFF_V + 2 * KBOX;
constexpr uint32_t A_SMEM = A_OFF_BAR + 256 + 1024;
// TMEM: S 0-127, dP / dS 128-255, dQ (d_nope 128 + band 64) 256-447
constexpr uint32_t A_S = 0, A_DP = 128, A_DQ = 256;
constexpr int A_NSM = 16;   // softmax warps: four threads per query row

struct DqK {
    int s_q, kv_need, q_offset, causal, hc, h0, nh, n_qt;
    float scale, scale_log2;
    const float *lse, *D;
    __nv_bfloat16 *dq_nope;         // [B][s_q][hc][128]
    float *dqr;                     // [B][s_q][hc][64]
    uint32_t idesc_s, idesc_dp, idesc_dq;
};

__global__ void __launch_bounds__(32 * (A_NSM + 4), 1)
    tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap mKn, const __grid_constant__ CUtensorMap mKr,
                     const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mQn,
                     const __grid_constant__ CUtensorMap mQr, const __grid_constant__ CUtensorMap mDo, DqK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + A_OFF_BAR);
    uint64_t *q_full = bars, *k_full = bars + 1, *k_empty = bars + 3, *v_full = bars + 5, *v_empty = bars + 6;
    uint64_t *s_full = bars + 7, *s_free = bars + 8, *dp_full = bars + 9, *ds_full = bars + 10, *dp_free = bars + 11;
    uint64_t *dq_done = bars + 12;
    uint32_t *tslot = (uint32_t *)(bars + 16);
    volatile int *abort = (volatile int *)(tslot + 1);
    unsigned *err = &g_tc_bwd_err;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (query tile, heaviest first; head; batch)
    const int nhb = p.nh * gridDim.y;
    const int u = blockIdx.x;
    const int qt = p.n_qt - 1 - u / p.nh, hl = u % p.nh, b = blockIdx.y, hq = p.h0 + hl;
    (void)nhb;
    const int q0 = qt * 128;
    const int kv_end = p.causal ? min(p.kv_need, p.q_offset + q0 + 128) : p.kv_need;
    const int nt = (kv_end + 127) / 128;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 1);
        mbar_init(dp_full, 1);
        mbar_init(ds_full, A_NSM);
        mbar_init(dp_free, 1);
        mbar_init(dq_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && nt > 0) {
            mbar_arrive_expect_tx(q_full, 5 * KBOX);
            tma_load_4d(smem + A_OFF_Q, &mQn, q_full, 0, hq, q0, b);
            tma_load_4d(smem + A_OFF_Q + KBOX, &mQn, q_full, 64, hq, q0, b);
            tma_load_4d(smem + A_OFF_Q + 2 * KBOX, &mQr, q_full, 0, hq, q0, b);
            tma_load_4d(smem + A_OFF_DO, &mDo, q_full, 0, hq, q0, b);
            tma_load_4d(smem + A_OFF_DO + KBOX, &mDo, q_full, 64, hq, q0, b);
            for (int T = 0; T < nt; ++T) {
                const int ks = T & 1;
                if (T >= 2 && !mbar_wait(&k_empty[ks], ((T >> 1) - 1) & 1, abort, err)) break;
                uint8_t *kd = smem + A_OFF_K + ks * 3 * KBOX;
                mbar_arrive_expect_tx(&k_full[ks], 3 * KBOX);
                tma_load_3d(kd, &mKn, &k_full[ks], hl * 128, T * 128, b);
                tma_load_3d(kd + KBOX, &mKn, &k_full[ks], hl * 128 + 64, T * 128, b);
                tma_load_3d(kd + 2 * KBOX, &mKr, &k_full[ks], 0, T * 128, b);
                if (T >= 1 && !mbar_wait(v_empty, (T - 1) & 1, abort, err)) break;
                mbar_arrive_expect_tx(v_full, 2 * KBOX);
                tma_load_3d(smem + A_OFF_V, &mV, v_full, T * 128, hl * 128, b);
                tma_load_3d(smem + A_OFF_V + KBOX, &mV, v_full, T * 128 + 64, hl * 128, b);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- S = Q K^T, dP = dO V^T
        bool ok = nt > 0 && __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort, err));
        for (int T = 0; T < nt && ok; ++T) {
            const int ks = T & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&k_full[ks], (T >> 1) & 1, abort, err));
            if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(s_free, (T - 1) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            const uint8_t *kd = smem + A_OFF_K + ks * 3 * KBOX;
            if (elect_one()) {
#pragma unroll
                for (int kb = 0; kb < 3; ++kb) {
                    const uint64_t da = sdesc_kmajor(smem + A_OFF_Q + kb * KBOX), db = sdesc_kmajor(kd + kb * KBOX);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_ss(tmem + A_S, da + 2 * k4, db + 2 * k4, p.idesc_s, (kb | k4) != 0);
                }
                mma_commit(s_full);
            }
            __syncwarp();
            ok = __all_sync(0xffffffffu, mbar_wait(v_full, T & 1, abort, err));
            // dS of the previous tile (in the dP columns) has been read by its dQ MMAs
            if (ok && T > 0) ok = __all_sync(0xffffffffu, mbar_wait(dp_free, (T - 1) & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                // B = V (keys x d_v) read from V^T as an MN-major operand: two 64-key blocks
                const uint64_t bv = sdesc_mnmajor(smem + A_OFF_V, KBOX);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ss(tmem + A_DP, sdesc_kmajor(smem + A_OFF_DO + (k >> 2) * KBOX) + 2 * (k & 3),
                           bv + (uint64_t)(k * (2048 >> 4)), p.idesc_dp, k != 0);
                mma_commit(dp_full);
                mma_commit(v_empty);
            }
            __syncwarp();
        }
    } else if (warp == 2) {
        // --------------------------------------------------------------- dQ += dS K
        bool ok = true;
        for (int T = 0; T < nt && ok; ++T) {
            ok = __all_sync(0xffffffffu, mbar_wait(ds_full, T & 1, abort, err));
            if (!ok) break;
            tc_fence_after();
            const uint8_t *kd = smem + A_OFF_K + (T & 1) * 3 * KBOX;
            if (elect_one()) {
                const uint64_t bk = sdesc_mnmajor(kd, KBOX);   // K^T: three 64-dim blocks
#pragma unroll
                for (int k = 0; k < 8; ++k)   // 16 keys per step
                    mma_ts(tmem + A_DQ, tmem + A_DP + k * 8, bk + (uint64_t)(k * (2048 >> 4)), p.idesc_dq, (T | k) != 0);
                mma_commit(&k_empty[T & 1]);
                mma_commit(dp_free);
                if (T == nt - 1) mma_commit(dq_done);
            }
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ------------------------------------------ dS (warps 4-19), epilogue
        const int quad = warp & 3, qr = (warp - 4) >> 2;   // quarter qr: keys [32 qr, 32 qr + 32)
        const int row = quad * 32 + lane, i = q0 + row;
        const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
        const long li = ((long)b * p.hc + hq) * p.s_q + i;
        const float lse2 = i < p.s_q ? p.lse[li] * 1.4426950408889634f : 0.f;
        const float Di = i < p.s_q ? p.D[li] : 0.f;
        const int pos = p.q_offset + i;
        bool ok = true;
        for (int T = 0; T < nt; ++T) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(s_full, T & 1, abort, err));
            ok = __all_sync(0xffffffffu, ok && mbar_wait(dp_full, T & 1, abort, err));
            tc_fence_after();
            uint32_t sr[32], dr[32];
            if (ok) {
                tmem_ld32(lb + A_S + 32 * qr, sr);
                tmem_ld32(lb + A_DP + 32 * qr, dr);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) sr[c] = dr[c] = 0u;
            }
            // all quarters have read S and dP before dS is written over dP and S is freed
            tc_fence_before();
            named_bar_sync(1, 32 * A_NSM);
            if (warp == 4 && lane == 0) mbar_arrive(s_free);
            // the visibility test only where the chunk can hold hidden keys (warp-uniform)
            const int j0 = T * 128 + 32 * qr;
            const bool edge = j0 + 32 > p.kv_need || (p.causal && j0 + 31 > p.q_offset + q0);
            const bool row_ok = i < p.s_q;
            const float nDs = -Di * p.scale;
            // (two whole loops rather than a test inside one, so that each stays one straight
            // run the compiler can interleave)
            uint32_t dk[16];
            if (edge) {
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float dsv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = j0 + c + e;
                        const bool vis = row_ok && key < p.kv_need && (!p.causal || key <= pos);
                        const float pr = vis ? ex2(fmaf(__uint_as_float(sr[c + e]), p.scale_log2, -lse2)) : 0.f;
                        dsv[e] = pr * fmaf(__uint_as_float(dr[c + e]), p.scale, nDs);
                    }
                    dk[c / 2] = pack_f16(dsv[0], dsv[1]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float dsv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pr = ex2(fmaf(__uint_as_float(sr[c + e]), p.scale_log2, -lse2));
                        dsv[e] = (row_ok ? pr : 0.f) * fmaf(__uint_as_float(dr[c + e]), p.scale, nDs);
                    }
                    dk[c / 2] = pack_f16(dsv[0], dsv[1]);
                }
            }
            if (ok) {
                tmem_st16(lb + A_DP + 16 * qr, dk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
        }
        // ---- epilogue: quarter qr stores dQ columns [48 qr, 48 qr + 48): d_nope 0-127 as
        // bf16, the rotated band 128-191 as fp32
        if (nt > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(dq_done, 0, abort, err));
        tc_fence_after();
        const bool store = ok && nt > 0 && i < p.s_q;
        const long qrow = ((long)b * p.s_q + i) * p.hc + hq;
#pragma unroll 1
        for (int part = 0; part < 6; ++part) {   // 8 columns at a time
            uint32_t r[8];
            const int col = 48 * qr + 8 * part;
            if (ok && nt > 0) {
                tmem_ld8(lb + A_DQ + col, r);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) r[c] = 0u;
            }
            if (!store) continue;
            if (col < 128) {
                uint32_t w[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) w[c] = pack_bf16(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
                *(uint4 *)(p.dq_nope + qrow * 128 + col) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                float *o = p.dqr + qrow * 64 + (col - 128);
                *(float4 *)o = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]),
                                           __uint_as_float(r[3]));
                *(float4 *)(o + 4) = make_float4(__uint_as_float(r[4]), __uint_as_float(r[5]), __uint_as_float(r[6]),
                                                 __uint_as_float(r[7]));
            }
        }
    }
    if (tid == 0 && *abort) settle();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_bwd_prep_tc(int B, int s_q, int hc, const void *q_nope, const void *dout, const void *out,
                               void *qn16, void *do16, float *D, cudaStream_t st) {
    const long rows = (long)B * s_q * hc;
    if (rows == 0) return cudaSuccess;
    ProfScope ps("bwd_prep", st);
    bwd_prep_tc_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(
        rows, hc, s_q, (const __nv_bfloat16 *)q_nope, (const __nv_bfloat16 *)dout, (const __nv_bfloat16 *)out,
        (__half *)qn16, (__half *)do16, D);
    return cudaGetLastError();
}

cudaError_t launch_transpose16(long R, long C, const void *x, void *y, cudaStream_t st) {
    if (R == 0 || C == 0) return cudaSuccess;
    ProfScope ps("bwd_rows", st);
    if (R % 8 == 0 && C % 8 == 0 && ((uintptr_t)x & 15) == 0 && ((uintptr_t)y & 15) == 0)
        transpose16_vec_kernel<<<dim3((unsigned)((C + 63) / 64), (unsigned)((R + 63) / 64)), 256, 0, st>>>(
            R, C, (const uint4 *)x, (uint4 *)y);
    else
        transpose16_kernel<<<dim3((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32)), 256, 0, st>>>(
            R, C, (const uint16_t *)x, (uint16_t *)y);
    return cudaGetLastError();
}

// Attention backward of one head shard on the tensor cores.  kws: K_nope [B][kv_pad][hs*128]
// fp16, vws: V^T [B][hs*128][kv_pad] fp16, kpe: rotated k_pe [B][kv_pad][64] fp16, qn16 /
// do16: fp16 q_nope / dO [B][s_q][hc][128], qpe: rotated q_pe fp16 [B][s_q][hc][64].
cudaError_t tc_bwd_attn(const TcPrefill &p, int h0, int nh, const void *kws, const void *vws, const void *kpe,
                        const void *qn16, const void *qpe, const void *do16, const float *lse, const float *D,
                        void *dq_nope, float *dqr, void *dkvt, float *dkr, cudaStream_t st) {
    const long kv_pad = (p.kv_need + 127) / 128 * 128;
    cudaError_t e;
    CUtensorMap mKn, mKr, mV, mQn[2], mQr[2], mDo[2];   // [0]: 128-row boxes, [1]: 64-row boxes
    {
        unsigned long long d[3] = {(unsigned long long)p.hs * 128, (unsigned long long)kv_pad, (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)p.hs * 256, (unsigned long long)kv_pad * p.hs * 256};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mKn, kws, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {64, (unsigned long long)kv_pad, (unsigned long long)p.B};
        unsigned long long s[2] = {128, (unsigned long long)kv_pad * 128};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mKr, kpe, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {(unsigned long long)kv_pad, (unsigned long long)p.hs * 128, (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)kv_pad * 2, (unsigned long long)p.hs * 128 * kv_pad * 2};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mV, vws, 3, d, s, box)) != cudaSuccess) return e;
    }
    for (int v = 0; v < 2; ++v) {
        const unsigned rows = v == 0 ? 128 : 64;
        unsigned box[4] = {64, 1, rows, 1};
        unsigned long long d[4] = {128, (unsigned long long)p.head_count, (unsigned long long)p.s_q,
                                   (unsigned long long)p.B};
        unsigned long long s[3] = {256, (unsigned long long)p.head_count * 256,
                                   (unsigned long long)p.s_q * p.head_count * 256};
        if ((e = make_tma_map(&mQn[v], qn16, 4, d, s, box)) != cudaSuccess) return e;
        if ((e = make_tma_map(&mDo[v], do16, 4, d, s, box)) != cudaSuccess) return e;
        unsigned long long dr[4] = {64, (unsigned long long)p.head_count, (unsigned long long)p.s_q,
                                    (unsigned long long)p.B};
        unsigned long long sr[3] = {128, (unsigned long long)p.head_count * 128,
                                    (unsigned long long)p.s_q * p.head_count * 128};
        if ((e = make_tma_map(&mQr[v], qpe, 4, dr, sr, box)) != cudaSuccess) return e;
    }
    const float scale_log2 = p.scale * 1.4426950408889634f;
    {   // key-stationary: dK, dV, dk_rot
        DkvK a{};
        a.s_q = p.s_q;
        a.kv_need = (int)p.kv_need;
        a.q_offset = p.q_offset;
        a.causal = p.causal;
        a.hc = p.head_count;
        a.h0 = h0;
        a.nh = nh;
        a.n_kt = (int)(kv_pad / 128);
        a.scale = p.scale;
        a.scale_log2 = scale_log2;
        a.lse = lse;
        a.D = D;
        a.dkvt = (__half *)dkvt;
        a.kv_pad = kv_pad;
        a.B = p.B;
        a.dkr = dkr;
        a.idesc_st = idesc_f16(128, 64, true);
        a.idesc_dpt = idesc_f16(128, 64, true, false, true);   // A = V, MN-major
        a.idesc_dv = idesc_f16(128, 128, true, true);           // B = dO^T, MN-major
        a.idesc_dk = idesc_f16(128, 192, true, true);           // B = Q^T, MN-major
        e = cudaFuncSetAttribute(tc_bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)B_SMEM);
        if (e != cudaSuccess) return e;
        ProfScope ps("tc_bwd_dkv", st);
        tc_bwd_dkv_kernel<<<dim3((unsigned)(a.n_kt * nh * p.B)), dim3(384), B_SMEM, st>>>(mKn, mKr, mV, mQn[1],
                                                                                            mQr[1], mDo[1], a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {   // query-stationary: dQ
        DqK a{};
        a.s_q = p.s_q;
        a.kv_need = (int)p.kv_need;
        a.q_offset = p.q_offset;
        a.causal = p.causal;
        a.hc = p.head_count;
        a.h0 = h0;
        a.nh = nh;
        a.n_qt = (p.s_q + 127) / 128;
        a.scale = p.scale;
        a.scale_log2 = scale_log2;
        a.lse = lse;
        a.D = D;
        a.dq_nope = (__nv_bfloat16 *)dq_nope;
        a.dqr = dqr;
        a.idesc_s = idesc_f16(128, 128, true);
        a.idesc_dp = idesc_f16(128, 128, true, true);   // B = V, MN-major
        a.idesc_dq = idesc_f16(128, 192, true, true);   // B = K^T, MN-major
        e = cudaFuncSetAttribute(tc_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)A_SMEM);
        if (e != cudaSuccess) return e;
        ProfScope ps("tc_bwd_dq", st);
        tc_bwd_dq_kernel<<<dim3((unsigned)(a.n_qt * nh), (unsigned)p.B), dim3(32 * (A_NSM + 4)), A_SMEM, st>>>(
            mKn, mKr, mV, mQn[0], mQr[0], mDo[0], a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t tc_bwd_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_bwd_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_bwd_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

}  // namespace mla
