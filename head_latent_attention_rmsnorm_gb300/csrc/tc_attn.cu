// tc_attn.cu -- explicit-form (LAGA per-rank) MLA prefill on the sm_103a tensor
// cores, and the host sequence that drives it.
//
// Method ("A Training-Memory Regression in MLA Sequence Parallelism ... LAGA",
// arXiv 2607.17644, "What carries the argument", Fig. 2 and the paper's section
// 3.3): rebuild per-head K_nope / V from the normalised latent through W_kv_b one
// head shard at a time, then head-dim causal attention with
//   s_ij = scale * (q_nope_i . K_nope_j + RoPE(q_pe_i) . RoPE(k_pe_j)),
// softmax over visible keys (j <= q_offset + i), output plus log-sum-exp.
//
// Kernel: persistent, one CTA per SM (256 threads) walking work units = (128-query
// tile, head, batch), heaviest first under the causal mask, in rounds that alternate
// direction; TMEM, barriers and the TMA rings carry over from one unit to the next.
//   warp 0    TMA producer of each unit's Q (staged in shared memory) and of the K tiles
//             (K_nope 128 + RoPE band 64 dims), 2-deep ring.
//   warp 6    TMA producer of V^T tiles, 2-deep ring (separate, so that a wait for a
//             free V slot never holds back the next K tile).
//   warp 1    tcgen05 issuer of the scores: S_j = Q K_j^T (M=128, N=128, K=192, Q from
//             TMEM) into TMEM S buffer j & 1, as soon as K_j has landed and P.V_{j-2}
//             (which read that buffer) is done.  Also owns the TMEM allocation.
//   warp 7    tcgen05 issuer of O += P_j V_j (M=128, N=128, K=128), P read from TMEM
//             where the softmax wrote it over S_j.  Two issuing threads keep the tensor
//             pipe fed: a thread that waits on an mbarrier between MMA batches leaves
//             the pipe idle for ~100-200 cycles, so neither issuer waits on the other.
//   warps 2-5 first move the row's Q (bf16 q_nope widened to fp16, q_pe rotated by
//             RoPE) into TMEM; then the softmax, one thread per query row (TMEM lane =
//             row; the tile's 128 scores in the thread's registers, so the row maximum
//             needs no exchange between threads and no CTA barrier): online softmax in
//             the log2 domain; O in TMEM is rescaled only when a row maximum grows by
//             more than 2^8 (the stale maximum keeps every p <= 256, exact after the
//             final division); epilogue O / l and lse.  (Sixteen warps with four threads
//             per row and a barrier for the row maximum ran the same tiles no faster.)
// Operands are fp16 (11-bit significand); K_nope, V^T and the rotated k_pe band are
// produced in fp16 by the reconstruction GEMMs and the prep launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_attn_err = 0;

namespace {

using namespace tc;

constexpr int BQ = 128, BKV = 128;
constexpr uint32_t BOX = 128 * 128;            // one 128-row x 64-element fp16 box
constexpr uint32_t K_BYTES = 3 * BOX;          // K_nope lo, K_nope hi, RoPE band
constexpr uint32_t V_BYTES = 2 * BOX;          // V^T: 128 dv rows x 2 key halves (what the TMA brings)
// Each V^T box is followed by 16 constant rows (a row of ones, 15 of zeros): the P.V MMA
// runs with N = 144, so O column 128 accumulates the row sum of P exactly as the MMA used
// it, and the softmax needs no sum of its own.
constexpr uint32_t ONES = 16 * 128;
constexpr uint32_t VBOX = BOX + ONES;          // one key half of a V slot
constexpr uint32_t V_SLOT = 2 * VBOX;
constexpr int KST = 2, VST = 2;
constexpr uint32_t QS_BYTES = 3 * BOX;         // staged Q of the next unit: q_nope lo, hi (bf16), rotated q_pe (fp16)
constexpr int NSM = 4;                        // softmax warps: one thread per query row
// Q staging, K/V rings, 1 KB alignment slack, 256 B of barriers
constexpr uint32_t SMEM_BYTES = QS_BYTES + KST * K_BYTES + VST * V_SLOT + 1024 + 256;
// TMEM columns: S buffers 0-127 and 128-255, O 256-399 (dv 0-127, row sum 128, zeros),
// Q (192 fp16 = 96 columns) 400-495
constexpr uint32_t T_O = 256, T_L = T_O + 128, T_Q = 400;
constexpr float RESCALE_LOG2 = 8.0f;

struct AttnK {
    int s_q, kv_need, q_offset, causal;
    int head_off;       // first query/output head of this shard
    float scale_log2;   // softmax scale * log2(e)
    __nv_bfloat16 *out;
    long out_b, out_i, out_h;
    int out_v8;   // the output rows' quarters are 32-byte aligned (32-byte stores)
    float *lse;
    long lse_b, lse_h;
    uint32_t idesc_s, idesc_pv;
    int nh, nb, n_qt, units;       // heads of this launch, batch, query tiles, work units
};

// One work unit = (128-query tile, head, batch).  Units are numbered heaviest first
// under the causal mask: (head, batch) fastest, query tiles from the latest down.
struct Work {
    int hl, b, q0, nt;
};
__device__ __forceinline__ Work work_of(const AttnK &p, int u) {
    const int nhb = p.nh * p.nb;
    const int hb = u % nhb;
    Work w;
    w.hl = hb % p.nh;
    w.b = hb / p.nh;
    w.q0 = (p.n_qt - 1 - u / nhb) * BQ;
    const int kv_end = p.causal ? min(p.kv_need, p.q_offset + w.q0 + BQ) : p.kv_need;
    w.nt = (kv_end + BKV - 1) / BKV;
    return w;
}
// Unit of round k for CTA c of G: rounds alternate direction over the heaviest-first
// list, so every CTA gets a mix of heavy and light units.
__device__ __forceinline__ int unit_at(int k, int c, int G) { return (k & 1) ? (k + 1) * G - 1 - c : k * G + c; }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(32 * (NSM + 4), 1)
    tc_attn_kernel(const __grid_constant__ CUtensorMap mQn, const __grid_constant__ CUtensorMap mQr,
                   const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mKr,
                   const __grid_constant__ CUtensorMap mV, AttnK p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQs = smem;
    uint8_t *sK = sQs + QS_BYTES;
    uint8_t *sV = sK + KST * K_BYTES;
    uint64_t *bars = (uint64_t *)(sV + VST * V_SLOT);
    uint64_t *q_ready = bars + 0;
    uint64_t *k_full = bars + 1, *k_empty = k_full + KST;
    uint64_t *v_full = k_empty + KST, *v_empty = v_full + VST;
    uint64_t *s_full = v_empty + VST, *p_full = s_full + 2, *pv_done = p_full + 2;
    uint64_t *o_done = pv_done + 2, *o_final = o_done + 1, *o_free = o_final + 1, *qs_full = o_free + 1;
    uint32_t *tslot = (uint32_t *)(bars + 24);
    volatile int *abort = (volatile int *)(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;

    if (tid == 0) {
        mbar_init(q_ready, NSM);
        for (int i = 0; i < KST; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VST; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], NSM);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(o_done, 1);
        mbar_init(o_final, 1);
        mbar_init(o_free, NSM);   // the softmax warps have read O out of TMEM
        mbar_init(qs_full, 1);    // a unit's Q has landed in the staging buffer
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    // the constant rows after every V^T box: row 0 ones (fp16 1.0), rows 1-15 zeros (a
    // row that is constant is unchanged by the 128-byte swizzle)
    for (int i = tid; i < VST * 2 * (int)(ONES / 16); i += blockDim.x) {
        const int box = i / (ONES / 16), off = i % (ONES / 16);   // 16-byte chunk of the block
        const uint32_t v = off < 8 ? 0x3c003c00u : 0u;             // first 128-byte row: ones
        *(uint4 *)(sV + (box >> 1) * V_SLOT + (box & 1) * VBOX + BOX + off * 16) = make_uint4(v, v, v, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;   // S0: cols 0-127, S1: 128-255, O: 256-383, Q: 384-479
    // The prologue overlaps the reconstruction GEMM (programmatic launch).  Every role
    // waits for it (pdl_wait) before touching K_nope, V^T, the rotated k_pe or the RoPE
    // table; the softmax warps first read their first unit's q rows, which are inputs.

    // Every role walks the same units in the same order and counts key tiles T across
    // units, so ring slots and barrier parities continue from one unit to the next.
    if (warp == 0) {
        // ------------------------------- Q of each unit and K tiles (TMA)
        if (lane == 0) {
            pdl_wait();
            tma_prefetch_desc(&mQn);
            tma_prefetch_desc(&mQr);
            tma_prefetch_desc(&mK);
            tma_prefetch_desc(&mKr);
            bool ok = true;
            int T = 0, n = 0;
            for (int k = 0; k * G < p.units && ok; ++k) {
                const int u = unit_at(k, c, G);
                if (u >= p.units) continue;
                const Work w = work_of(p, u);
                // this unit's Q into the staging buffer, once the softmax warps have moved
                // the previous unit's Q into TMEM (this runs a couple of key tiles ahead of
                // them, so the load has that long to land)
                if (n > 0 && !mbar_wait(q_ready, (n - 1) & 1, abort, &g_tc_attn_err)) break;
                ++n;
                mbar_arrive_expect_tx(qs_full, QS_BYTES);
                tma_load_4d(sQs, &mQn, qs_full, 0, p.head_off + w.hl, w.q0, w.b);
                tma_load_4d(sQs + BOX, &mQn, qs_full, 64, p.head_off + w.hl, w.q0, w.b);
                tma_load_4d(sQs + 2 * BOX, &mQr, qs_full, 0, p.head_off + w.hl, w.q0, w.b);
                for (int j = 0; j < w.nt; ++j, ++T) {
                    const int ks = T % KST;
                    if (T >= KST && !mbar_wait(&k_empty[ks], ((T / KST) - 1) & 1, abort, &g_tc_attn_err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *kd = sK + ks * K_BYTES;
                    mbar_arrive_expect_tx(&k_full[ks], K_BYTES);
                    tma_load_3d(kd, &mK, &k_full[ks], w.hl * 128, j * BKV, w.b);
                    tma_load_3d(kd + BOX, &mK, &k_full[ks], w.hl * 128 + 64, j * BKV, w.b);
                    tma_load_3d(kd + 2 * BOX, &mKr, &k_full[ks], 0, j * BKV, w.b);
                }
            }
        }
    } else if (warp == 2 + NSM) {
        // ----------------------------------------------------- V^T tiles (TMA)
        if (lane == 0) {
            pdl_wait();
            tma_prefetch_desc(&mV);
            bool ok = true;
            int T = 0;
            for (int k = 0; k * G < p.units && ok; ++k) {
                const int u = unit_at(k, c, G);
                if (u >= p.units) continue;
                const Work w = work_of(p, u);
                for (int j = 0; j < w.nt; ++j, ++T) {
                    const int vs = T % VST;
                    if (T >= VST && !mbar_wait(&v_empty[vs], ((T / VST) - 1) & 1, abort, &g_tc_attn_err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *vd = sV + vs * V_SLOT;
                    mbar_arrive_expect_tx(&v_full[vs], V_BYTES);
                    tma_load_3d(vd, &mV, &v_full[vs], j * BKV, w.hl * 128, w.b);
                    tma_load_3d(vd + VBOX, &mV, &v_full[vs], j * BKV + 64, w.hl * 128, w.b);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- score MMA issuer
        // The whole warp runs the loop (warp-uniform control flow keeps the operands in
        // uniform registers) and one elected lane issues the MMAs.
        {
            pdl_wait();
            bool ok = true;
            int T = 0, n = 0;   // key tiles, units so far
            for (int k = 0; k * G < p.units && ok; ++k) {
                const int u = unit_at(k, c, G);
                if (u >= p.units) continue;
                const Work w = work_of(p, u);
                // this unit's Q is in TMEM
                if (!__all_sync(0xffffffffu, mbar_wait(q_ready, n & 1, abort, &g_tc_attn_err))) break;
                ++n;
                for (int j = 0; j < w.nt; ++j, ++T) {
                    const int ks = T % KST;
                    bool go = __all_sync(0xffffffffu, mbar_wait(&k_full[ks], (T / KST) & 1, abort, &g_tc_attn_err));
                    // S buffer T & 1 last held P_{T-2}: P.V_{T-2} must have read it
                    if (go && T >= 2)
                        go = __all_sync(0xffffffffu, mbar_wait(&pv_done[T & 1], ((T - 2) >> 1) & 1, abort, &g_tc_attn_err));
                    if (!go) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t s_tm = tmem + (T & 1) * 128;
                    const uint8_t *kd = sK + ks * K_BYTES;
                    if (elect_one()) {
#pragma unroll
                        for (int kb = 0; kb < 3; ++kb) {
                            const uint64_t db = sdesc_kmajor(kd + kb * BOX);
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                mma_ts(s_tm, tmem + T_Q + (kb * 4 + k4) * 8, db + 2 * k4, p.idesc_s, (kb | k4) != 0);
                        }
                        mma_commit(&s_full[T & 1]);
                        mma_commit(&k_empty[ks]);
                    }
                    __syncwarp();
                }
            }
        }
    } else if (warp == 3 + NSM) {
        // ------------------------------------------------------------ P.V issuer
        // (warp-uniform loop, one elected lane issues, as for the scores)
        {
            pdl_wait();
            bool ok = true;
            int T = 0, n = 0;
            for (int k = 0; k * G < p.units && ok; ++k) {
                const int u = unit_at(k, c, G);
                if (u >= p.units) continue;
                const Work w = work_of(p, u);
                // the epilogue of the previous unit has read O before P.V_0 overwrites it
                if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(o_free, (n - 1) & 1, abort, &g_tc_attn_err))) break;
                ++n;
                for (int j = 0; j < w.nt; ++j, ++T) {
                    const int vs = T % VST;
                    bool go = __all_sync(0xffffffffu, mbar_wait(&p_full[T & 1], (T >> 1) & 1, abort, &g_tc_attn_err));
                    go = go && __all_sync(0xffffffffu, mbar_wait(&v_full[vs], (T / VST) & 1, abort, &g_tc_attn_err));
                    if (!go) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_tm = tmem + (T & 1) * 128;
                    const uint8_t *vd = sV + vs * V_SLOT;
                    if (elect_one()) {
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            const uint64_t db = sdesc_kmajor(vd + kb * VBOX);   // 144 rows: V^T + constant rows
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                mma_ts(tmem + T_O, p_tm + kb * 32 + k4 * 8, db + 2 * k4, p.idesc_pv, (j | kb | k4) != 0);
                        }
                        mma_commit(&v_empty[vs]);
                        mma_commit(&pv_done[T & 1]);
                        mma_commit(o_done);
                    }
                    __syncwarp();
                }
                if (elect_one()) mma_commit(o_final);
                __syncwarp();
            }
        }
    } else if (warp >= 2 && warp < 2 + NSM) {
        // ---------------------------------------------------------- softmax warps
        // One thread per query row (TMEM lane = row: warp w reaches lanes 32 (w & 3) ..);
        // a tile's 128 scores of the row sit in the thread's registers, so its maximum
        // needs no exchange with other threads and the warps never wait on one another.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        // A failed wait clears `ok` (warp-uniform); the loops run on so that every role
        // keeps its barrier counts.
        bool ok = true;
        int T = 0, n = 0;
        // this CTA's units in order: round k, skipping rounds past the end
        auto next_unit = [&](int k) -> int {
            for (; k * G < p.units; ++k)
                if (unit_at(k, c, G) < p.units) return k;
            return k;
        };
        // ---- a unit's Q from the staging buffer into TMEM (the previous unit's score MMAs
        // have all completed: their S tiles were read).  Run for unit n + 1 right after unit
        // n's last tile, before unit n's epilogue, so that the next unit's first score MMAs
        // overlap the last P.V and the epilogue.  The row's q_nope (bf16, two 64-dim boxes)
        // widened to fp16 into columns 0-63, its rotated q_pe (fp16) into columns 64-95; rows
        // past s_q arrive as zeros.  16-byte chunk c of row r of a staged box sits at chunk
        // c ^ (r & 7).
        auto load_q = [&](int nn) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(qs_full, nn & 1, abort, &g_tc_attn_err));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t *qrow_s = sQs + h * BOX + row * 128;
                uint32_t qn[2][16];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 v = *(const uint4 *)(qrow_s + ((cc ^ (row & 7)) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        qn[cc >> 2][4 * (cc & 3) + i] =
                            pack_f16(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xffff0000u));
                }
                tmem_st16(lane_base + T_Q + 32 * h, qn[0]);
                tmem_st16(lane_base + T_Q + 32 * h + 16, qn[1]);
            }
            {
                const uint8_t *prow = sQs + 2 * BOX + row * 128;
                uint32_t pe[2][16];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 v = *(const uint4 *)(prow + ((cc ^ (row & 7)) << 4));
                    pe[cc >> 2][4 * (cc & 3)] = v.x, pe[cc >> 2][4 * (cc & 3) + 1] = v.y;
                    pe[cc >> 2][4 * (cc & 3) + 2] = v.z, pe[cc >> 2][4 * (cc & 3) + 3] = v.w;
                }
                tmem_st16(lane_base + T_Q + 64, pe[0]);
                tmem_st16(lane_base + T_Q + 80, pe[1]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        };
        int k = next_unit(0);
        if (k * G < p.units) load_q(0);
        for (; k * G < p.units;) {
            const int u = unit_at(k, c, G);
            const Work w = work_of(p, u);
            const int hq = p.head_off + w.hl, b = w.b, q0 = w.q0, nt = w.nt;
            const int pos = p.q_offset + q0 + row;
            float m = -INFINITY;
            for (int j = 0; j < nt; ++j, ++T) {
                const int sb = T & 1;
                ok = __all_sync(0xffffffffu, ok && mbar_wait(&s_full[sb], (T >> 1) & 1, abort, &g_tc_attn_err));
                tc_fence_after();
                uint32_t sr[4][32];
                if (ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_ld32(lane_base + sb * 128 + 32 * q, sr[q]);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int i = 0; i < 32; ++i) sr[q][i] = 0u;
                }
                float x[128];
#pragma unroll
                for (int cc = 0; cc < 128; ++cc) x[cc] = __uint_as_float(sr[cc >> 5][cc & 31]);
                // keys that can be hidden lie only in a unit's last tiles (a warp-uniform
                // test); the masking is a pass of its own so that the maximum and the
                // exponentials stay straight runs
                const int j0 = j * BKV;
                if ((j0 + BKV > p.kv_need) || (p.causal && j0 + BKV - 1 > p.q_offset + q0)) {
                    // the row sees keys j0 .. j0 + lim - 1 of this tile
                    const int lim = min(p.kv_need, p.causal ? pos + 1 : p.kv_need) - j0;
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc) x[cc] = cc < lim ? x[cc] : -INFINITY;
                }
                // independent accumulators: the reduction is a latency chain otherwise
                float mx[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
                for (int cc = 8; cc < 128; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], x[cc]);
                const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                                 p.scale_log2;
                const float m_new = fmaxf(m, mt);
                const bool need = m_new > m + RESCALE_LOG2;   // also true on the first finite maximum
                if (__any_sync(0xffffffffu, need)) {
                    const float m_use = need ? m_new : m;
                    const float alpha = (m == -INFINITY) ? 0.f : ex2(m - m_use);
                    // O holds this unit's sum only after its first P.V; before that it is
                    // overwritten (accumulate off), so there is nothing to rescale
                    if (j > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, (T - 1) & 1, abort, &g_tc_attn_err));
                    if (j > 0 && ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int q = 0; q < 4; ++q) {
                            uint32_t o[32];
                            tmem_ld32(lane_base + T_O + 32 * q, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(lane_base + T_O + 32 * q, o);
                        }
                        const uint32_t lv = tmem_ld1(lane_base + T_L);   // the row sum, rescaled with the row
                        tmem_ld_wait();
                        tmem_st1(lane_base + T_L, __float_as_uint(__uint_as_float(lv) * alpha));
                        tmem_st_wait();
                    }
                    m = m_use;
                }
                const float nm = (m == -INFINITY) ? 0.f : -m;
                // P over the S columns it came from, 32 keys (16 columns) at a time
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_f16(ex2(fmaf(x[32 * q + 2 * i], p.scale_log2, nm)),
                                         ex2(fmaf(x[32 * q + 2 * i + 1], p.scale_log2, nm)));
                    if (ok) tmem_st16(lane_base + sb * 128 + 16 * q, pk);
                }
                if (ok) tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
            }
            const int k_next = next_unit(k + 1);
            if (k_next * G < p.units) load_q(n + 1);
            // ---- epilogue: the row sum is O's column 128; the row's 128 outputs in bf16
            if (nt > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(o_final, n & 1, abort, &g_tc_attn_err));
            tc_fence_after();
            const int qi = q0 + row;
            uint32_t o[4][32];
            float l = 0.f;
            if (nt > 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld32(lane_base + T_O + 32 * q, o[q]);
                const uint32_t lv = tmem_ld1(lane_base + T_L);
                tmem_ld_wait();
                l = __uint_as_float(lv);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[q][i] = 0u;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);   // the next unit's P.V_0 may overwrite O
            if (ok && qi < p.s_q) {
                // the row's 256 bytes in 32-byte stores (16-byte ones when the rows are not
                // 32-byte aligned)
                uint32_t *dst = (uint32_t *)(p.out + b * p.out_b + (long)qi * p.out_i + (long)hq * p.out_h);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t wv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        wv[i] = pack_bf16(__uint_as_float(o[q][2 * i]) * inv, __uint_as_float(o[q][2 * i + 1]) * inv);
                    if (p.out_v8) {
                        st_global_v8(dst + 16 * q, wv);
                        st_global_v8(dst + 16 * q + 8, wv + 8);
                    } else {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            ((uint4 *)(dst + 16 * q))[v] = make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                    }
                }
                p.lse[b * p.lse_b + (long)hq * p.lse_h + qi] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            ++n;
            k = k_next;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

bool tc_explicit_supported(int Dk, int Dn, int Dr, int Dv) {
    return prep_tc_supported(Dk, Dr) && Dn == 128 && Dv == 128;
}

// The per-head K / V reconstruction of one head shard (heads h0 .. h0 + nh of the call),
// both products in one persistent launch:
//   K_nope[b][j][hl*Dn + d] = chat[b][j] . W_K(head_begin+h0+hl)[d]
//   V^T[b][hl*Dv + d][j]    = W_V(head_begin+h0+hl)[d] . chat[b][j]
// w16: fp16 copy of the call's W_kv_b rows [head_count][Dn+Dv][Dk].
cudaError_t tc_reconstruct(const TcPrefill &p, int h0, int nh, const void *chat, const void *w16, void *kws,
                           void *vws, cudaStream_t st) {
    const long kv_pad = (p.kv_need + 127) / 128 * 128;
    const long Dh = p.Dn + p.Dv;
    TmaOperand latent{chat, p.Dk, kv_pad, p.B, (long)p.Dk * 2, kv_pad * p.Dk * 2, (int)kv_pad, 0, 1};
    const char *ws = (const char *)w16 + (long)h0 * Dh * p.Dk * 2;
    TmaOperand wk{ws, p.Dk, p.Dn, nh, (long)p.Dk * 2, Dh * p.Dk * 2, p.Dn, 0, 0};
    TmaOperand wv{ws + (long)p.Dn * p.Dk * 2, p.Dk, p.Dv, nh, (long)p.Dk * 2, Dh * p.Dk * 2, p.Dv, 0, 0};
    const GemmProblem kv[2] = {
        {latent, wk, (int)kv_pad, nh * p.Dn, p.Dk, p.B, kws, (long)p.hs * p.Dn, 1, kv_pad * p.hs * p.Dn, 0},
        {wv, latent, nh * p.Dv, (int)kv_pad, p.Dk, p.B, vws, kv_pad, 1, (long)p.hs * p.Dv * kv_pad, 0}};
    return tc_gemm_group(kv, 2, true, st);
}

cudaError_t tc_explicit_prefill(const TcPrefill &p, const void *q_nope, const void *w_kv_b, void *out, float *lse,
                                const void *chat, const void *kpe, const void *qpe, void *kws, void *vws,
                                const void *w16, cudaStream_t st) {
    (void)w_kv_b;   // read through its fp16 copy w16
    const long kv_pad = (p.kv_need + 127) / 128 * 128;
    cudaError_t e;
    // maps that do not change across shards
    CUtensorMap mQn, mQr, mKr;
    {
        unsigned long long d[4] = {(unsigned long long)p.Dn, (unsigned long long)p.head_count,
                                   (unsigned long long)p.s_q, (unsigned long long)p.B};
        unsigned long long s[3] = {(unsigned long long)p.Dn * 2, (unsigned long long)p.head_count * p.Dn * 2,
                                   (unsigned long long)p.s_q * p.head_count * p.Dn * 2};
        unsigned box[4] = {64, 1, 128, 1};
        if ((e = make_tma_map(&mQn, q_nope, 4, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[4] = {(unsigned long long)p.Dr, (unsigned long long)p.head_count,
                                   (unsigned long long)p.s_q, (unsigned long long)p.B};
        unsigned long long s[3] = {(unsigned long long)p.Dr * 2, (unsigned long long)p.head_count * p.Dr * 2,
                                   (unsigned long long)p.s_q * p.head_count * p.Dr * 2};
        unsigned box[4] = {64, 1, 128, 1};
        if ((e = make_tma_map(&mQr, qpe, 4, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {(unsigned long long)p.Dr, (unsigned long long)kv_pad, (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)p.Dr * 2, (unsigned long long)kv_pad * p.Dr * 2};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mKr, kpe, 3, d, s, box)) != cudaSuccess) return e;
    }
    CUtensorMap mK, mV;
    {
        unsigned long long d[3] = {(unsigned long long)p.hs * p.Dn, (unsigned long long)kv_pad,
                                   (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)p.hs * p.Dn * 2, (unsigned long long)kv_pad * p.hs * p.Dn * 2};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mK, kws, 3, d, s, box)) != cudaSuccess) return e;
    }
    {
        unsigned long long d[3] = {(unsigned long long)kv_pad, (unsigned long long)p.hs * p.Dv,
                                   (unsigned long long)p.B};
        unsigned long long s[2] = {(unsigned long long)kv_pad * 2, (unsigned long long)p.hs * p.Dv * kv_pad * 2};
        unsigned box[3] = {64, 128, 1};
        if ((e = make_tma_map(&mV, vws, 3, d, s, box)) != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(tc_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, n_sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;

    AttnK a;
    a.s_q = p.s_q;
    a.kv_need = (int)p.kv_need;
    a.q_offset = p.q_offset;
    a.causal = p.causal;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.out = (__nv_bfloat16 *)out;
    a.out_b = (long)p.s_q * p.head_count * p.Dv;
    a.out_i = (long)p.head_count * p.Dv;
    a.out_h = p.Dv;
    a.out_v8 = ((uintptr_t)out % 32) == 0;
    a.lse = lse;
    a.lse_b = (long)p.head_count * p.s_q;
    a.lse_h = p.s_q;
    a.idesc_s = idesc_f16(128, 128, true);
    a.idesc_pv = idesc_f16(128, 144, true);   // 128 dv columns + the row-sum column block

    for (int s = 0; s < p.n_shards; ++s) {
        const int h0 = s * p.hs;
        const int nh = std::min(p.hs, p.head_count - h0);
        if ((e = tc_reconstruct(p, h0, nh, chat, w16, kws, vws, st)) != cudaSuccess) return e;
        a.head_off = h0;
        a.nh = nh;
        a.nb = p.B;
        a.n_qt = (p.s_q + BQ - 1) / BQ;
        a.units = nh * p.B * a.n_qt;
        // persistent: one CTA per SM walks the units
        dim3 grid(std::min(a.units, n_sms)), block(32 * (NSM + 4));
        {
            ProfScope ps("tc_attn", st);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = grid;
            cfg.blockDim = block;
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the GEMM's tail
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, tc_attn_kernel, mQn, mQr, mK, mKr, mV, a);
        }
        if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t tc_attn_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_attn_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_attn_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

}  // namespace mla

