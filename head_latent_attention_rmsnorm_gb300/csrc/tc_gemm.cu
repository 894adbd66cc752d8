// tc_gemm.cu -- batched "TN" GEMM on the sm_103a tensor cores:
//   C[z](m, n) = sum_k A[z](m, k) * B[z](n, k)      (fp16 or bf16 in, fp32 accumulate)
// A and B are K-major (k contiguous) and reached through 3-D TMA maps (k, row, z); A
// may instead be m-major (m contiguous, one row per k: the decode absorb reads W_K in
// place that way);
// C is written with arbitrary element strides as fp16, bf16 or fp32.
//
// This carries the K_nope / V reconstruction of the explicit path -- LAGA's local
// up-projection of the gathered latent at head-shard granularity ("A Training-Memory
// Regression in MLA Sequence Parallelism ... LAGA", arXiv 2607.17644, "What carries
// the argument"; the paper's section 3.3 "H_r slice of W_kv_b(latent)") -- and the
// absorb / un-absorb products of the absorbed form and of decode (same page, Fig. 2).
//
// Persistent kernel: one CTA per SM walks the 128 x BN output tiles of one or two
// problems (tile t, t + gridDim.x, ...); 256-wide problems use the pair kernel below
// (two SMs per 256 x 256 tile).  Warp 0 lane 0 streams 64-wide k-blocks of
// A and B through a 4-stage TMA ring that runs across tile boundaries; the MMA
// issuer (warp 1, a warp-uniform loop issuing from one elected lane) accumulates each
// tile into one of two TMEM accumulators (M=128, K=16 per instruction); warps 2-5 drain
// a finished accumulator (thread = row) and store it while the next tile accumulates
// into the other one.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_gemm_err = 0;

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4;

struct GemmP {
    int M, N, K;
    int a_rows_per_z, a_zbase, a_z_per_batch;
    int b_rows_per_z, b_zbase, b_z_per_batch;
    void *C;
    long c_m, c_n, c_batch;
    int out_kind;  // 0 fp16, 1 bf16, 2 fp32
    int tiles_n, tiles_m, tiles;
    int c_stage;   // pair kernel: C staged per warp and written in whole 128-byte rows (16-bit, n contiguous, aligned)
    int acc;       // fp32 C accumulated (single-CTA kernel)
};

struct GemmK {
    GemmP pr[2];
    int total;         // tiles of both problems
    uint32_t idesc;    // M = 128, N = BN (the pair kernel: M = 256, N = 128 per issuing warp)
    int a_mn;          // A stored m-major (both problems): two 64-row boxes per stage
};

struct Tile {
    int prob, m0, n0, batch;
};

__device__ __forceinline__ Tile tile_of(const GemmK &p, int t) {
    Tile r;
    r.prob = t < p.pr[0].tiles ? 0 : 1;
    const GemmP &q = p.pr[r.prob];
    int u = r.prob ? t - p.pr[0].tiles : t;
    r.n0 = (u % q.tiles_n);
    u /= q.tiles_n;
    r.m0 = (u % q.tiles_m) * BM;
    r.batch = u / q.tiles_m;
    return r;
}

template <int BN>
__global__ void __launch_bounds__(256, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                   const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1, GemmK p) {
    using namespace tc;
    constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    constexpr uint32_t ACC_COLS = BN < 32 ? 32 : BN;   // one accumulator; two are allocated
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = (uint64_t *)(sB + STAGES * B_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES, *acc_empty = acc_full + 2;
    uint32_t *tslot = (uint32_t *)(acc_empty + 2);
    volatile int *abort = (volatile int *)(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);   // the four epilogue warps
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 2 * ACC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the prologue above overlaps the previous kernel; its outputs are read below
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&ta0);
            tma_prefetch_desc(&tb0);
            if (p.pr[1].tiles) {
                tma_prefetch_desc(&ta1);
                tma_prefetch_desc(&tb1);
            }
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.total && ok; t += gridDim.x) {
                const Tile w = tile_of(p, t);
                const GemmP &q = p.pr[w.prob];
                const CUtensorMap *ma = w.prob ? &ta1 : &ta0, *mb = w.prob ? &tb1 : &tb0;
                const int n0 = w.n0 * BN;
                const int a_r = w.m0 % q.a_rows_per_z, a_z = q.a_zbase + w.m0 / q.a_rows_per_z + w.batch * q.a_z_per_batch;
                const int b_r = n0 % q.b_rows_per_z, b_z = q.b_zbase + n0 / q.b_rows_per_z + w.batch * q.b_z_per_batch;
                for (int kb = 0; kb < q.K / BK; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= STAGES && !mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, abort, &g_tc_gemm_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
                    if (p.a_mn) {   // 64 m x 64 k boxes: m-major (k rows of 128 bytes)
                        tma_load_3d(sA + s * A_BYTES, ma, &full[s], a_r, kb * BK, a_z);
                        tma_load_3d(sA + s * A_BYTES + A_BYTES / 2, ma, &full[s], a_r + 64, kb * BK, a_z);
                    } else {
                        tma_load_3d(sA + s * A_BYTES, ma, &full[s], kb * BK, a_r, a_z);
                    }
                    tma_load_3d(sB + s * B_BYTES, mb, &full[s], kb * BK, b_r, b_z);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // (warp-uniform loop; one elected lane issues)
        {
            int it = 0, lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.total && ok; t += gridDim.x, ++lt) {
                const Tile w = tile_of(p, t);
                const int a = lt & 1;
                // the epilogue has drained what tile lt-2 left in accumulator a
                if (lt >= 2 && !__all_sync(0xffffffffu, mbar_wait(&acc_empty[a], ((lt >> 1) - 1) & 1, abort, &g_tc_gemm_err)))
                    break;
                const uint32_t d = tmem + a * ACC_COLS;
                const int nk = p.pr[w.prob].K / BK;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / STAGES) & 1, abort, &g_tc_gemm_err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // A k-major: 16 k = 32 bytes along a row; m-major: 16 k = 16 rows of 128 bytes
                    // (the two 64-m boxes 8 KB apart)
                    const uint64_t da = p.a_mn ? sdesc_mnmajor(sA + s * A_BYTES, A_BYTES / 2) : sdesc_kmajor(sA + s * A_BYTES);
                    const uint32_t dk = p.a_mn ? (2048 >> 4) : 2;
                    const uint64_t db = sdesc_kmajor(sB + s * B_BYTES);
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_ss(d, da + (uint64_t)(dk * k), db + 2 * k, p.idesc, (kb | k) != 0);
                        mma_commit(&empty[s]);
                    }
                    __syncwarp();
                }
                if (elect_one()) mma_commit(&acc_full[a]);
                __syncwarp();
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------ epilogue: thread = row
        const int quad = warp & 3;
        int lt = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.total; t += gridDim.x, ++lt) {
            const Tile w = tile_of(p, t);
            const GemmP &q = p.pr[w.prob];
            const int a = lt & 1;
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[a], (lt >> 1) & 1, abort, &g_tc_gemm_err));
            tc_fence_after();
            const long row = w.m0 + quad * 32 + lane;
            const int n0 = w.n0 * BN;
            char *C = (char *)q.C;
            const int esz = q.out_kind == 2 ? 4 : 2;
            for (int c = 0; c < BN / 32 && ok; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + a * ACC_COLS + c * 32, r);
                tmem_ld_wait();
                const int nb = n0 + c * 32;
                if (row >= q.M || nb >= q.N) continue;
                const long base = q.c_batch * w.batch + row * q.c_m;
                if (q.c_n == 1 && nb + 32 <= q.N) {
                    if (esz == 2) {
                        uint32_t o[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float x0 = __uint_as_float(r[2 * i]), x1 = __uint_as_float(r[2 * i + 1]);
                            o[i] = q.out_kind == 0 ? pack_f16(x0, x1) : pack_bf16(x0, x1);
                        }
                        uint4 *dst = (uint4 *)(C + (base + nb) * 2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    } else {
                        float4 *dst = (float4 *)(C + (base + nb) * 4);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float4 v = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                            if (q.acc) {
                                const float4 o = dst[i];
                                v.x += o.x, v.y += o.y, v.z += o.z, v.w += o.w;
                            }
                            dst[i] = v;
                        }
                    }
                } else {
                    for (int i = 0; i < 32; ++i) {
                        const int n = nb + i;
                        if (n >= q.N) break;
                        const float x = __uint_as_float(r[i]);
                        const long off = base + (long)n * q.c_n;
                        if (q.out_kind == 0) ((__half *)C)[off] = __float2half_rn(x);
                        else if (q.out_kind == 1) ((__nv_bfloat16 *)C)[off] = __float2bfloat16_rn(x);
                        else ((float *)C)[off] = q.acc ? ((float *)C)[off] + x : x;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * ACC_COLS);
}

// ---------------------------------------------------------------- pair kernel ----
// The same GEMM on 256 x 256 tiles computed by a cluster of two CTAs (two SMs) with
// cta_group::2 MMAs (M = 256, N = 256): CTA r holds A rows [m0 + 128 r, +128) and B rows
// (output columns) [n0 + 128 r, +128), so every MMA reads half of its operand bytes from
// each SM.  Per CTA and tile the TMA writes 256 KB of operands into shared memory, the
// N = 256 MMAs read A and B once (256 KB; the earlier N = 128 form from two issuers read A
// twice) and the epilogue stages 64 KB in and out.  Measured, that traffic does not pace
// the kernel: halving the A reads, a sixth stage and multicast operand loads left the
// ~2.9 us per tile unchanged (about 0.92 of the tensor pipe's per-SM rate).  The leader
// (rank 0) issues the MMAs from one warp; both CTAs load, and
// both drain their own accumulator rows: 16-bit outputs through a per-warp shared-memory
// staging of the whole tile slice (accumulator released before the stores), written in
// whole 128-byte rows.
constexpr int PST = 5;   // stages of the pair kernel's ring
constexpr uint32_t PA_BYTES = 128 * BK * 2, PB_BYTES = 128 * BK * 2;
constexpr uint32_t PC_BYTES = 4 * 4 * 4096;   // four epilogue warps x a 32-row x 256-column 16-bit tile slice

__device__ __forceinline__ Tile pair_tile_of(const GemmK &p, int t) {
    Tile r;
    r.prob = t < p.pr[0].tiles ? 0 : 1;
    const GemmP &q = p.pr[r.prob];
    int u = r.prob ? t - p.pr[0].tiles : t;
    r.n0 = (u % q.tiles_n) * 256;
    u /= q.tiles_n;
    r.m0 = (u % q.tiles_m) * 256;
    r.batch = u / q.tiles_m;
    return r;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                        const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1, GemmK p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + PST * PA_BYTES;
    uint8_t *sC = sB + PST * PB_BYTES;                    // epilogue staging: two 4 KB buffers per warp
    uint64_t *full = (uint64_t *)(sC + PC_BYTES);         // leader: both CTAs' bytes of a stage landed
    uint64_t *empty = full + PST;                         // both: the stage's MMAs are done
    uint64_t *acc_full = empty + PST, *acc_empty = acc_full + 2;
    uint32_t *tslot = (uint32_t *)(acc_empty + 2);
    volatile int *abort = (volatile int *)(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;

    if (tid == 0) {
        for (int s = 0; s < PST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);   // the issuer's commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 8);   // the epilogue warps of both CTAs
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tslot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&ta0);
            tma_prefetch_desc(&tb0);
            if (p.pr[1].tiles) {
                tma_prefetch_desc(&ta1);
                tma_prefetch_desc(&tb1);
            }
            const uint32_t full0 = map_peer(smem_u32(full), 0);   // the leader's barriers
            int it = 0;
            bool ok = true;
            for (int t = pair; t < p.total && ok; t += pairs) {
                const Tile w = pair_tile_of(p, t);
                const GemmP &q = p.pr[w.prob];
                const CUtensorMap *ma = w.prob ? &ta1 : &ta0, *mb = w.prob ? &tb1 : &tb0;
                const int ar = w.m0 + 128 * (int)rank;
                const int a_r = ar % q.a_rows_per_z, a_z = q.a_zbase + ar / q.a_rows_per_z + w.batch * q.a_z_per_batch;
                const int br = w.n0 + 128 * (int)rank;
                const int b_r = br % q.b_rows_per_z, b_z = q.b_zbase + br / q.b_rows_per_z + w.batch * q.b_z_per_batch;
                for (int kb = 0; kb < q.K / BK; ++kb, ++it) {
                    const int s = it % PST;
                    if (it >= PST && !mbar_wait(&empty[s], ((it / PST) - 1) & 1, abort, &g_tc_gemm_err)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (PA_BYTES + PB_BYTES));
                    const uint32_t bar = full0 + s * 8;
                    tma_load_3d_pair(sA + s * PA_BYTES, ma, bar, kb * BK, a_r, a_z);
                    tma_load_3d_pair(sB + s * PB_BYTES, mb, bar, kb * BK, b_r, b_z);
                }
            }
        }
    } else if (rank == 0 && warp == 1) {
        // ----------------------------------------------------- MMA issuer (leader)
        // (warp-uniform loop; one elected lane issues)
        {
            int it = 0, lt = 0;
            bool ok = true;
            for (int t = pair; t < p.total && ok; t += pairs, ++lt) {
                const Tile w = pair_tile_of(p, t);
                const int a = lt & 1;
                // both CTAs' epilogues have drained what tile lt-2 left in accumulator a
                if (lt >= 2 &&
                    !__all_sync(0xffffffffu, mbar_wait_cluster(&acc_empty[a], ((lt >> 1) - 1) & 1, abort, &g_tc_gemm_err)))
                    break;
                const uint32_t d = tmem + a * 256;
                const int nk = p.pr[w.prob].K / BK;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % PST;
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / PST) & 1, abort, &g_tc_gemm_err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = sdesc_kmajor(sA + s * PA_BYTES);
                    const uint64_t db = sdesc_kmajor(sB + s * PB_BYTES);
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) mma_ss_pair(d, da + 2 * k, db + 2 * k, p.idesc, (kb | k) != 0);
                        mma_commit_pair(&empty[s], 3);
                    }
                    __syncwarp();
                }
                if (elect_one()) mma_commit_pair(&acc_full[a], 3);
                __syncwarp();
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------ epilogue (both CTAs): thread = row
        const int quad = warp & 3;
        const uint32_t acc_empty0 = map_peer(smem_u32(acc_empty), 0);
        int lt = 0;
        bool ok = true;
        for (int t = pair; t < p.total; t += pairs, ++lt) {
            const Tile w = pair_tile_of(p, t);
            const GemmP &q = p.pr[w.prob];
            const int a = lt & 1;
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[a], (lt >> 1) & 1, abort, &g_tc_gemm_err));
            tc_fence_after();
            if (q.c_stage) {
                // The warp's 32 rows x 256 columns: TMEM -> 16-bit -> four 128-byte-swizzled
                // 32 x 64 buffers (chunk j of a row at j ^ (row mod 8)); the accumulator is
                // released as soon as it has been read, then the buffers are read back four
                // rows per instruction and stored in whole 128-byte rows.  (TMA tile stores
                // from here queued in the TMA unit behind the producer's operand loads, and
                // releasing the accumulator after the stores waited for them to land.)
                char *const C = (char *)q.C;
                const long cbase = q.c_batch * w.batch, c_m = q.c_m;
                const int row0 = w.m0 + 128 * (int)rank + quad * 32, M = q.M, N = q.N;
                const bool f16out = q.out_kind == 0;
                const uint32_t sbuf0 = smem_u32(sC + (warp - 2) * 16384);
                const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + a * 256;
                __syncwarp();   // every lane has read the previous tile's buffers
                uint32_t r[2][64];
                if (ok) {
                    tmem_ld32(tq, *reinterpret_cast<uint32_t(*)[32]>(&r[0][0]));
                    tmem_ld32(tq + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[0][32]));
                    tmem_ld_wait();
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    if (ok && cc < 3) {   // the next chunk's columns load while this one is packed
                        tmem_ld32(tq + (cc + 1) * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[(cc + 1) & 1][0]));
                        tmem_ld32(tq + (cc + 1) * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[(cc + 1) & 1][32]));
                    }
                    uint32_t o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x0 = __uint_as_float(r[cc & 1][2 * i]), x1 = __uint_as_float(r[cc & 1][2 * i + 1]);
                        o[i] = f16out ? pack_f16(x0, x1) : pack_bf16(x0, x1);
                    }
                    const uint32_t buf = sbuf0 + cc * 4096;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), o[4 * j], o[4 * j + 1], o[4 * j + 2],
                                     o[4 * j + 3]);
                    if (ok && cc < 3) tmem_ld_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_peer(acc_empty0 + a * 8);
                // 32-byte piece j of a 128-byte row per lane: eight rows per store instruction
                const int j = lane & 3;
#pragma unroll 1
                for (int cc = 0; cc < 4 && ok; ++cc) {
                    const int n = w.n0 + cc * 64;
                    if (n >= N) break;
                    const uint32_t buf = sbuf0 + cc * 4096;
                    uint32_t v[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = 8 * i + (lane >> 2);
                        const uint4 a0 = ld_shared_v4(buf + rr * 128 + (((2 * j) ^ (rr & 7)) << 4));
                        const uint4 a1 = ld_shared_v4(buf + rr * 128 + (((2 * j + 1) ^ (rr & 7)) << 4));
                        v[i][0] = a0.x, v[i][1] = a0.y, v[i][2] = a0.z, v[i][3] = a0.w;
                        v[i][4] = a1.x, v[i][5] = a1.y, v[i][6] = a1.z, v[i][7] = a1.w;
                    }
                    char *dst = C + (cbase + (long)(row0 + (lane >> 2)) * c_m + n) * 2 + j * 32;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (row0 + 8 * i + (lane >> 2) < M) st_global_v8(dst + (long)(8 * i) * c_m * 2, v[i]);
                }
                continue;
            }
            const long row = w.m0 + 128 * (long)rank + quad * 32 + lane;
            char *C = (char *)q.C;
            const int esz = q.out_kind == 2 ? 4 : 2;
            for (int c = 0; c < 8 && ok; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + a * 256 + c * 32, r);
                tmem_ld_wait();
                const int nb = w.n0 + c * 32;
                if (row >= q.M || nb >= q.N) continue;
                const long base = q.c_batch * w.batch + row * q.c_m;
                if (q.c_n == 1 && nb + 32 <= q.N) {
                    if (esz == 2) {
                        uint32_t o[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float x0 = __uint_as_float(r[2 * i]), x1 = __uint_as_float(r[2 * i + 1]);
                            o[i] = q.out_kind == 0 ? pack_f16(x0, x1) : pack_bf16(x0, x1);
                        }
                        uint4 *dst = (uint4 *)(C + (base + nb) * 2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    } else {
                        uint4 *dst = (uint4 *)(C + (base + nb) * 4);
#pragma unroll
                        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
                    }
                } else {
                    for (int i = 0; i < 32; ++i) {
                        const int n = nb + i;
                        if (n >= q.N) break;
                        const float x = __uint_as_float(r[i]);
                        const long off = base + (long)n * q.c_n;
                        if (q.out_kind == 0) ((__half *)C)[off] = __float2half_rn(x);
                        else if (q.out_kind == 1) ((__nv_bfloat16 *)C)[off] = __float2bfloat16_rn(x);
                        else ((float *)C)[off] = x;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(acc_empty0 + a * 8);   // the leader's barrier (own CTA for rank 0)
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the leader's MMAs read this CTA's shared memory until here
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

template <int BN>
size_t gemm_smem() {
    return STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 256;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

cudaError_t launch_gemm_pair(const CUtensorMap *maps, const GemmK &p, cudaStream_t st) {
    const size_t sm = PST * (PA_BYTES + PB_BYTES) + PC_BYTES + 1024 + 256;
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    const int grid = 2 * std::min(p.total, num_sms() / 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the previous kernel's tail
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel, maps[0], maps[1], maps[2], maps[3], p);
}

template <int BN>
cudaError_t launch_gemm(const CUtensorMap *maps, const GemmK &p, cudaStream_t st) {
    const size_t sm = gemm_smem<BN>();
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    // 64-wide tiles need 97 KB of shared memory and 128 TMEM columns: two CTAs per SM
    const int grid = std::min(p.total, num_sms() * (BN == 64 ? 2 : 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the previous kernel's tail
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN>, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace

cudaError_t tc_gemm_group(const GemmProblem *probs, int n_probs, bool f16, cudaStream_t st) {
    if (n_probs < 1 || n_probs > 2) return cudaErrorInvalidValue;
    int maxN = 0;
    for (int i = 0; i < n_probs; ++i) {
        if (probs[i].K % BK || probs[i].K != probs[0].K || probs[i].a_mn != probs[0].a_mn) return cudaErrorInvalidValue;
        if (probs[i].accumulate && probs[i].out_kind != 2) return cudaErrorInvalidValue;
        maxN = std::max(maxN, probs[i].N);
    }
    int BN = maxN >= 256 ? 256 : (maxN >= 128 ? 128 : 64);
    if (probs[0].a_mn && BN == 256) return cudaErrorInvalidValue;   // m-major A: single-CTA tiles only
    // 256-wide problems run on SM pairs: 256 x 256 tiles, A and B boxes of 128 rows per
    // CTA (a B box must not straddle two z blocks of the operand: otherwise 128-wide
    // single-CTA tiles)
    bool pair = BN == 256;
    for (int i = 0; i < n_probs; ++i) {
        if (pair && probs[i].accumulate) return cudaErrorInvalidValue;   // accumulation: single-CTA tiles only
        if (probs[i].B.rows_per_z % 128 != 0) pair = false;
    }
    if (BN == 256 && !pair) BN = 128;
    const int TM = pair ? 256 : BM, TN = BN;
    CUtensorMap maps[4];
    GemmK p{};
    p.total = 0;
    for (int i = 0; i < 2; ++i) {
        GemmP &q = p.pr[i];
        if (i >= n_probs) {
            q.tiles = 0;
            maps[2 * i] = maps[0];
            maps[2 * i + 1] = maps[1];
            continue;
        }
        const GemmProblem &g = probs[i];
        cudaError_t e = g.a_mn ? make_operand_map_mn(&maps[2 * i], g.A) : make_operand_map(&maps[2 * i], g.A, BM);
        if (e != cudaSuccess) return e;
        e = make_operand_map(&maps[2 * i + 1], g.B, pair ? 128 : BN);
        if (e != cudaSuccess) return e;
        q.M = g.M;
        q.N = g.N;
        q.K = g.K;
        q.a_rows_per_z = g.A.rows_per_z;
        q.a_zbase = g.A.zbase;
        q.a_z_per_batch = g.A.z_per_batch;
        q.b_rows_per_z = g.B.rows_per_z;
        q.b_zbase = g.B.zbase;
        q.b_z_per_batch = g.B.z_per_batch;
        q.C = g.C;
        q.c_m = g.c_m;
        q.c_n = g.c_n;
        q.c_batch = g.c_batch;
        q.out_kind = g.out_kind;
        q.acc = g.accumulate ? 1 : 0;
        q.tiles_n = (g.N + TN - 1) / TN;
        q.tiles_m = (g.M + TM - 1) / TM;
        q.tiles = (g.M == 0 || g.N == 0) ? 0 : q.tiles_n * q.tiles_m * g.batch;
        p.total += q.tiles;
        // the pair kernel writes 16-bit, n-contiguous outputs with 32-byte aligned rows in
        // whole 128-byte row pieces (columns in whole 64-column chunks)
        q.c_stage = pair && g.out_kind != 2 && g.c_n == 1 && g.N % 64 == 0 && (g.c_m * 2) % 32 == 0 &&
                    (g.batch <= 1 || (g.c_batch * 2) % 32 == 0) && ((uintptr_t)g.C % 32) == 0;
    }
    if (p.total == 0) return cudaSuccess;
    p.a_mn = probs[0].a_mn ? 1 : 0;
    ProfScope ps("tc_gemm", st);
    switch (BN) {
        case 256:
            p.idesc = tc::idesc_f16(256, 256, f16);   // cta_group::2: M = 256 across the pair
            return launch_gemm_pair(maps, p, st);
        case 128:
            p.idesc = tc::idesc_f16(BM, 128, f16, false, p.a_mn != 0);
            return launch_gemm<128>(maps, p, st);
        default:
            p.idesc = tc::idesc_f16(BM, 64, f16, false, p.a_mn != 0);
            return launch_gemm<64>(maps, p, st);
    }
}

cudaError_t tc_gemm(const TmaOperand &A, const TmaOperand &B, int M, int N, int K, int batch, bool f16,
                    void *C, long c_m, long c_n, long c_batch, int out_kind, cudaStream_t st, bool a_mn,
                    bool accumulate) {
    if (M == 0 || N == 0 || batch == 0) return cudaSuccess;
    GemmProblem g{A, B, M, N, K, batch, C, c_m, c_n, c_batch, out_kind, a_mn, accumulate};
    return tc_gemm_group(&g, 1, f16, st);
}

namespace {
// A wait that nothing ends: one thread waits on a fresh mbarrier (phase 0, which no
// thread ever arrives at) with the library's bounded wait and a short limit.  The wait
// runs out, records the timeout in the same error word the GEMM kernels use, and the
// kernel returns.  No TMA, bulk copy, MMA or TMEM allocation is in flight.
__global__ void wait_probe_kernel(uint64_t limit_ns) {
    using namespace tc;
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, &abort_flag, &g_tc_gemm_err, limit_ns);
}
}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st) {
    ProfScope ps("wait_probe", st);
    wait_probe_kernel<<<1, 32, 0, st>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t tc_gemm_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_gemm_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_gemm_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

}  // namespace mla
