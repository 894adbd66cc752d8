// tc_gemm.cu -- batched "TN" GEMM on the sm_103a tensor cores:
//   C[z](m, n) = sum_k A[z](m, k) * B[z](n, k)      (fp16 or bf16 in, fp32 accumulate)
// A and B are K-major (k contiguous) and reached through 3-D TMA maps (k, row, z);
// C is written with arbitrary element strides as fp16, bf16 or fp32.
//
// This carries the K_nope / V reconstruction of the explicit path -- LAGA's local
// up-projection of the gathered latent at head-shard granularity ("A Training-Memory
// Regression in MLA Sequence Parallelism ... LAGA", arXiv 2607.17644, "What carries
// the argument"; the paper's section 3.3 "H_r slice of W_kv_b(latent)") -- and the
// absorb / un-absorb products of the absorbed form and of decode (same page, Fig. 2).
//
// One CTA computes one 128 x BN tile.  Warp 0 lane 0 streams 64-wide k-blocks of A
// and B through a 4-stage TMA ring; warp 1 lane 0 issues tcgen05.mma (M=128, N=BN,
// K=16 per instruction) into a TMEM accumulator; then all four warps drain TMEM
// (thread = row) and store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mla_internal.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {

__device__ unsigned g_tc_gemm_err = 0;

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4;

struct GemmK {
    int M, N, K;
    int a_rows_per_z, a_zbase, a_z_per_batch;
    int b_rows_per_z, b_zbase, b_z_per_batch;
    void *C;
    long c_m, c_n, c_batch;
    int out_kind;  // 0 fp16, 1 bf16, 2 fp32
    uint32_t idesc;
};

template <int BN>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, GemmK p) {
    using namespace tc;
    constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
    constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = (uint64_t *)(sB + STAGES * B_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *accb = empty + STAGES;
    uint32_t *tslot = (uint32_t *)(accb + 1);
    volatile int *abort = (volatile int *)(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM, batch = blockIdx.z;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accb, 1);
        *abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&ta);
        tma_prefetch_desc(&tb);
    }
    if (warp == 1) {
        tmem_alloc(tslot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int nk = p.K / BK;

    if (warp == 0 && lane == 0) {
        const int a_r = m0 % p.a_rows_per_z, a_z = p.a_zbase + m0 / p.a_rows_per_z + batch * p.a_z_per_batch;
        const int b_r = n0 % p.b_rows_per_z, b_z = p.b_zbase + n0 / p.b_rows_per_z + batch * p.b_z_per_batch;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % STAGES;
            if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1, abort, &g_tc_gemm_err)) break;
            mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
            tma_load_3d(sA + s * A_BYTES, &ta, &full[s], kb * BK, a_r, a_z);
            tma_load_3d(sB + s * B_BYTES, &tb, &full[s], kb * BK, b_r, b_z);
        }
    } else if (warp == 1 && lane == 0) {
        bool ok = true;
        for (int kb = 0; kb < nk && ok; ++kb) {
            const int s = kb % STAGES;
            if (!mbar_wait(&full[s], (kb / STAGES) & 1, abort, &g_tc_gemm_err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t da = sdesc_kmajor(sA + s * A_BYTES), db = sdesc_kmajor(sB + s * B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
                mma_ss(tmem, da + 2 * k, db + 2 * k, p.idesc, (kb | k) != 0);
            mma_commit(&empty[s]);
        }
        mma_commit(accb);
    }
    __syncwarp();

    // ---- epilogue: thread = row, 32 columns per TMEM load
    const bool ok = mbar_wait(accb, 0, abort, &g_tc_gemm_err);
    tc_fence_after();
    const long row = m0 + warp * 32 + lane;
    if (ok) {
        char *C = (char *)p.C;
        const int esz = p.out_kind == 2 ? 4 : 2;
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
            tmem_ld_wait();
            const int nb = n0 + c * 32;
            if (row >= p.M || nb >= p.N) continue;
            const long base = p.c_batch * batch + row * p.c_m;
            if (p.c_n == 1 && nb + 32 <= p.N) {
                if (esz == 2) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0 = __uint_as_float(r[2 * i]), x1 = __uint_as_float(r[2 * i + 1]);
                        w[i] = p.out_kind == 0 ? pack_f16(x0, x1) : pack_bf16(x0, x1);
                    }
                    uint4 *dst = (uint4 *)(C + (base + nb) * 2);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                } else {
                    uint4 *dst = (uint4 *)(C + (base + nb) * 4);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
                }
            } else {
                for (int i = 0; i < 32; ++i) {
                    const int n = nb + i;
                    if (n >= p.N) break;
                    const float x = __uint_as_float(r[i]);
                    const long off = base + (long)n * p.c_n;
                    if (p.out_kind == 0) ((__half *)C)[off] = __float2half_rn(x);
                    else if (p.out_kind == 1) ((__nv_bfloat16 *)C)[off] = __float2bfloat16_rn(x);
                    else ((float *)C)[off] = x;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int BN>
size_t gemm_smem() {
    return STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 256;
}

}  // namespace

cudaError_t tc_gemm(const TmaOperand &A, const TmaOperand &B, int M, int N, int K, int batch, bool f16,
                    void *C, long c_m, long c_n, long c_batch, int out_kind, cudaStream_t st) {
    if (M == 0 || N == 0 || batch == 0) return cudaSuccess;
    if (K % BK) return cudaErrorInvalidValue;
    const int BN = N >= 256 ? 256 : (N >= 128 ? 128 : 64);
    CUtensorMap ma, mb;
    cudaError_t e = make_operand_map(&ma, A, BM);
    if (e != cudaSuccess) return e;
    e = make_operand_map(&mb, B, BN);
    if (e != cudaSuccess) return e;
    GemmK p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.a_rows_per_z = A.rows_per_z;
    p.a_zbase = A.zbase;
    p.a_z_per_batch = A.z_per_batch;
    p.b_rows_per_z = B.rows_per_z;
    p.b_zbase = B.zbase;
    p.b_z_per_batch = B.z_per_batch;
    p.C = C;
    p.c_m = c_m;
    p.c_n = c_n;
    p.c_batch = c_batch;
    p.out_kind = out_kind;
    p.idesc = tc::idesc_f16(BM, BN, f16);
    dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM, batch), block(128);
    ProfScope ps("tc_gemm", st);
    switch (BN) {
        case 256: {
            size_t sm = gemm_smem<256>();
            e = cudaFuncSetAttribute(tc_gemm_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e == cudaSuccess) tc_gemm_kernel<256><<<grid, block, sm, st>>>(ma, mb, p);
            break;
        }
        case 128: {
            size_t sm = gemm_smem<128>();
            e = cudaFuncSetAttribute(tc_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e == cudaSuccess) tc_gemm_kernel<128><<<grid, block, sm, st>>>(ma, mb, p);
            break;
        }
        default: {
            size_t sm = gemm_smem<64>();
            e = cudaFuncSetAttribute(tc_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e == cudaSuccess) tc_gemm_kernel<64><<<grid, block, sm, st>>>(ma, mb, p);
        }
    }
    if (e != cudaSuccess) return e;
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
