// tc_internal.h -- host-side helpers shared by the tensor-core translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

// A K-major 16-bit operand reached through a 3-D TMA map (k, row, z).  A tile of
// `tile` GEMM rows starting at r0 is loaded from (row = r0 % rows_per_z,
// z = zbase + r0 / rows_per_z + batch * z_per_batch); when rows_per_z < tile one
// box spans tile / rows_per_z consecutive z-slices.
struct TmaOperand {
    const void *ptr;
    long k_extent;    // elements along k (contiguous)
    long rows;        // rows of one z-slice present in memory
    long z_extent;    // z-slices present in memory
    long row_stride;  // bytes between rows
    long z_stride;    // bytes between z-slices
    int rows_per_z;
    int zbase;
    int z_per_batch;
};

// Encodes a tiled TMA map for 16-bit elements with 128-byte swizzle and a box of
// {64, ...}.  rank <= 5; strides in bytes for dims 1..rank-1.
cudaError_t make_tma_map(CUtensorMap *map, const void *ptr, int rank, const unsigned long long *dims,
                         const unsigned long long *strides, const unsigned *box);
cudaError_t make_operand_map(CUtensorMap *map, const TmaOperand &op, int tile_rows);
// An m-major operand (m contiguous): boxes of 64 m x 64 k of one z-slice.
cudaError_t make_operand_map_mn(CUtensorMap *map, const TmaOperand &op);

// C[batch](m, n) = sum_k A(m, k) B(n, k); K % 64 == 0.  out_kind: 0 fp16, 1 bf16, 2 fp32.
struct GemmProblem {
    TmaOperand A, B;
    int M, N, K, batch;
    void *C;
    long c_m, c_n, c_batch;
    int out_kind;
    // A stored m-major (m contiguous, one row per k): then A.k_extent is the m extent and
    // A.rows the k extent.  Tiles of 64 or 128 columns only (not the pair kernel).
    bool a_mn = false;
    // C += A B^T instead of C = A B^T (fp32 C, tiles of 64 or 128 columns only).
    bool accumulate = false;
};
cudaError_t tc_gemm(const TmaOperand &A, const TmaOperand &B, int M, int N, int K, int batch, bool f16,
                    void *C, long c_m, long c_n, long c_batch, int out_kind, cudaStream_t st, bool a_mn = false,
                    bool accumulate = false);
// One persistent launch over the tiles of one or two problems (same K, same operand
// type): the explicit path's K_nope and V^T products share one launch.
cudaError_t tc_gemm_group(const GemmProblem *probs, int n_probs, bool f16, cudaStream_t st);

cudaError_t tc_gemm_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t tc_attn_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t tc_latent_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t tc_decode_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t tc_fused_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t tc_bwd_read_and_clear_error(unsigned *flags, cudaStream_t st);
cudaError_t simt_read_and_clear_error(unsigned *flags, cudaStream_t st);   // the row kernels' bounded waits

// Split-KV latent decode attention (tc_decode.cu): partial latent outputs and
// log-sum-exps of every (sequence, key split, 128 heads).  qa: q_abs [B][H][512] fp16;
// qp: rotated q_pe [B][H][64] fp16; cache [B][L][512], kpe [B][L][64] bf16;
// po [n_splits][B][H][512] fp32 (po16: fp16), pl [n_splits][B][H] fp32.  H % 128 == 0.
// shard_rows > 0 (TPLA, two latent shards): the rows are [B][2][shard_rows] with
// shard_rows % 128 == 0, rows of shard i attend over latent dims [256 i, 256 i + 256)
// and the RoPE band only, and only those dims of their partial output are written.
cudaError_t launch_decode_attn(const void *qa, const void *qp, const void *cache, const void *kpe, int B, long L,
                               int H, int n_splits, long chunk, float scale, float *po, float *pl, cudaStream_t st,
                               int shard_rows = 0, bool po16 = false);

}  // namespace mla
