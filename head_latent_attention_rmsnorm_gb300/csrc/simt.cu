// simt.cu -- CUDA-core kernels of libmla: any dimensions, fp32 arithmetic, storage
// types chosen per tensor at run time (fp16, bf16 or fp32).  They carry the fp32
// dtype (which tensor cores cannot hold to a 1e-4 error), every shape the
// tensor-core kernels do not cover, and the small prep steps both paths share
// (RMSNorm of the latent, RoPE, storage conversion).
//
// Method: "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
// (arXiv 2607.17644), "What carries the argument" and Fig. 2 (explicit and absorbed
// dataflows); "TPLA: Tensor Parallel Latent Attention ..." (arXiv 2508.15881), "What
// carries the argument" (RMSNorm of the latent); "Helix Parallelism ..." (arXiv
// 2507.07120), "What carries the argument" (log-sum-exp rescale of split partials).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>

#include "mla_internal.h"
#include "tc_common.cuh"
#include "tc_internal.h"

namespace mla {
namespace {

// Element access by storage code (TY_F16, TY_BF16, TY_F32); the code is uniform
// across a launch, so the branch never diverges.
__device__ __forceinline__ float ldx(const void *p, int ty, long i) {
    if (ty == TY_F32) return ((const float *)p)[i];
    if (ty == TY_BF16) return __bfloat162float(((const __nv_bfloat16 *)p)[i]);
    return __half2float(((const __half *)p)[i]);
}
__device__ __forceinline__ void stx(void *p, int ty, long i, float v) {
    if (ty == TY_F32) ((float *)p)[i] = v;
    else if (ty == TY_BF16) ((__nv_bfloat16 *)p)[i] = __float2bfloat16_rn(v);
    else ((__half *)p)[i] = __float2half_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// cos/sin of pos * base^(-2t/Dr) for positions [pos0, pos0 + n_pos), t < Dr/2.
// The angle is formed and reduced to [-pi, pi] in double precision (positions reach
// 10^4..10^5, where a float angle would already be off by ~1e-3 rad); the reduced
// angle then goes through the float sincos.  theta_t is computed once per block.
// (cos, sin) of pos * theta: the angle reduced by the nearest multiple of 2 pi in
// double (a multiply by 1/(2 pi) picks the multiple; an off-by-one choice only leaves
// the angle just outside [-pi, pi]), then the float sincos.
__device__ __forceinline__ float2 rope_cs(long pos, double theta) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    const double a = (double)pos * theta;
    const double r = fma(-rint(a * inv_two_pi), two_pi, a);
    float s, c;
    sincosf((float)r, &s, &c);
    return make_float2(c, s);
}

// The frequencies base^(-2t/Dr), computed in double on the host (the device's fp64
// pow is a long latency chain at GB300's fp64 rate).
constexpr int ROPE_MAX_HALF = 320;   // Dr <= 640 - Dn (validated by the callers)
struct RopeTheta {
    double v[ROPE_MAX_HALF];
};

__global__ void rope_table_kernel(long pos0, long n_pos, int half, const __grid_constant__ RopeTheta th, float2 *tab) {
    long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_pos * half) return;
    tab[i] = rope_cs(pos0 + i / half, th.v[i % half]);
}

// ---------------------------------------------- fused prep (tensor-core path) ----
constexpr int PREP_DR = 64;          // RoPE width of the fused prep: one lane per frequency
constexpr int PREP_W_PER_LANE = 8;   // 16-byte weight chunks a lane converts per task

struct PrepTc {
    int B, s_kv, n_rows, pad_rows, Dk;
    long n_pos;                              // table positions [0, n_pos)
    const __nv_bfloat16 *c_kv, *k_pe, *rms_w;
    float eps;
    float2 *tab;
    __half *chat, *kpe;
    const uint4 *w_src;                      // bf16 weights, 8 per chunk
    uint4 *w_dst;                            // their fp16 copy
    long w_chunks;
    long row_tasks, tab_tasks, w_tasks;      // warps of each kind, in this order
    // q_pe rows [B][s_q][n_hq][64] at positions q_offset + i, rotated into fp16 qpe
    const __nv_bfloat16 *q_pe;
    __half *qpe;
    int s_q, q_offset, n_hq;
    double theta[PREP_DR / 2];
};

// RoPE of every q_pe row at position `pos` (one query index of every batch row b in
// [b0, b1) and every head), with lane t holding (cos, sin) of frequency t.  Eight rows
// per pass: lane l takes row l / 4 and the pairs (t, t + 32) for t in [8 (l % 4), +8),
// as two 16-byte reads and two 16-byte writes; the eight (cos, sin) it needs are the same
// for every row (one position) and are gathered once.
__device__ __forceinline__ void rope_q_at(const PrepTc &a, long pos, int b0, int b1, float2 cs, int lane) {
    const long i = pos - a.q_offset;
    if (i < 0 || i >= a.s_q) return;   // uniform across the warp
    const int ch = lane & 3, rsub = lane >> 2;
    float2 r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        r[e] = make_float2(__shfl_sync(0xffffffffu, cs.x, 8 * ch + e), __shfl_sync(0xffffffffu, cs.y, 8 * ch + e));
    const long rows = (long)(b1 - b0) * a.n_hq;
    for (long r0 = 0; r0 < rows; r0 += 8) {
        const long rr = r0 + rsub;
        if (rr >= rows) continue;
        const int b = b0 + (int)(rr / a.n_hq), h = (int)(rr % a.n_hq);
        const long base = (((long)b * a.s_q + i) * a.n_hq + h) * PREP_DR + 8 * ch;
        const uint4 xa = *(const uint4 *)(a.q_pe + base), xb = *(const uint4 *)(a.q_pe + base + 32);
        const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // elements 2k, 2k + 1 of this lane's 8
            const float a0 = __uint_as_float(wa[k] << 16), a1 = __uint_as_float(wa[k] & 0xffff0000u);
            const float c0 = __uint_as_float(wb[k] << 16), c1 = __uint_as_float(wb[k] & 0xffff0000u);
            const float2 r0 = r[2 * k], r1 = r[2 * k + 1];
            __half2 lo = __floats2half2_rn(a0 * r0.x - c0 * r0.y, a1 * r1.x - c1 * r1.y);
            __half2 hi = __floats2half2_rn(c0 * r0.x + a0 * r0.y, c1 * r1.x + a1 * r1.y);
            oa[k] = *(uint32_t *)&lo;
            ob[k] = *(uint32_t *)&hi;
        }
        *(uint4 *)(a.qpe + base) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        *(uint4 *)(a.qpe + base + 32) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
}

__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *(uint32_t *)&h;
}

// One warp per task: a latent row (b, j) of [0, B*pad_rows), a table-only position of
// [pad_rows, n_pos), or a run of 32*PREP_W_PER_LANE weight chunks.
__global__ void __launch_bounds__(256, 5) prep_tc_kernel(const __grid_constant__ PrepTc a) {
    // the reconstruction GEMM may launch now (it waits for this grid before its loads)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    long g = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (g < a.row_tasks) {
        const long b = g / a.pad_rows, j = g % a.pad_rows;
        const int Dk = a.Dk, nc = Dk / 256;
        const bool live = j < a.n_rows;
        // this row's latent and k_pe loads first: their latency overlaps the angle and the
        // q_pe rotation below
        uint4 xr[4];
        float x0 = 0.f, x1 = 0.f;
        if (live) {
            const uint4 *x = (const uint4 *)(a.c_kv + (b * a.s_kv + j) * Dk);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (c < nc) xr[c] = x[c * 32 + lane];
            const __nv_bfloat16 *kx = a.k_pe + (b * a.s_kv + j) * PREP_DR;
            x0 = __bfloat162float(kx[lane]);
            x1 = __bfloat162float(kx[lane + 32]);
        }
        const float2 cs = rope_cs(j, a.theta[lane]);
        if (b == 0 && j < a.n_pos) a.tab[j * (PREP_DR / 2) + lane] = cs;
        if (a.qpe) rope_q_at(a, j, (int)b, (int)b + 1, cs, lane);
        uint4 *y = (uint4 *)(a.chat + g * Dk);
        __half *kp = a.kpe + g * PREP_DR;
        if (!live) {
            for (int c = 0; c < nc; ++c) y[c * 32 + lane] = make_uint4(0, 0, 0, 0);
            kp[lane] = kp[lane + 32] = __float2half_rn(0.f);
            return;
        }
        const uint4 *w = (const uint4 *)a.rms_w;
        float v[4][8];
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c < nc) {
                uint4 q = xr[c];
                const __nv_bfloat16 *e = (const __nv_bfloat16 *)&q;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[c][i] = __bfloat162float(e[i]);
                    ss += v[c][i] * v[c][i];
                }
            }
        }
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)Dk + a.eps);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c < nc) {
                uint4 q = w[c * 32 + lane];
                const __nv_bfloat16 *e = (const __nv_bfloat16 *)&q;
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = f16x2(v[c][2 * i] * inv * __bfloat162float(e[2 * i]),
                                 v[c][2 * i + 1] * inv * __bfloat162float(e[2 * i + 1]));
                y[c * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        // half-split pairs (t, t + 32): lane t rotates both by its own frequency
        kp[lane] = __float2half_rn(x0 * cs.x - x1 * cs.y);
        kp[lane + 32] = __float2half_rn(x1 * cs.x + x0 * cs.y);
    } else if ((g -= a.row_tasks) < a.tab_tasks) {
        const long pos = a.pad_rows + g;
        const float2 cs = rope_cs(pos, a.theta[lane]);
        a.tab[pos * (PREP_DR / 2) + lane] = cs;
        if (a.qpe) rope_q_at(a, pos, 0, a.B, cs, lane);
    } else if ((g -= a.tab_tasks) < a.w_tasks) {
        const long c0 = g * 32 * PREP_W_PER_LANE + lane;
#pragma unroll
        for (int k = 0; k < PREP_W_PER_LANE; ++k) {
            const long c = c0 + 32 * k;
            if (c < a.w_chunks) {
                const uint4 q = a.w_src[c];
                const uint32_t in[4] = {q.x, q.y, q.z, q.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)   // bf16 -> fp32 is a shift; fp32 -> fp16 rounds
                    o[i] = f16x2(__uint_as_float(in[i] << 16), __uint_as_float(in[i] & 0xffff0000u));
                a.w_dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Rotates one Dr-wide band (half-split pairs t, t+Dr/2) with table row `cs`.
__device__ __forceinline__ void rope_band(const void *x, int tx, long xo, void *y, int ty, long yo, int Dr,
                                          const float2 *cs, int lane) {
    int half = Dr / 2;
    for (int t = lane; t < half; t += 32) {
        float2 r = cs[t];
        float x0 = ldx(x, tx, xo + t), x1 = ldx(x, tx, xo + t + half);
        stx(y, ty, yo + t, x0 * r.x - x1 * r.y);
        stx(y, ty, yo + t + half, x1 * r.x + x0 * r.y);
    }
}

// RMSNorm of c_kv rows and RoPE of k_pe rows.  Rows j in [n_rows, pad_rows) of each
// batch are written as zeros, so that padded tiles read later hold finite values.
__global__ void latent_prep_kernel(int B, int s_kv, int n_rows, int pad_rows, int Dk, int Dr, const void *c_kv,
                                   const void *k_pe, const void *rms_w, int tin, float eps, const float2 *tab,
                                   void *chat, void *kpe, int tout) {
    long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (row >= (long)B * pad_rows) return;
    long b = row / pad_rows, j = row % pad_rows;
    if (j >= n_rows) {
        for (int k = lane; k < Dk; k += 32) stx(chat, tout, row * Dk + k, 0.f);
        for (int k = lane; k < Dr; k += 32) stx(kpe, tout, row * Dr + k, 0.f);
        return;
    }
    long xo = (b * s_kv + j) * Dk;
    float ss = 0.f;
    for (int k = lane; k < Dk; k += 32) {
        float v = ldx(c_kv, tin, xo + k);
        ss += v * v;
    }
    ss = warp_sum(ss);
    float inv = 1.0f / sqrtf(ss / (float)Dk + eps);
    for (int k = lane; k < Dk; k += 32)
        stx(chat, tout, row * Dk + k, ldx(c_kv, tin, xo + k) * inv * ldx(rms_w, tin, k));
    rope_band(k_pe, tin, (b * s_kv + j) * Dr, kpe, tout, row * Dr, Dr, tab + j * (Dr / 2), lane);
}

// Same, bf16 inputs with Dk a multiple of 256: each lane moves 16-byte vectors.
template <typename TO>
__global__ void latent_prep_vec_kernel(int B, int s_kv, int n_rows, int pad_rows, int Dk, int Dr,
                                       const __nv_bfloat16 *c_kv, const __nv_bfloat16 *k_pe,
                                       const __nv_bfloat16 *rms_w, float eps, const float2 *tab, TO *chat,
                                       TO *kpe) {
    long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (row >= (long)B * pad_rows) return;
    long b = row / pad_rows, j = row % pad_rows;
    const int nc = Dk / 256;                     // 16-byte chunks per lane
    TO *y = chat + row * Dk;
    if (j >= n_rows) {
        for (int k = lane; k < Dk; k += 32) y[k] = TO(0.f);
        for (int k = lane; k < Dr; k += 32) kpe[row * Dr + k] = TO(0.f);
        return;
    }
    const uint4 *x = (const uint4 *)(c_kv + (b * s_kv + j) * Dk);
    const uint4 *w = (const uint4 *)rms_w;
    float v[4][8];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < nc) {
            uint4 q = x[c * 32 + lane];
            const __nv_bfloat16 *e = (const __nv_bfloat16 *)&q;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[c][i] = __bfloat162float(e[i]);
                ss += v[c][i] * v[c][i];
            }
        }
    }
    ss = warp_sum(ss);
    float inv = 1.0f / sqrtf(ss / (float)Dk + eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < nc) {
            uint4 q = w[c * 32 + lane];
            const __nv_bfloat16 *e = (const __nv_bfloat16 *)&q;
            TO *dst = y + (c * 32 + lane) * 8;
            if (sizeof(TO) == 2) {
                __align__(16) __half hv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) hv[i] = __float2half_rn(v[c][i] * inv * __bfloat162float(e[i]));
                *(uint4 *)dst = *(const uint4 *)hv;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = TO(v[c][i] * inv * __bfloat162float(e[i]));
            }
        }
    }
    rope_band(k_pe, TY_BF16, (b * s_kv + j) * Dr, kpe, sizeof(TO) == 4 ? TY_F32 : TY_F16, row * Dr, Dr,
              tab + j * (Dr / 2), lane);
}

__global__ void rope_rows_kernel(long rows, int Dr, const void *x, int tin, long pos0, long pos_div, long pos_mod,
                                 const float2 *tab, long tab_pos0, void *y, int tout) {
    long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (r >= rows) return;
    long pos = pos0 + (r / pos_div) % pos_mod;
    rope_band(x, tin, r * Dr, y, tout, r * Dr, Dr, tab + (pos - tab_pos0) * (Dr / 2), threadIdx.x % 32);
}

// RoPE of rows that all sit at one position (the decode query): the block computes the
// position's (cos, sin) pairs into shared memory as rope_table_kernel would, then one warp
// rotates each row.
__global__ void rope_rows_at_kernel(long rows, int Dr, const void *x, int tin, long pos,
                                    const __grid_constant__ RopeTheta th, void *y, int tout) {
    __shared__ float2 cs[ROPE_MAX_HALF];
    for (int i = threadIdx.x; i < Dr / 2; i += blockDim.x) cs[i] = rope_cs(pos, th.v[i]);
    __syncthreads();
    long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (r >= rows) return;
    rope_band(x, tin, r * Dr, y, tout, r * Dr, Dr, cs, threadIdx.x % 32);
}

__global__ void convert_kernel(const void *x, int tin, void *y, int tout, long n) {
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
        stx(y, tout, i, ldx(x, tin, i));
}

// ---------------------------------------------------------------- GEMM ----
constexpr int GT = 64, GK = 16;

__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
    __shared__ float As[GK][GT + 1], Bs[GK][GT + 1];
    int zb = blockIdx.z / g.nzh, zh = blockIdx.z % g.nzh;
    const long ao = zb * g.a_zb + zh * g.a_zh, bo = zb * g.b_zb + zh * g.b_zh, co = zb * g.c_zb + zh * g.c_zh;
    int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
    int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += GK) {
        for (int i = threadIdx.x; i < GK * GT; i += 256) {
            int kk = i / GT, mm = i % GT;
            int m = m0 + mm, n = n0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.M && k < g.K) ? ldx(g.A, g.ta, ao + m * g.a_m + k * g.a_k) : 0.f;
            Bs[kk][mm] = (n < g.N && k < g.K) ? ldx(g.B, g.tb, bo + n * g.b_n + k * g.b_k) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
            if (m < g.M && n < g.N) {
                const long o = co + m * g.c_m + n * g.c_n;
                stx(g.C, g.tc, o, g.accumulate ? ldx(g.C, g.tc, o) + acc[i][j] : acc[i][j]);
            }
        }
}

// ----------------------------------------------------------- attention ----
constexpr int AW = 8;      // warps (= query rows) per block
constexpr int AKT = 16;    // keys per shared-memory tile
constexpr int QMAX = 640;  // D1 + D2 limit (registers per lane: QMAX/32)
constexpr int VMAX = 512;  // Dv limit

__global__ void __launch_bounds__(AW * 32) attn_simt_kernel(AttnArgs a) {
    extern __shared__ float sm[];
    const int Dq = a.D1 + a.D2;
    float *sK = sm;                 // [AKT][Dq]
    float *sV = sm + AKT * Dq;      // [AKT][Dv]
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = blockIdx.y / a.n_h, h = blockIdx.y % a.n_h;
    const int split = blockIdx.z;
    const long r = (long)blockIdx.x * AW + warp;
    const bool active = r < a.n_rows;

    long kb = (long)split * a.chunk;
    long ke = kb + a.chunk < a.kv_len ? kb + a.chunk : a.kv_len;
    if (kb > a.kv_len) kb = a.kv_len;
    long r_last = (long)blockIdx.x * AW + AW - 1;
    if (r_last > a.n_rows - 1) r_last = a.n_rows - 1;
    long kend_blk = ke, kend_row = ke;
    if (a.causal) {
        long lim = a.pos0 + r_last + 1;
        kend_blk = lim < ke ? lim : ke;
        long limr = a.pos0 + r + 1;
        kend_row = limr < ke ? limr : ke;
    }

    const long q1o = b * a.q1_b + h * a.q1_h + r * a.q1_r;
    const long q2o = b * a.q2_b + h * a.q2_h + r * a.q2_r;
    float q[QMAX / 32];
#pragma unroll
    for (int t = 0; t < QMAX / 32; ++t) {
        int d = lane + 32 * t;
        float v = 0.f;
        if (active && d < a.D1) v = ldx(a.q1, a.tq1, q1o + d);
        else if (active && d < Dq) v = ldx(a.q2, a.tq2, q2o + (d - a.D1));
        q[t] = v;
    }
    float o[VMAX / 32];
#pragma unroll
    for (int t = 0; t < VMAX / 32; ++t) o[t] = 0.f;
    float m = -INFINITY, l = 0.f;

    const long k1o = b * a.k1_b + h * a.k1_h, k2o = b * a.k2_b + h * a.k2_h, vo = b * a.v_b + h * a.v_h;

    for (long k0 = kb; k0 < kend_blk; k0 += AKT) {
        __syncthreads();
        for (int i = threadIdx.x; i < AKT * Dq; i += blockDim.x) {
            int kk = i / Dq, d = i % Dq;
            long key = k0 + kk;
            float v = 0.f;
            if (key < kend_blk)
                v = d < a.D1 ? ldx(a.k1, a.tk1, k1o + key * a.k1_r + d)
                             : ldx(a.k2, a.tk2, k2o + key * a.k2_r + (d - a.D1));
            sK[i] = v;
        }
        for (int i = threadIdx.x; i < AKT * a.Dv; i += blockDim.x) {
            int kk = i / a.Dv, d = i % a.Dv;
            long key = k0 + kk;
            sV[i] = key < kend_blk ? ldx(a.v, a.tv, vo + key * a.v_r + d) : 0.f;
        }
        __syncthreads();
        if (!active) continue;
        float s[AKT];
        float mt = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < AKT; ++kk) {
            float part = 0.f;
#pragma unroll
            for (int t = 0; t < QMAX / 32; ++t) {
                int d = lane + 32 * t;
                if (d < Dq) part = fmaf(q[t], sK[kk * Dq + d], part);
            }
            part = warp_sum(part) * a.scale;
            s[kk] = (k0 + kk < kend_row) ? part : -INFINITY;
            mt = fmaxf(mt, s[kk]);
        }
        float mn = fmaxf(m, mt);
        if (mn == -INFINITY) continue;
        float alpha = expf(m - mn);   // m = -inf -> 0
        l *= alpha;
#pragma unroll
        for (int t = 0; t < VMAX / 32; ++t) o[t] *= alpha;
#pragma unroll
        for (int kk = 0; kk < AKT; ++kk) {
            float pk = expf(s[kk] - mn);
            l += pk;
#pragma unroll
            for (int t = 0; t < VMAX / 32; ++t) {
                int d = lane + 32 * t;
                if (d < a.Dv) o[t] = fmaf(pk, sV[kk * a.Dv + d], o[t]);
            }
        }
        m = mn;
    }
    if (!active) return;
    float inv = l > 0.f ? 1.f / l : 0.f;
    float lse = l > 0.f ? m + logf(l) : -INFINITY;
    if (a.part_out) {
        float *po = a.part_out + split * a.po_s + b * a.po_b + h * a.po_h + r * a.po_r;
#pragma unroll
        for (int t = 0; t < VMAX / 32; ++t) {
            int d = lane + 32 * t;
            if (d < a.Dv) po[d] = o[t] * inv;
        }
        if (lane == 0) a.part_lse[split * a.pl_s + b * a.pl_b + h * a.pl_h + r * a.pl_r] = lse;
    } else {
        const long oo = b * a.o_b + h * a.o_h + r * a.o_r;
#pragma unroll
        for (int t = 0; t < VMAX / 32; ++t) {
            int d = lane + 32 * t;
            if (d < a.Dv) stx(a.out, a.to, oo + d, o[t] * inv);
        }
        if (lane == 0) a.lse[b * a.l_b + h * a.l_h + r * a.l_r] = lse;
    }
}

// --------------------------------------------------------- lse combine ----
__global__ void lse_combine_kernel(int n, long rows, int D, const float *po, const float *pl, void *out, int to,
                                   float *lse) {
    long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (r >= rows) return;
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, pl[(long)s * rows + r]);
    m = warp_max(m);
    if (m == -INFINITY) {
        for (int d = lane; d < D; d += 32) stx(out, to, r * D + d, 0.f);
        if (lane == 0) lse[r] = -INFINITY;
        return;
    }
    float z = 0.f;
    for (int s = lane; s < n; s += 32) z += expf(pl[(long)s * rows + r] - m);
    z = warp_sum(z);
    float L = m + logf(z);
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int s = 0; s < n; ++s) {
            float w = expf(pl[(long)s * rows + r] - L);
            if (w > 0.f) acc = fmaf(w, po[((long)s * rows + r) * D + d], acc);
        }
        stx(out, to, r * D + d, acc);
    }
    if (lane == 0) lse[r] = L;
}

// The same merge for n <= 32 splits and D a multiple of 128 (up to 1024): lane s owns
// split s's weight, each lane accumulates D/128 float4 columns in registers with all
// of them loaded as 16-byte vectors.  Same weights and the same split order as
// lse_combine_kernel, so the results are identical.
template <typename TO, typename TP = float>
__global__ void lse_combine_vec_kernel(int n, long rows, int D, const TP *po, const float *pl, TO *out,
                                       float *lse) {
    const long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    const int nc = D / 128;
    const float ls = lane < n ? pl[(long)lane * rows + r] : -INFINITY;
    const float m = warp_max(ls);
    if (m == -INFINITY) {
        for (int d = lane; d < D; d += 32) out[r * D + d] = TO(0.f);
        if (lane == 0) lse[r] = -INFINITY;
        return;
    }
    const float z = warp_sum(lane < n ? expf(ls - m) : 0.f);
    const float L = m + logf(z);
    const float w = lane < n ? expf(ls - L) : 0.f;
    float4 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);
        if (ws > 0.f) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < nc) {
                    float4 v;
                    if (sizeof(TP) == 4) {
                        v = ((const float4 *)(po + ((long)s * rows + r) * D))[lane + k * 32];
                    } else {   // fp16 partials: four per lane, the same elements
                        const uint2 u = ((const uint2 *)(po + ((long)s * rows + r) * D))[lane + k * 32];
                        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
                        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
                        v = make_float4(lo.x, lo.y, hi.x, hi.y);
                    }
                    acc[k].x = fmaf(ws, v.x, acc[k].x);
                    acc[k].y = fmaf(ws, v.y, acc[k].y);
                    acc[k].z = fmaf(ws, v.z, acc[k].z);
                    acc[k].w = fmaf(ws, v.w, acc[k].w);
                }
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < nc) {
            TO *dst = out + r * D + (k * 32 + lane) * 4;
            if (sizeof(TO) == 4) {
                *(float4 *)dst = acc[k];
            } else {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
                *(uint2 *)dst = make_uint2(*(uint32_t *)&lo, *(uint32_t *)&hi);
            }
        }
    if (lane == 0) lse[r] = L;
}

inline unsigned blocks_for(long n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace

cudaError_t launch_rope_table(long pos0, long n_pos, int Dr, float base, float2 *tab, cudaStream_t st) {
    long n = n_pos * (Dr / 2);
    if (n == 0) return cudaSuccess;
    if (Dr / 2 > ROPE_MAX_HALF) return cudaErrorInvalidValue;
    RopeTheta th;
    for (int t = 0; t < Dr / 2; ++t) th.v[t] = pow((double)base, -2.0 * (double)t / (double)Dr);
    ProfScope ps("rope_table", st);
    rope_table_kernel<<<blocks_for(n, 256), 256, 0, st>>>(pos0, n_pos, Dr / 2, th, tab);
    return cudaGetLastError();
}

cudaError_t launch_latent_prep(int tin, int tout, int B, int s_kv, int n_rows, int pad_rows, int Dk, int Dr,
                               const void *c_kv, const void *k_pe, const void *rms_w, float eps, const float2 *tab,
                               void *chat, void *kpe, cudaStream_t st) {
    long rows = (long)B * pad_rows;
    if (rows == 0) return cudaSuccess;
    ProfScope ps("latent_prep", st);
    bool vec = tin == TY_BF16 && Dk % 256 == 0 && Dk <= 1024 && (((uintptr_t)c_kv | (uintptr_t)rms_w) & 15) == 0;
    if (vec && tout == TY_F16)
        latent_prep_vec_kernel<__half><<<blocks_for(rows, 8), 256, 0, st>>>(
            B, s_kv, n_rows, pad_rows, Dk, Dr, (const __nv_bfloat16 *)c_kv, (const __nv_bfloat16 *)k_pe,
            (const __nv_bfloat16 *)rms_w, eps, tab, (__half *)chat, (__half *)kpe);
    else if (vec && tout == TY_F32)
        latent_prep_vec_kernel<float><<<blocks_for(rows, 8), 256, 0, st>>>(
            B, s_kv, n_rows, pad_rows, Dk, Dr, (const __nv_bfloat16 *)c_kv, (const __nv_bfloat16 *)k_pe,
            (const __nv_bfloat16 *)rms_w, eps, tab, (float *)chat, (float *)kpe);
    else
        latent_prep_kernel<<<blocks_for(rows, 8), 256, 0, st>>>(B, s_kv, n_rows, pad_rows, Dk, Dr, c_kv, k_pe,
                                                                rms_w, tin, eps, tab, chat, kpe, tout);
    return cudaGetLastError();
}

cudaError_t launch_rope_rows(int tin, int tout, long rows, int Dr, const void *x, long pos0, long pos_div,
                             long pos_mod, const float2 *tab, long tab_pos0, void *y, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    ProfScope ps("rope_rows", st);
    rope_rows_kernel<<<blocks_for(rows, 8), 256, 0, st>>>(rows, Dr, x, tin, pos0, pos_div, pos_mod, tab, tab_pos0,
                                                          y, tout);
    return cudaGetLastError();
}

cudaError_t launch_rope_rows_at(int tin, int tout, long rows, int Dr, const void *x, long pos, float base, void *y,
                                cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (Dr / 2 > ROPE_MAX_HALF) return cudaErrorInvalidValue;
    RopeTheta th;
    for (int t = 0; t < Dr / 2; ++t) th.v[t] = pow((double)base, -2.0 * (double)t / (double)Dr);
    ProfScope ps("rope_rows", st);
    rope_rows_at_kernel<<<blocks_for(rows, 8), 256, 0, st>>>(rows, Dr, x, tin, pos, th, y, tout);
    return cudaGetLastError();
}

bool prep_tc_supported(int Dk, int Dr) { return Dr == PREP_DR && Dk % 256 == 0 && Dk > 0 && Dk <= 1024; }

cudaError_t launch_prep_tc(int B, int s_kv, int n_rows, int pad_rows, int Dk, long n_pos, float base,
                           const void *c_kv, const void *k_pe, const void *rms_w, float eps, float2 *tab, void *chat,
                           void *kpe, const void *w_src, void *w16, long n_w, const void *q_pe, void *qpe, int s_q,
                           int q_offset, int n_hq, cudaStream_t st) {
    PrepTc a;
    a.B = B;
    a.s_kv = s_kv;
    a.n_rows = n_rows;
    a.pad_rows = pad_rows;
    a.Dk = Dk;
    a.n_pos = n_pos;
    a.c_kv = (const __nv_bfloat16 *)c_kv;
    a.k_pe = (const __nv_bfloat16 *)k_pe;
    a.rms_w = (const __nv_bfloat16 *)rms_w;
    a.eps = eps;
    a.tab = tab;
    a.chat = (__half *)chat;
    a.kpe = (__half *)kpe;
    a.w_src = (const uint4 *)w_src;
    a.w_dst = (uint4 *)w16;
    a.w_chunks = n_w / 8;
    a.q_pe = (const __nv_bfloat16 *)q_pe;
    a.qpe = (__half *)qpe;
    a.s_q = s_q;
    a.q_offset = q_offset;
    a.n_hq = n_hq;
    a.row_tasks = (long)B * pad_rows;
    a.tab_tasks = n_pos > pad_rows ? n_pos - pad_rows : 0;
    a.w_tasks = (a.w_chunks + 32 * PREP_W_PER_LANE - 1) / (32 * PREP_W_PER_LANE);
    for (int t = 0; t < PREP_DR / 2; ++t) a.theta[t] = pow((double)base, -2.0 * t / (double)PREP_DR);
    const long warps = a.row_tasks + a.tab_tasks + a.w_tasks;
    if (warps == 0) return cudaSuccess;
    ProfScope ps("prep", st);
    prep_tc_kernel<<<blocks_for(warps, 8), 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_convert(int tin, const void *x, int tout, void *y, long n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    ProfScope ps("convert", st);
    long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    convert_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, tin, y, tout, n);
    return cudaGetLastError();
}

cudaError_t launch_gemm_simt(const GemmArgs &g, cudaStream_t st) {
    if (g.M == 0 || g.N == 0 || g.nzb * g.nzh == 0) return cudaSuccess;
    dim3 grid(blocks_for(g.N, GT), blocks_for(g.M, GT), g.nzb * g.nzh), block(256);
    ProfScope ps("gemm_simt", st);
    gemm_simt_kernel<<<grid, block, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t st) {
    if (a.n_rows == 0 || a.n_b * a.n_h == 0 || a.n_splits == 0) return cudaSuccess;
    size_t smem = sizeof(float) * AKT * (size_t)(a.D1 + a.D2 + a.Dv);
    dim3 grid(blocks_for(a.n_rows, AW), a.n_b * a.n_h, a.n_splits), block(AW * 32);
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope ps("attn_simt", st);
    attn_simt_kernel<<<grid, block, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_lse_combine(int tout, int n, long rows, int D, const float *po, const float *pl, void *out,
                               float *lse, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    ProfScope ps("lse_combine", st);
    const bool vec = n <= 32 && D % 128 == 0 && D <= 1024 && ((uintptr_t)po & 15) == 0;
    if (vec && tout == TY_F32 && ((uintptr_t)out & 15) == 0)
        lse_combine_vec_kernel<float><<<blocks_for(rows, 8), 256, 0, st>>>(n, rows, D, po, pl, (float *)out, lse);
    else if (vec && tout == TY_BF16 && ((uintptr_t)out & 7) == 0)
        lse_combine_vec_kernel<__nv_bfloat16>
            <<<blocks_for(rows, 8), 256, 0, st>>>(n, rows, D, po, pl, (__nv_bfloat16 *)out, lse);
    else
        lse_combine_kernel<<<blocks_for(rows, 8), 256, 0, st>>>(n, rows, D, po, pl, out, tout, lse);
    return cudaGetLastError();
}

cudaError_t launch_lse_combine16(int n, long rows, int D, const void *po, const float *pl, void *out, float *lse,
                                 cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (n > 32 || D % 128 != 0 || D > 1024 || (((uintptr_t)po | (uintptr_t)out) & 7) != 0) return cudaErrorInvalidValue;
    ProfScope ps("lse_combine", st);
    lse_combine_vec_kernel<__nv_bfloat16, __half><<<blocks_for(rows, 8), 256, 0, st>>>(
        n, rows, D, (const __half *)po, pl, (__nv_bfloat16 *)out, lse);
    return cudaGetLastError();
}

// ------------------------------------------------------------- latent shards ----
__device__ __forceinline__ long ty_size_dev(int ty) { return ty == TY_F32 ? 4 : 2; }

// A 16-byte piece as 4 fp32 or 8 fp16/bf16 values, and back.
__device__ __forceinline__ void unpack16(uint4 v, int ty, float *f) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (ty == TY_F32) {
            f[t] = __uint_as_float(u[t]);
        } else if (ty == TY_BF16) {
            f[2 * t] = __uint_as_float(u[t] << 16);
            f[2 * t + 1] = __uint_as_float(u[t] & 0xffff0000u);
        } else {
            const __half2 h = *(const __half2 *)&u[t];
            f[2 * t] = __low2float(h);
            f[2 * t + 1] = __high2float(h);
        }
    }
}

__device__ __forceinline__ uint4 pack16(const float *f, int ty) {
    uint32_t u[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (ty == TY_F32) {
            u[t] = __float_as_uint(f[t]);
        } else if (ty == TY_BF16) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * t], f[2 * t + 1]);
            u[t] = *(const uint32_t *)&h;
        } else {
            const __half2 h = __floats2half2_rn(f[2 * t], f[2 * t + 1]);
            u[t] = *(const uint32_t *)&h;
        }
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// TPLA ("The reading"): the latent row is cut into g equal shards and each shard is
// RMS-normalised on its own with the matching slice of the weight (g = 1: the plain
// RMSNorm of the LAGA page's step 1).  One warp per (row, shard); with `vec` each lane
// moves 16-byte pieces (the shard's byte width is then a multiple of 16).
__global__ void rmsnorm_shards_kernel(int ty, long rows, int D, int g, float eps, bool vec, const void *x,
                                      const void *w, void *y) {
    const long u = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (u >= rows * g) return;
    const long r = u / g;
    const int ds = D / g, k0 = (int)(u % g) * ds;
    const long o = r * D + k0;
    float ss = 0.f;
    if (vec) {
        const int per = ty == TY_F32 ? 4 : 8, nv = ds / per;
        const uint4 *src = (const uint4 *)((const char *)x + o * ty_size_dev(ty));
        for (int c = lane; c < nv; c += 32) {
            const uint4 v = src[c];
            float f[8];
            unpack16(v, ty, f);
            for (int t = 0; t < per; ++t) ss = fmaf(f[t], f[t], ss);
        }
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)ds + eps);
        uint4 *dst = (uint4 *)((char *)y + o * ty_size_dev(ty));
        const uint4 *wv = (const uint4 *)((const char *)w + (long)k0 * ty_size_dev(ty));
        for (int c = lane; c < nv; c += 32) {
            float f[8], fw[8];
            unpack16(src[c], ty, f);
            unpack16(wv[c], ty, fw);
            for (int t = 0; t < per; ++t) f[t] = f[t] * inv * fw[t];
            dst[c] = pack16(f, ty);
        }
        return;
    }
    for (int k = lane; k < ds; k += 32) {
        const float v = ldx(x, ty, o + k);
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)ds + eps);
    for (int k = lane; k < ds; k += 32) stx(y, ty, o + k, ldx(x, ty, o + k) * inv * ldx(w, ty, k0 + k));
}

// The same norm with whole rows in registers: each warp takes two rows, lane l holds
// their 16-byte pieces l, l + 32, ... (NP per row, all loaded before any arithmetic),
// and every shard covers a whole number of 512-byte rounds, so piece p of every lane
// lies in shard p / (NP / g) and each shard's sum is one warp reduction.
template <int NP>
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(int ty, long rows, int D, int g, float eps,
                                                           const uint4 *x, const uint4 *w, uint4 *y) {
    constexpr int RW = 2;
    const long r0 = ((long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * RW;
    const int lane = threadIdx.x % 32;
    if (r0 >= rows) return;
    const int per = ty == TY_F32 ? 4 : 8, sp = NP / g, ds = D / g;
    uint4 v[RW][NP];
#pragma unroll
    for (int q = 0; q < RW; ++q)
#pragma unroll
        for (int p = 0; p < NP; ++p)
            v[q][p] = r0 + q < rows ? x[(r0 + q) * (NP * 32) + p * 32 + lane] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < RW; ++q) {
        float ps[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float f[8];
            unpack16(v[q][p], ty, f);
            float a = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (t < per) a = fmaf(f[t], f[t], a);
            ps[p] = a;
        }
        float inv[NP];
        for (int i = 0; i < g; ++i) {
            float a = 0.f;
#pragma unroll
            for (int p = 0; p < NP; ++p)
                if (p / sp == i) a += ps[p];
            a = 1.0f / sqrtf(warp_sum(a) / (float)ds + eps);
#pragma unroll
            for (int p = 0; p < NP; ++p)
                if (p / sp == i) inv[p] = a;
        }
        if (r0 + q >= rows) break;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float f[8], fw[8];
            unpack16(v[q][p], ty, f);
            unpack16(w[p * 32 + lane], ty, fw);
#pragma unroll
            for (int t = 0; t < 8; ++t) f[t] = f[t] * inv[p] * fw[t];
            y[(r0 + q) * (NP * 32) + p * 32 + lane] = pack16(f, ty);
        }
    }
}

// Backward of the per-shard RMSNorm: with r the shard's sqrt(mean x^2 + eps) and ds its
// width, dx_k = dy_k w_k / r - x_k (sum_shard dy w x) / (ds r^3) and dw_k = sum_rows
// dy_k x_k / r.  Whole rows in registers as in rmsnorm_rows_kernel (NP pieces of 16
// bytes per lane, shards of whole 512-byte rounds); each warp walks rows with a grid
// stride.  Its rows' x and dy arrive by bulk copies into a ring of PF shared-memory slots
// (one mbarrier each), so PF rows per warp are in flight without holding registers; a
// slot is refilled with the row PF strides ahead once the warp has used the one it held.
// The dw terms and the weight row stay in registers; the block's warps add their dw terms
// into shared memory in a fixed order and the block writes one partial row of dw (fp32).
constexpr int RMS_BWD_PF = 4;
__device__ unsigned g_rms_err = 0;

template <int NP>
constexpr uint32_t rms_bwd_smem() {
    return 8 * RMS_BWD_PF * (2 * NP * 512 + 8) + NP * 256 * 4 + 16;
}

template <int NP>
__global__ void __launch_bounds__(256) rmsnorm_bwd_rows_kernel(int ty, long rows, int D, int g, float eps,
                                                               const uint4 *x, const uint4 *w, const uint4 *dy,
                                                               uint4 *dx, float *dw_part) {
    using namespace tc;
    constexpr int PF = RMS_BWD_PF;
    constexpr uint32_t ROW = NP * 512;   // bytes of one row of x (and of dy)
    extern __shared__ __align__(16) uint8_t sm[];
    const int lane = threadIdx.x % 32, wib = threadIdx.x / 32, nwb = blockDim.x / 32;
    uint8_t *slots = sm + wib * PF * 2 * ROW;                           // [PF][x, dy] of this warp
    uint64_t *bar = (uint64_t *)(sm + 8 * PF * 2 * ROW) + wib * PF;    // [PF] of this warp
    float *red = (float *)(sm + 8 * PF * (2 * ROW + 8));
    volatile int *abort = (volatile int *)(red + NP * 256);
    const int per = ty == TY_F32 ? 4 : 8, sp = NP / g;
    const float ds = (float)(D / g);
    if (threadIdx.x == 0) *abort = 0;
    if (lane == 0)
        for (int s = 0; s < PF; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    __syncthreads();
    float acc[NP][8];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[p][t] = 0.f;
    uint4 wr[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) wr[p] = w[p * 32 + lane];
    const long stride = (long)gridDim.x * nwb, r_first = (long)blockIdx.x * nwb + wib;
    auto issue = [&](int s, long r) {
        if (lane == 0 && r < rows) {
            mbar_arrive_expect_tx(&bar[s], 2 * ROW);
            bulk_load(slots + s * 2 * ROW, (const uint8_t *)x + r * ROW, ROW, &bar[s]);
            bulk_load(slots + s * 2 * ROW + ROW, (const uint8_t *)dy + r * ROW, ROW, &bar[s]);
        }
    };
#pragma unroll
    for (int s = 0; s < PF; ++s) issue(s, r_first + s * stride);
    bool ok = true;
    long k = 0;   // rows this warp has walked
    for (long r = r_first; r < rows && ok; r += stride, ++k) {
        const int s = (int)(k % PF);
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[s], (uint32_t)(k / PF) & 1, abort, &g_rms_err));
        if (!ok) break;
        uint4 xv[NP], gv[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            xv[p] = *(const uint4 *)(slots + s * 2 * ROW + p * 512 + lane * 16);
            gv[p] = *(const uint4 *)(slots + s * 2 * ROW + ROW + p * 512 + lane * 16);
        }
        float ss[NP], gg[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float xf[8], gf[8], wf[8];
            unpack16(xv[p], ty, xf);
            unpack16(gv[p], ty, gf);
            unpack16(wr[p], ty, wf);
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (t < per) {
                    a = fmaf(xf[t], xf[t], a);
                    b = fmaf(gf[t] * wf[t], xf[t], b);
                }
            ss[p] = a;
            gg[p] = b;
        }
        // every lane has its values of the slot (used above): the slot may be refilled
        fence_proxy_async_smem();
        __syncwarp();
        issue(s, r + PF * stride);
        // every piece's two sums across the warp at once (independent shuffle chains),
        // then each shard adds its pieces' totals
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                ss[p] += __shfl_xor_sync(0xffffffffu, ss[p], off);
                gg[p] += __shfl_xor_sync(0xffffffffu, gg[p], off);
            }
        float inv[NP], coef[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int q = 0; q < NP; ++q)
                if (q / sp == p / sp) {
                    a += ss[q];
                    b += gg[q];
                }
            inv[p] = 1.0f / sqrtf(a / ds + eps);
            coef[p] = b * inv[p] * inv[p] * inv[p] / ds;
        }
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float xf[8], gf[8], wf[8], o[8];
            unpack16(xv[p], ty, xf);
            unpack16(gv[p], ty, gf);
            unpack16(wr[p], ty, wf);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                o[t] = gf[t] * wf[t] * inv[p] - xf[t] * coef[p];
                acc[p][t] = fmaf(gf[t] * xf[t], inv[p], acc[p][t]);
            }
            dx[r * (NP * 32) + p * 32 + lane] = pack16(o, ty);
        }
    }
    if (!ok) {
        // after a failed wait: the copies of rows k .. k + PF - 1 were issued; let them land
        // (each wait bounded again) before the block exits
        int no_abort = 0;
        for (long kk = k; kk < k + PF && r_first + kk * stride < rows; ++kk)
            mbar_wait_limit(&bar[kk % PF], (uint32_t)(kk / PF) & 1, &no_abort, &g_rms_err, WAIT_NS);
    }
    for (int v = 0; v < nwb; ++v) {   // warp v adds its terms: the same order in every run
        if (wib == v)
#pragma unroll
            for (int p = 0; p < NP; ++p)
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    if (t < per) {
                        const int kc = (p * 32 + lane) * per + t;
                        red[kc] = (v == 0 ? 0.f : red[kc]) + acc[p][t];
                    }
        __syncthreads();
    }
    for (int kc = threadIdx.x; kc < D; kc += blockDim.x) dw_part[(long)blockIdx.x * D + kc] = red[kc];
}

// The same gradient for any shape: one warp per (row, shard) writes dx and the shard's
// 1/r; then dw in two fixed-order passes: block column y of rmsnorm_dw_kernel sums its
// contiguous run of rows per column into partial row y, and dw_reduce_kernel adds the
// partial rows in order.
__global__ void rmsnorm_bwd_kernel(int ty, long rows, int D, int g, float eps, const void *x, const void *w,
                                   const void *dy, void *dx, float *inv_r) {
    const long u = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (u >= rows * g) return;
    const int ds = D / g, k0 = (int)(u % g) * ds;
    const long o = (u / g) * D + k0;
    float ss = 0.f, gs = 0.f;
    for (int k = lane; k < ds; k += 32) {
        const float xv = ldx(x, ty, o + k);
        ss = fmaf(xv, xv, ss);
        gs = fmaf(ldx(dy, ty, o + k) * ldx(w, ty, k0 + k), xv, gs);
    }
    const float ri = 1.0f / sqrtf(warp_sum(ss) / (float)ds + eps);
    const float c = warp_sum(gs) * ri * ri * ri / (float)ds;
    for (int k = lane; k < ds; k += 32)
        stx(dx, ty, o + k, ldx(dy, ty, o + k) * ldx(w, ty, k0 + k) * ri - ldx(x, ty, o + k) * c);
    if (lane == 0) inv_r[u] = ri;
}

__global__ void rmsnorm_dw_kernel(int ty, long rows, int D, int g, const void *x, const void *dy, const float *inv_r,
                                  long rows_per_part, float *dw_part) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= D) return;
    const int i = k / (D / g);
    const long r0 = (long)blockIdx.y * rows_per_part, r1 = min(rows, r0 + rows_per_part);
    float a = 0.f;
    for (long r = r0; r < r1; ++r) a = fmaf(ldx(dy, ty, r * D + k) * ldx(x, ty, r * D + k), inv_r[r * g + i], a);
    dw_part[(long)blockIdx.y * D + k] = a;
}

// The general-shape dw pass with 16-byte loads (row bytes a multiple of 16, aligned
// pointers): thread c of block column y sums dy_k x_k / r over its run of rows for the
// per16 columns [per16 c, per16 c + per16), each column with its own shard's 1/r.
__global__ void rmsnorm_dw_vec_kernel(int ty, long rows, int D, int g, const uint4 *x, const uint4 *dy,
                                      const float *inv_r, long rows_per_part, float *dw_part) {
    const int per = ty == TY_F32 ? 4 : 8, nc = D / per;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= nc) return;
    const int ds = D / g;
    int sh[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) sh[t] = min((c * per + t) / ds, g - 1);
    const long r0 = (long)blockIdx.y * rows_per_part, r1 = min(rows, r0 + rows_per_part);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (long r = r0; r < r1; ++r) {
        float xf[8], gf[8];
        unpack16(x[r * nc + c], ty, xf);
        unpack16(dy[r * nc + c], ty, gf);
#pragma unroll
        for (int t = 0; t < 8; ++t)
            if (t < per) a[t] = fmaf(gf[t] * xf[t], inv_r[r * g + sh[t]], a[t]);
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
        if (t < per) dw_part[(long)blockIdx.y * D + c * per + t] = a[t];
}

// dw[k] = sum over the partial rows in order
__global__ void dw_reduce_kernel(int nparts, int D, const float *part, float *dw) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= D) return;
    float a = 0.f;
    for (int b = 0; b < nparts; ++b) a += part[(long)b * D + k];
    dw[k] = a;
}

// TPLA decode, query side: every head becomes g query rows, one per latent shard.  Row
// (b, i, h) keeps q_abs[b][h] on shard i's dims and zero elsewhere, so its score over
// the full latent row is the shard-local score q_abs_i . c_i; the rotated q_pe is
// replicated (every shard also reads the whole RoPE band).
// qa [B][H][Dk], qp [B][H][Dr] -> qx [B][g][H][Dk], qpx [B][g][H][Dr]; storage `ty`.
// With `vec` every shard's byte width and Dr's are multiples of 16 and pieces of 16
// bytes move at a time.
__global__ void tpla_expand_kernel(int ty, int B, int H, int g, int Dk, int Dr, bool vec, const void *qa,
                                   const void *qp, void *qx, void *qpx) {
    const long es = ty_size_dev(ty), per = vec ? 16 / es : 1;
    const long nk = Dk / per, nr = Dr / per, row_units = nk + nr;
    const long total = (long)B * g * H * row_units, ds = Dk / g;
    for (long u = (long)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (long)gridDim.x * blockDim.x) {
        const long row = u / row_units, c = u % row_units;   // row = (b * g + i) * H + h
        const long h = row % H, bi = row / H, i = bi % g, b = bi / g;
        const long src_row = b * H + h;
        if (c < nk) {
            const long k = c * per;
            const bool keep = k / ds == i;
            if (vec) {
                const uint4 v = keep ? ((const uint4 *)qa)[src_row * nk + c] : make_uint4(0, 0, 0, 0);
                ((uint4 *)qx)[row * nk + c] = v;
            } else {
                stx(qx, ty, row * Dk + k, keep ? ldx(qa, ty, src_row * Dk + k) : 0.f);
            }
        } else {
            const long t = c - nk;
            if (vec)
                ((uint4 *)qpx)[row * nr + t] = ((const uint4 *)qp)[src_row * nr + t];
            else
                stx(qpx, ty, row * Dr + t, ldx(qp, ty, src_row * Dr + t));
        }
    }
}

// TPLA decode, output side: rows (b, i, h) of the split partials are merged by the
// log-sum-exp rescale, only over shard i's dims, into o_lat[b][h] (each shard fills its
// own dims, so the later W_V product sums the shards' up-projections), and each row's
// log-sum-exp goes to shard_lse[i][b][h].
// po [n][B][g][H][Dk], pl [n][B][g][H] (fp32) -> out [B][H][Dk] (storage `to`).
__global__ void tpla_combine_kernel(int n, int B, int H, int g, int Dk, bool vec, const float *po, const float *pl,
                                    void *out, int to, float *slse) {
    const long rows = (long)B * g * H;
    const long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    const long h = r % H, bi = r / H, i = bi % g, b = bi / g;
    const int ds = Dk / g, k0 = (int)i * ds;
    const long orow = (b * H + h) * Dk + k0;
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, pl[(long)s * rows + r]);
    m = warp_max(m);
    float L = -INFINITY;
    if (m != -INFINITY) {
        float z = 0.f;
        for (int s = lane; s < n; s += 32) z += expf(pl[(long)s * rows + r] - m);
        L = m + logf(warp_sum(z));
    }
    if (vec) {
        // lane s holds split s's weight; 16-byte loads of the shard's partial columns
        const float wl = lane < n && m != -INFINITY ? expf(pl[(long)lane * rows + r] - L) : 0.f;
        for (int c = lane; c < ds / 4; c += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s = 0; s < n; ++s) {
                const float wt = __shfl_sync(0xffffffffu, wl, s);
                if (wt > 0.f) {
                    const float4 v = *(const float4 *)(po + ((long)s * rows + r) * Dk + k0 + 4 * c);
                    acc.x = fmaf(wt, v.x, acc.x);
                    acc.y = fmaf(wt, v.y, acc.y);
                    acc.z = fmaf(wt, v.z, acc.z);
                    acc.w = fmaf(wt, v.w, acc.w);
                }
            }
            stx(out, to, orow + 4 * c, acc.x);
            stx(out, to, orow + 4 * c + 1, acc.y);
            stx(out, to, orow + 4 * c + 2, acc.z);
            stx(out, to, orow + 4 * c + 3, acc.w);
        }
        if (lane == 0) slse[(i * B + b) * H + h] = L;
        return;
    }
    for (int d = lane; d < ds; d += 32) {
        float acc = 0.f;
        if (m != -INFINITY)
            for (int s = 0; s < n; ++s) {
                const float wt = expf(pl[(long)s * rows + r] - L);
                if (wt > 0.f) acc = fmaf(wt, po[((long)s * rows + r) * Dk + k0 + d], acc);
            }
        stx(out, to, orow + d, acc);
    }
    if (lane == 0) slse[(i * B + b) * H + h] = L;
}

cudaError_t launch_rmsnorm_shards(int ty, long rows, int D, int g, float eps, const void *x, const void *w, void *y,
                                  cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    ProfScope ps("rmsnorm", st);
    const bool vec = ((long)(D / g) * (long)ty_size(ty)) % 16 == 0 && ((uintptr_t)x & 15) == 0 &&
                     ((uintptr_t)y & 15) == 0 && ((uintptr_t)w & 15) == 0;
    const long row_bytes = (long)D * (long)ty_size(ty), np = row_bytes / 512;
    if (vec && ((long)(D / g) * (long)ty_size(ty)) % 512 == 0 && (np == 1 || np == 2 || np == 4 || np == 8)) {
        const unsigned blocks = blocks_for((rows + 1) / 2, 8);
        const uint4 *xv = (const uint4 *)x, *wv = (const uint4 *)w;
        uint4 *yv = (uint4 *)y;
        if (np == 1) rmsnorm_rows_kernel<1><<<blocks, 256, 0, st>>>(ty, rows, D, g, eps, xv, wv, yv);
        if (np == 2) rmsnorm_rows_kernel<2><<<blocks, 256, 0, st>>>(ty, rows, D, g, eps, xv, wv, yv);
        if (np == 4) rmsnorm_rows_kernel<4><<<blocks, 256, 0, st>>>(ty, rows, D, g, eps, xv, wv, yv);
        if (np == 8) rmsnorm_rows_kernel<8><<<blocks, 256, 0, st>>>(ty, rows, D, g, eps, xv, wv, yv);
        return cudaGetLastError();
    }
    rmsnorm_shards_kernel<<<blocks_for(rows * g, 8), 256, 0, st>>>(ty, rows, D, g, eps, vec, x, w, y);
    return cudaGetLastError();
}

namespace {
constexpr long BWD_BLOCKS = 152L * 2;   // fused backward: blocks of 8 warps (two resident per SM), grid-strided over rows
long bwd_np(int ty, int D, int g) {    // pieces per lane of the fused kernel, 0 = other shapes
    const long es = (long)ty_size(ty), np = (long)D * es / 512;
    const bool ok = ((long)(D / g) * es) % 512 == 0 && (np == 1 || np == 2 || np == 4);
    return ok ? np : 0;
}
}  // namespace

namespace {
// Partial rows of the general-shape dw pass: runs of at least 64 rows, at most 1024 parts.
long dw_parts(long rows) { return std::max<long>(1, std::min<long>(1024, (rows + 63) / 64)); }
}  // namespace

template <int NP>
cudaError_t launch_rms_bwd_rows(long nb, int ty, long rows, int D, int g, float eps, const uint4 *x, const uint4 *w,
                                const uint4 *dy, uint4 *dx, float *ws, cudaStream_t st) {
    constexpr uint32_t smem = rms_bwd_smem<NP>();
    cudaError_t e = cudaFuncSetAttribute(rmsnorm_bwd_rows_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    rmsnorm_bwd_rows_kernel<NP><<<(unsigned)nb, 256, smem, st>>>(ty, rows, D, g, eps, x, w, dy, dx, ws);
    return cudaGetLastError();
}

size_t rmsnorm_bwd_ws(int ty, long rows, int D, int g) {
    const size_t fused = (size_t)std::min<long>(BWD_BLOCKS, std::max<long>((rows + 7) / 8, 1)) * D * 4;
    // 1/r of every (row, shard), 256-byte aligned, then the partial dw rows
    const size_t plain = ((size_t)rows * g * 4 + 255) / 256 * 256 + (size_t)dw_parts(rows) * D * 4;
    return std::max(fused, plain);
}

cudaError_t launch_rmsnorm_bwd(int ty, long rows, int D, int g, float eps, const void *x, const void *w,
                               const void *dy, void *dx, float *dw, float *ws, cudaStream_t st) {
    ProfScope ps("rmsnorm_bwd", st);
    const long np = bwd_np(ty, D, g);
    const bool vec = np && ((uintptr_t)x & 15) == 0 && ((uintptr_t)w & 15) == 0 && ((uintptr_t)dy & 15) == 0 &&
                     ((uintptr_t)dx & 15) == 0;
    if (rows > 0 && vec) {
        const long nb = std::min<long>(BWD_BLOCKS, (rows + 7) / 8);
        const uint4 *xv = (const uint4 *)x, *wv = (const uint4 *)w, *gv = (const uint4 *)dy;
        uint4 *dxv = (uint4 *)dx;
        cudaError_t e = cudaSuccess;
        if (np == 1) e = launch_rms_bwd_rows<1>(nb, ty, rows, D, g, eps, xv, wv, gv, dxv, ws, st);
        if (np == 2) e = launch_rms_bwd_rows<2>(nb, ty, rows, D, g, eps, xv, wv, gv, dxv, ws, st);
        if (np == 4) e = launch_rms_bwd_rows<4>(nb, ty, rows, D, g, eps, xv, wv, gv, dxv, ws, st);
        if (e != cudaSuccess) return e;
        dw_reduce_kernel<<<blocks_for(D, 256), 256, 0, st>>>((int)nb, D, ws, dw);
    } else if (rows > 0) {
        rmsnorm_bwd_kernel<<<blocks_for(rows * g, 8), 256, 0, st>>>(ty, rows, D, g, eps, x, w, dy, dx, ws);
        const long parts = dw_parts(rows), per = (rows + parts - 1) / parts;
        float *part = ws + ((size_t)rows * g * 4 + 255) / 256 * 64;
        const long es = (long)ty_size(ty);
        const bool dw_vec = ((long)D * es) % 16 == 0 && ((uintptr_t)x & 15) == 0 && ((uintptr_t)dy & 15) == 0;
        if (dw_vec) {
            const int nc = (int)((long)D * es / 16);
            rmsnorm_dw_vec_kernel<<<dim3(blocks_for(nc, 64), (unsigned)parts), 64, 0, st>>>(
                ty, rows, D, g, (const uint4 *)x, (const uint4 *)dy, ws, per, part);
        } else {
            rmsnorm_dw_kernel<<<dim3(blocks_for(D, 128), (unsigned)parts), 128, 0, st>>>(ty, rows, D, g, x, dy, ws,
                                                                                          per, part);
        }
        dw_reduce_kernel<<<blocks_for(D, 256), 256, 0, st>>>((int)parts, D, part, dw);
    } else {
        dw_reduce_kernel<<<blocks_for(D, 256), 256, 0, st>>>(0, D, ws, dw);   // no rows: dw = 0
    }
    return cudaGetLastError();
}

cudaError_t simt_read_and_clear_error(unsigned *flags, cudaStream_t st) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_rms_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    if (v) {
        unsigned z = 0;
        e = cudaMemcpyToSymbolAsync(g_rms_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *flags |= v;
    return e;
}

cudaError_t launch_tpla_expand(int ty, int B, int H, int g, int Dk, int Dr, const void *qa, const void *qp, void *qx,
                               void *qpx, cudaStream_t st) {
    if ((long)B * H == 0) return cudaSuccess;
    ProfScope ps("tpla_expand", st);
    const long es = (long)ty_size(ty);
    const bool vec = ((long)(Dk / g) * es) % 16 == 0 && (Dr * es) % 16 == 0 && ((uintptr_t)qa & 15) == 0 &&
                     ((uintptr_t)qp & 15) == 0 && ((uintptr_t)qx & 15) == 0 && ((uintptr_t)qpx & 15) == 0;
    const long per = vec ? 16 / es : 1, units = (long)B * g * H * ((Dk + Dr) / per);
    const long blocks = std::min<long>((units + 255) / 256, 152L * 16);
    tpla_expand_kernel<<<(unsigned)blocks, 256, 0, st>>>(ty, B, H, g, Dk, Dr, vec, qa, qp, qx, qpx);
    return cudaGetLastError();
}

cudaError_t launch_tpla_combine(int tout, int n, int B, int H, int g, int Dk, const float *po, const float *pl,
                                void *out, float *slse, cudaStream_t st) {
    const long rows = (long)B * g * H;
    if (rows == 0) return cudaSuccess;
    ProfScope ps("tpla_combine", st);
    const bool vec = n <= 32 && (Dk / g) % 128 == 0 && ((uintptr_t)po & 15) == 0;
    tpla_combine_kernel<<<blocks_for(rows, 8), 256, 0, st>>>(n, B, H, g, Dk, vec, po, pl, out, tout, slse);
    return cudaGetLastError();
}

}  // namespace mla
