// simt.cu -- CUDA-core kernels of libmla: any dimensions, fp32 or bf16 storage,
// fp32 arithmetic.  They carry the fp32 dtype (which tensor cores cannot hold to a
// 1e-4 error) and every shape the tensor-core kernels do not cover.
//
// Method: "A Training-Memory Regression in MLA Sequence Parallelism ... LAGA"
// (arXiv 2607.17644), "What carries the argument" and Fig. 2 (explicit and absorbed
// dataflows); "Helix Parallelism ..." (arXiv 2507.07120), "What carries the
// argument" (log-sum-exp rescale of split partials).
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.h"

namespace mla {
namespace {

template <typename T> __device__ __forceinline__ float ldf(const T *p);
template <> __device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ T stf(float x);
template <> __device__ __forceinline__ float stf<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 stf<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
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

// Rotates one Dr-wide band at `pos` (half-split pairs).  The angle pos*theta_t is
// formed and reduced in double precision: positions reach 10^4..10^5, where a float
// angle would already be off by ~1e-3 rad.
template <typename T>
__device__ void rope_band(const T *x, T *y, int Dr, double pos, double base, int lane) {
    int half = Dr / 2;
    for (int t = lane; t < half; t += 32) {
        double theta = pow(base, -2.0 * (double)t / (double)Dr);
        double s, c;
        sincos(pos * theta, &s, &c);
        float x0 = ldf(x + t), x1 = ldf(x + t + half);
        float cf = (float)c, sf = (float)s;
        y[t] = stf<T>(x0 * cf - x1 * sf);
        y[t + half] = stf<T>(x1 * cf + x0 * sf);
    }
}

// Rows j in [n_rows, pad_rows) of each batch are written as zeros, so that padded
// tiles read by later kernels hold finite values.
template <typename T>
__global__ void latent_prep_kernel(int B, int s_kv, int n_rows, int pad_rows, int Dk, int Dr,
                                   const T *c_kv, const T *k_pe, const T *rms_w, float eps,
                                   float base, T *chat, T *kpe) {
    long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (row >= (long)B * pad_rows) return;
    long b = row / pad_rows, j = row % pad_rows;
    if (j >= n_rows) {
        for (int k = lane; k < Dk; k += 32) chat[row * Dk + k] = stf<T>(0.f);
        for (int k = lane; k < Dr; k += 32) kpe[row * Dr + k] = stf<T>(0.f);
        return;
    }
    const T *x = c_kv + (b * s_kv + j) * Dk;
    float ss = 0.f;
    for (int k = lane; k < Dk; k += 32) {
        float v = ldf(x + k);
        ss += v * v;
    }
    ss = warp_sum(ss);
    float inv = 1.0f / sqrtf(ss / (float)Dk + eps);
    T *y = chat + row * Dk;
    for (int k = lane; k < Dk; k += 32) y[k] = stf<T>(ldf(x + k) * inv * ldf(rms_w + k));
    rope_band(k_pe + (b * s_kv + j) * Dr, kpe + row * Dr, Dr, (double)j, (double)base, lane);
}

template <typename T>
__global__ void rope_rows_kernel(long rows, int Dr, const T *x, long pos0, long pos_div,
                                 long pos_mod, float base, T *y) {
    long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (r >= rows) return;
    long pos = pos0 + (r / pos_div) % pos_mod;
    rope_band(x + r * Dr, y + r * Dr, Dr, (double)pos, (double)base, threadIdx.x % 32);
}

// ---------------------------------------------------------------- GEMM ----
constexpr int GT = 64, GK = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
    __shared__ float As[GK][GT + 1], Bs[GK][GT + 1];
    int zb = blockIdx.z / g.nzh, zh = blockIdx.z % g.nzh;
    const T *A = (const T *)g.A + zb * g.a_zb + zh * g.a_zh;
    const T *Bm = (const T *)g.B + zb * g.b_zb + zh * g.b_zh;
    T *C = (T *)g.C + zb * g.c_zb + zh * g.c_zh;
    int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
    int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += GK) {
        for (int i = threadIdx.x; i < GK * GT; i += 256) {
            int kk = i / GT, mm = i % GT;
            int m = m0 + mm, n = n0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.M && k < g.K) ? ldf(A + m * g.a_m + k * g.a_k) : 0.f;
            Bs[kk][mm] = (n < g.N && k < g.K) ? ldf(Bm + n * g.b_n + k * g.b_k) : 0.f;
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
            if (m < g.M && n < g.N) C[m * g.c_m + n * g.c_n] = stf<T>(acc[i][j]);
        }
}

// ----------------------------------------------------------- attention ----
constexpr int AW = 8;      // warps (= query rows) per block
constexpr int AKT = 16;    // keys per shared-memory tile
constexpr int QMAX = 640;  // D1 + D2 limit (registers per lane: QMAX/32)
constexpr int VMAX = 512;  // Dv limit

template <typename T>
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

    const T *q1 = (const T *)a.q1 + b * a.q1_b + h * a.q1_h + r * a.q1_r;
    const T *q2 = (const T *)a.q2 + b * a.q2_b + h * a.q2_h + r * a.q2_r;
    float q[QMAX / 32];
#pragma unroll
    for (int t = 0; t < QMAX / 32; ++t) {
        int d = lane + 32 * t;
        float v = 0.f;
        if (active && d < a.D1) v = ldf(q1 + d);
        else if (active && d < Dq) v = ldf(q2 + (d - a.D1));
        q[t] = v;
    }
    float o[VMAX / 32];
#pragma unroll
    for (int t = 0; t < VMAX / 32; ++t) o[t] = 0.f;
    float m = -INFINITY, l = 0.f;

    const T *K1 = (const T *)a.k1 + b * a.k1_b + h * a.k1_h;
    const T *K2 = (const T *)a.k2 + b * a.k2_b + h * a.k2_h;
    const T *V = (const T *)a.v + b * a.v_b + h * a.v_h;

    for (long k0 = kb; k0 < kend_blk; k0 += AKT) {
        __syncthreads();
        for (int i = threadIdx.x; i < AKT * Dq; i += blockDim.x) {
            int kk = i / Dq, d = i % Dq;
            long key = k0 + kk;
            float v = 0.f;
            if (key < kend_blk) v = d < a.D1 ? ldf(K1 + key * a.k1_r + d) : ldf(K2 + key * a.k2_r + (d - a.D1));
            sK[i] = v;
        }
        for (int i = threadIdx.x; i < AKT * a.Dv; i += blockDim.x) {
            int kk = i / a.Dv, d = i % a.Dv;
            long key = k0 + kk;
            sV[i] = key < kend_blk ? ldf(V + key * a.v_r + d) : 0.f;
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
            float p = expf(s[kk] - mn);
            l += p;
#pragma unroll
            for (int t = 0; t < VMAX / 32; ++t) {
                int d = lane + 32 * t;
                if (d < a.Dv) o[t] = fmaf(p, sV[kk * a.Dv + d], o[t]);
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
        T *out = (T *)a.out + b * a.o_b + h * a.o_h + r * a.o_r;
#pragma unroll
        for (int t = 0; t < VMAX / 32; ++t) {
            int d = lane + 32 * t;
            if (d < a.Dv) out[d] = stf<T>(o[t] * inv);
        }
        if (lane == 0) a.lse[b * a.l_b + h * a.l_h + r * a.l_r] = lse;
    }
}

// --------------------------------------------------------- lse combine ----
template <typename T>
__global__ void lse_combine_kernel(int n, long rows, int D, const float *po, const float *pl,
                                   T *out, float *lse) {
    long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (r >= rows) return;
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, pl[(long)s * rows + r]);
    m = warp_max(m);
    T *o = out + r * D;
    if (m == -INFINITY) {
        for (int d = lane; d < D; d += 32) o[d] = stf<T>(0.f);
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
        o[d] = stf<T>(acc);
    }
    if (lane == 0) lse[r] = L;
}

inline unsigned blocks_for(long n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace

cudaError_t launch_latent_prep(mla_dtype dt, int B, int s_kv, int n_rows, int pad_rows, int Dk,
                               int Dr, const void *c_kv, const void *k_pe, const void *rms_w,
                               float eps, float base, void *chat, void *kpe, cudaStream_t st) {
    long rows = (long)B * pad_rows;
    if (rows == 0) return cudaSuccess;
    dim3 grid(blocks_for(rows, 8)), block(256);
    ProfScope ps("latent_prep", st);
    if (dt == MLA_F32)
        latent_prep_kernel<float><<<grid, block, 0, st>>>(B, s_kv, n_rows, pad_rows, Dk, Dr,
            (const float *)c_kv, (const float *)k_pe, (const float *)rms_w, eps, base, (float *)chat,
            (float *)kpe);
    else
        latent_prep_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(B, s_kv, n_rows, pad_rows, Dk, Dr,
            (const __nv_bfloat16 *)c_kv, (const __nv_bfloat16 *)k_pe, (const __nv_bfloat16 *)rms_w, eps,
            base, (__nv_bfloat16 *)chat, (__nv_bfloat16 *)kpe);
    return cudaGetLastError();
}

cudaError_t launch_rope_rows(mla_dtype dt, long rows, int Dr, const void *x, long pos0,
                             long pos_div, long pos_mod, float base, void *y, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    dim3 grid(blocks_for(rows, 8)), block(256);
    ProfScope ps("rope_rows", st);
    if (dt == MLA_F32)
        rope_rows_kernel<float><<<grid, block, 0, st>>>(rows, Dr, (const float *)x, pos0, pos_div, pos_mod,
                                                        base, (float *)y);
    else
        rope_rows_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(rows, Dr, (const __nv_bfloat16 *)x, pos0,
                                                                pos_div, pos_mod, base, (__nv_bfloat16 *)y);
    return cudaGetLastError();
}

cudaError_t launch_gemm_simt(mla_dtype dt, const GemmArgs &g, cudaStream_t st) {
    if (g.M == 0 || g.N == 0 || g.nzb * g.nzh == 0) return cudaSuccess;
    dim3 grid(blocks_for(g.N, GT), blocks_for(g.M, GT), g.nzb * g.nzh), block(256);
    ProfScope ps("gemm_simt", st);
    if (dt == MLA_F32) gemm_simt_kernel<float><<<grid, block, 0, st>>>(g);
    else gemm_simt_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_attn_simt(mla_dtype dt, const AttnArgs &a, cudaStream_t st) {
    if (a.n_rows == 0 || a.n_b * a.n_h == 0 || a.n_splits == 0) return cudaSuccess;
    size_t smem = sizeof(float) * AKT * (size_t)(a.D1 + a.D2 + a.Dv);
    dim3 grid(blocks_for(a.n_rows, AW), a.n_b * a.n_h, a.n_splits), block(AW * 32);
    cudaError_t e;
    ProfScope ps("attn_simt", st);
    if (dt == MLA_F32) {
        e = cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attn_simt_kernel<float><<<grid, block, smem, st>>>(a);
    } else {
        e = cudaFuncSetAttribute(attn_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        attn_simt_kernel<__nv_bfloat16><<<grid, block, smem, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_lse_combine(mla_dtype dt, int n, long rows, int D, const float *po,
                               const float *pl, void *out, float *lse, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    dim3 grid(blocks_for(rows, 8)), block(256);
    ProfScope ps("lse_combine", st);
    if (dt == MLA_F32)
        lse_combine_kernel<float><<<grid, block, 0, st>>>(n, rows, D, po, pl, (float *)out, lse);
    else
        lse_combine_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(n, rows, D, po, pl, (__nv_bfloat16 *)out, lse);
    return cudaGetLastError();
}

}  // namespace mla
