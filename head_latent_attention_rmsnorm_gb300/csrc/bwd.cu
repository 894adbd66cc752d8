// bwd.cu -- CUDA-core kernels of the explicit prefill's backward pass (any dimensions up
// to 256 per band, fp32 arithmetic), and the row kernels both backward paths share.
//
// Method ("A Training-Memory Regression in MLA Sequence Parallelism ... LAGA", arXiv
// 2607.17644, "What carries the argument": the sequence-parallel method gives the same
// gradients as the baseline, so the backward pass is part of what it computes).  The
// pages print no backward formulas; these are the chain rule through the forward's
// steps in reverse order, for an upstream gradient dO of the output (the log-sum-exp is
// not differentiated):
//   D_i = dO_i . o_i,  dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i)
//   dq_nope_i = scale sum_j dS_ij K_j,   dq_rot_i = scale sum_j dS_ij k_rot_j
//   dK_j = scale sum_i dS_ij q_nope_i,   dk_rot_j = scale sum_i dS_ij q_rot_i (all heads)
//   dV_j = sum_i P_ij dO_i
//   RoPE's transpose rotates by the opposite angle; the reconstruction's gradients are
//   dW = dKV^T chat and dchat = dKV W; RMSNorm's is dx = dy w / r - x (dy . w x) / (d r^3).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ __forceinline__ float ld_any(const void *p, int ty, long i) {
    if (ty == TY_F32) return ((const float *)p)[i];
    if (ty == TY_BF16) return __bfloat162float(((const __nv_bfloat16 *)p)[i]);
    return __half2float(((const __half *)p)[i]);
}
__device__ __forceinline__ void st_any(void *p, int ty, long i, float v) {
    if (ty == TY_F32) ((float *)p)[i] = v;
    else if (ty == TY_BF16) ((__nv_bfloat16 *)p)[i] = __float2bfloat16_rn(v);
    else ((__half *)p)[i] = __float2half_rn(v);
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
inline unsigned nblocks(long n, int per) { return (unsigned)((n + per - 1) / per); }
// fp32 pair -> packed bf16x2 (low half = first argument), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *(const uint32_t *)&h;
}

constexpr int PL = 8;   // values per lane: bands up to 256 wide

// D[b][h][i] = dO[b][i][h][:] . out[b][i][h][:]  (warp per row)
__global__ void rowdot_kernel(long rows, int hc, int s_q, int Dv, const void *dout, const void *out, int ty, float *D) {
    const long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    float a = 0.f;
    for (int d = lane; d < Dv; d += 32) a = fmaf(ld_any(dout, ty, r * Dv + d), ld_any(out, ty, r * Dv + d), a);
    a = wsum(a);
    // r = (b * s_q + i) * hc + h
    const long h = r % hc, bi = r / hc, i = bi % s_q, b = bi / s_q;
    if (lane == 0) D[(b * hc + h) * s_q + i] = a;
}

// Shard-local views of the tensors both attention-backward kernels read.
struct BwdAttn {
    int B, s_q, hc, h0, nh, Dn, Dr, Dv;
    long kv;          // keys with K/V rows (kv_need)
    long kv_pad;      // row pitch of the rotated k_pe
    int causal;
    long q_off;
    float scale;
    const void *q_nope; int tq;        // [B][s_q][hc][Dn]
    const float *qr;                   // rotated q_pe [B][s_q][hc][Dr]
    const float *K, *V;                // [B][hs][kv][Dn], [B][hs][kv][Dv] (shard)
    long k_b, k_h, v_b, v_h;
    const float *kr;                   // rotated k_pe [B][kv_pad][Dr]
    const float *lse, *D;              // [B][hc][s_q]
    const void *dout; int tdo;         // [B][s_q][hc][Dv]
    void *dq_nope; int tdq;            // [B][s_q][hc][Dn]
    float *dqr;                        // [B][s_q][hc][Dr]
    float *dK, *dV, *dkr;              // [B][hs][kv][Dn|Dv|Dr]
};

// Warp per (batch, shard head, query row): dq_nope and the rotated dq over its visible keys.
__global__ void __launch_bounds__(256) attn_bwd_dq_simt_kernel(BwdAttn a) {
    const int lane = threadIdx.x % 32;
    const long i = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int z = blockIdx.y, b = z / a.nh, hl = z % a.nh, hq = a.h0 + hl;
    if (i >= a.s_q) return;
    const long qrow = ((long)b * a.s_q + i) * a.hc + hq;
    float q[PL], qr[PL], dO[PL], dq[PL], dqr[PL];
#pragma unroll
    for (int k = 0; k < PL; ++k) {
        const int dn = lane + 32 * k, dr = dn, dv = dn;
        q[k] = dn < a.Dn ? ld_any(a.q_nope, a.tq, qrow * a.Dn + dn) : 0.f;
        qr[k] = dr < a.Dr ? a.qr[qrow * a.Dr + dr] : 0.f;
        dO[k] = dv < a.Dv ? ld_any(a.dout, a.tdo, qrow * a.Dv + dv) : 0.f;
        dq[k] = dqr[k] = 0.f;
    }
    const long li = ((long)b * a.hc + hq) * a.s_q + i;
    const float lse = a.lse[li], Di = a.D[li];
    const long pos = a.q_off + i;
    const long n = a.causal ? min(pos + 1, a.kv) : a.kv;
    const float *K = a.K + b * a.k_b + hl * a.k_h, *V = a.V + b * a.v_b + hl * a.v_h;
    const float *kr = a.kr + (long)b * a.kv_pad * a.Dr;
    for (long j = 0; j < n; ++j) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int k = 0; k < PL; ++k) {
            const int d = lane + 32 * k;
            if (d < a.Dn) s = fmaf(q[k], K[j * a.Dn + d], s);
            if (d < a.Dr) s = fmaf(qr[k], kr[j * a.Dr + d], s);
            if (d < a.Dv) dp = fmaf(dO[k], V[j * a.Dv + d], dp);
        }
        s = wsum(s) * a.scale;
        dp = wsum(dp);
        const float p = lse > -INFINITY ? expf(s - lse) : 0.f;
        const float ds = p * (dp - Di) * a.scale;
#pragma unroll
        for (int k = 0; k < PL; ++k) {
            const int d = lane + 32 * k;
            if (d < a.Dn) dq[k] = fmaf(ds, K[j * a.Dn + d], dq[k]);
            if (d < a.Dr) dqr[k] = fmaf(ds, kr[j * a.Dr + d], dqr[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < PL; ++k) {
        const int d = lane + 32 * k;
        if (d < a.Dn) st_any(a.dq_nope, a.tdq, qrow * a.Dn + d, dq[k]);
        if (d < a.Dr) a.dqr[qrow * a.Dr + d] = dqr[k];
    }
}

// Warp per (batch, shard head, key j < kv): dK_j, dV_j and this head's share of dk_rot_j
// over the queries that see key j.
__global__ void __launch_bounds__(256) attn_bwd_dkv_simt_kernel(BwdAttn a) {
    const int lane = threadIdx.x % 32;
    const long j = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int z = blockIdx.y, b = z / a.nh, hl = z % a.nh, hq = a.h0 + hl;
    if (j >= a.kv) return;
    const float *K = a.K + b * a.k_b + hl * a.k_h, *V = a.V + b * a.v_b + hl * a.v_h;
    const float *kr = a.kr + (long)b * a.kv_pad * a.Dr;
    float kk[PL], kkr[PL], vv[PL], dk[PL], dkr[PL], dv[PL];
#pragma unroll
    for (int k = 0; k < PL; ++k) {
        const int d = lane + 32 * k;
        kk[k] = d < a.Dn ? K[j * a.Dn + d] : 0.f;
        kkr[k] = d < a.Dr ? kr[j * a.Dr + d] : 0.f;
        vv[k] = d < a.Dv ? V[j * a.Dv + d] : 0.f;
        dk[k] = dkr[k] = dv[k] = 0.f;
    }
    const long i0 = a.causal ? max(0L, j - a.q_off) : 0;
    for (long i = i0; i < a.s_q; ++i) {
        const long qrow = ((long)b * a.s_q + i) * a.hc + hq;
        const long li = ((long)b * a.hc + hq) * a.s_q + i;
        const float lse = a.lse[li];
        if (!(lse > -INFINITY)) continue;
        float q[PL], qr[PL], dO[PL];
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int k = 0; k < PL; ++k) {
            const int d = lane + 32 * k;
            q[k] = d < a.Dn ? ld_any(a.q_nope, a.tq, qrow * a.Dn + d) : 0.f;
            qr[k] = d < a.Dr ? a.qr[qrow * a.Dr + d] : 0.f;
            dO[k] = d < a.Dv ? ld_any(a.dout, a.tdo, qrow * a.Dv + d) : 0.f;
            s = fmaf(q[k], kk[k], fmaf(qr[k], kkr[k], s));
            dp = fmaf(dO[k], vv[k], dp);
        }
        s = wsum(s) * a.scale;
        dp = wsum(dp);
        const float p = expf(s - lse);
        const float ds = p * (dp - a.D[li]) * a.scale;
#pragma unroll
        for (int k = 0; k < PL; ++k) {
            dk[k] = fmaf(ds, q[k], dk[k]);
            dkr[k] = fmaf(ds, qr[k], dkr[k]);
            dv[k] = fmaf(p, dO[k], dv[k]);
        }
    }
    const long o = ((long)b * a.nh + hl) * a.kv + j;
#pragma unroll
    for (int k = 0; k < PL; ++k) {
        const int d = lane + 32 * k;
        if (d < a.Dn) a.dK[o * a.Dn + d] = dk[k];
        if (d < a.Dv) a.dV[o * a.Dv + d] = dv[k];
        if (d < a.Dr) a.dkr[o * a.Dr + d] = dkr[k];
    }
}

// acc[b][j][d] (+)= sum over the shard's heads of part[b][hl][j][d], in head order.
__global__ void head_sum_kernel(int B, int nh, long kv, int Dr, long acc_pitch, const float *part, float *acc,
                                int accumulate) {
    const long n = (long)B * kv * Dr;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const int d = (int)(x % Dr);
        const long j = (x / Dr) % kv, b = x / (Dr * kv);
        float s = accumulate ? acc[(b * acc_pitch + j) * Dr + d] : 0.f;
        for (int hl = 0; hl < nh; ++hl) s += part[(((long)b * nh + hl) * kv + j) * Dr + d];
        acc[(b * acc_pitch + j) * Dr + d] = s;
    }
}

// y = RoPE(x, -pos) row by row (the transpose of the forward rotation): row r of
// `rows` sits at position pos0 + (r / pos_div) % pos_mod; rows whose position is at or
// beyond `pos_end` are written as zeros.  x fp32 [rows][Dr] with row pitch x_pitch.
__global__ void rope_inv_kernel(long rows, int Dr, const float *x, long x_pitch, long pos0, long pos_div,
                                long pos_mod, long pos_end, const float2 *tab, void *y, int ty, long y_pitch) {
    const long r = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    const long pos = pos0 + (r / pos_div) % pos_mod;
    const int half = Dr / 2;
    for (int t = lane; t < half; t += 32) {
        float y0 = 0.f, y1 = 0.f;
        if (pos < pos_end) {
            const float2 cs = tab[pos * half + t];
            const float x0 = x[r * x_pitch + t], x1 = x[r * x_pitch + t + half];
            y0 = x0 * cs.x + x1 * cs.y;
            y1 = x1 * cs.x - x0 * cs.y;
        }
        st_any(y, ty, r * y_pitch + t, y0);
        st_any(y, ty, r * y_pitch + t + half, y1);
    }
}

// RMSNorm backward with an fp32 upstream gradient: warp per row r < n_rows of one batch
// (x, dx with pitch Dk; dy fp32 with pitch Dk); rows [n_rows, s_kv) of dx are zeros.
// Each block's warps add their dw terms in a fixed order into one partial row.
constexpr int RW = 8;
__global__ void __launch_bounds__(RW * 32) rms_bwd_kernel(long n_rows, long s_kv, int Dk, float eps, const void *x,
                                                          const void *w, int ty, const float *dy, void *dx,
                                                          float *part) {
    extern __shared__ float sm[];   // [RW][Dk] dw terms of this block's warps
    const int lane = threadIdx.x % 32, wi = threadIdx.x / 32;
    for (int k = threadIdx.x; k < RW * Dk; k += blockDim.x) sm[k] = 0.f;
    __syncthreads();
    for (long r = (long)blockIdx.x * RW + wi; r < s_kv; r += (long)gridDim.x * RW) {
        if (r >= n_rows) {
            for (int k = lane; k < Dk; k += 32) st_any(dx, ty, r * Dk + k, 0.f);
            continue;
        }
        float ss = 0.f, g = 0.f;
        for (int k = lane; k < Dk; k += 32) {
            const float xv = ld_any(x, ty, r * Dk + k);
            ss = fmaf(xv, xv, ss);
            g = fmaf(dy[r * Dk + k] * ld_any(w, ty, k), xv, g);
        }
        ss = wsum(ss);
        g = wsum(g);
        const float ri = 1.0f / sqrtf(ss / (float)Dk + eps);
        const float c = g * ri * ri * ri / (float)Dk;
        for (int k = lane; k < Dk; k += 32) {
            const float xv = ld_any(x, ty, r * Dk + k), d = dy[r * Dk + k];
            st_any(dx, ty, r * Dk + k, d * ld_any(w, ty, k) * ri - xv * c);
            sm[wi * Dk + k] += d * xv * ri;
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < Dk; k += blockDim.x) {
        float s = 0.f;
        for (int i = 0; i < RW; ++i) s += sm[i * Dk + k];
        part[(long)blockIdx.x * Dk + k] = s;
    }
}

// The same backward for bf16 x, w, dx with Dk a multiple of 256 and 16-byte aligned rows:
// lane l holds the 8-element pieces l, l + 32, ... of a row (NC = Dk / 256 of them), so
// every load and store is 16 bytes (x, w, dx) or 32 bytes (dy) per lane; the warp's two
// sums reduce together; dw terms stay in registers and the block's warps add them into
// one partial row in a fixed order.
template <int NC>
__global__ void __launch_bounds__(RW * 32) rms_bwd_vec_kernel(long n_rows, long s_kv, float eps, const uint4 *x,
                                                              const uint4 *w, const float4 *dy, uint4 *dx,
                                                              float *part) {
    constexpr int Dk = NC * 256;
    __shared__ float red[Dk];
    const int lane = threadIdx.x % 32, wi = threadIdx.x / 32;
    float acc[NC][8];
    float wf[NC][8];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 q = w[c * 32 + lane];
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wf[c][2 * e] = __uint_as_float(u[e] << 16);
            wf[c][2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[c][t] = 0.f;
    }
    for (long r = (long)blockIdx.x * RW + wi; r < s_kv; r += (long)gridDim.x * RW) {
        if (r >= n_rows) {
#pragma unroll
            for (int c = 0; c < NC; ++c) dx[r * (Dk / 8) + c * 32 + lane] = make_uint4(0, 0, 0, 0);
            continue;
        }
        float xf[NC][8], gf[NC][8];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 q = x[r * (Dk / 8) + c * 32 + lane];
            const float4 g0 = dy[r * (Dk / 4) + 2 * (c * 32 + lane)], g1 = dy[r * (Dk / 4) + 2 * (c * 32 + lane) + 1];
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xf[c][2 * e] = __uint_as_float(u[e] << 16);
                xf[c][2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
            }
            gf[c][0] = g0.x, gf[c][1] = g0.y, gf[c][2] = g0.z, gf[c][3] = g0.w;
            gf[c][4] = g1.x, gf[c][5] = g1.y, gf[c][6] = g1.z, gf[c][7] = g1.w;
        }
        float ss = 0.f, g = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                ss = fmaf(xf[c][t], xf[c][t], ss);
                g = fmaf(gf[c][t] * wf[c][t], xf[c][t], g);
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            g += __shfl_xor_sync(0xffffffffu, g, off);
        }
        const float ri = 1.0f / sqrtf(ss / (float)Dk + eps);
        const float cc = g * ri * ri * ri / (float)Dk;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float y0 = gf[c][2 * e] * wf[c][2 * e] * ri - xf[c][2 * e] * cc;
                const float y1 = gf[c][2 * e + 1] * wf[c][2 * e + 1] * ri - xf[c][2 * e + 1] * cc;
                o[e] = pack_bf16x2(y0, y1);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) acc[c][t] = fmaf(gf[c][t] * xf[c][t], ri, acc[c][t]);
            dx[r * (Dk / 8) + c * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    for (int v = 0; v < RW; ++v) {   // warp v adds its terms: the same order in every run
        if (wi == v)
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int k = (c * 32 + lane) * 8 + t;
                    red[k] = (v == 0 ? 0.f : red[k]) + acc[c][t];
                }
        __syncthreads();
    }
    for (int k = threadIdx.x; k < Dk; k += blockDim.x) part[(long)blockIdx.x * Dk + k] = red[k];
}

// dw[k] (+)= sum of the partial rows: thread (gi, c) of a block of 32 x 32 sums the fixed
// run of parts [gi * n / 32, (gi + 1) * n / 32) of column k = 32 blockIdx.x + c, then the 32
// run sums are added in order (the same order in every run).
__global__ void __launch_bounds__(1024) part_sum_kernel(int nparts, int Dk, const float *part, float *dw,
                                                        int accumulate) {
    __shared__ float s32[32][33];
    const int c = threadIdx.x % 32, gi = threadIdx.x / 32, k = blockIdx.x * 32 + c;
    float s = 0.f;
    if (k < Dk)
        for (int i = gi * nparts / 32; i < (gi + 1) * nparts / 32; ++i) s += part[(long)i * Dk + k];
    s32[gi][c] = s;
    __syncthreads();
    if (gi == 0 && k < Dk) {
        float t = accumulate ? dw[k] : 0.f;
        for (int j = 0; j < 32; ++j) t += s32[j][c];
        dw[k] = t;
    }
}

}  // namespace

cudaError_t launch_bwd_rowdot(int ty, int B, int s_q, int hc, int Dv, const void *dout, const void *out, float *D,
                              cudaStream_t st) {
    const long rows = (long)B * s_q * hc;
    if (rows == 0) return cudaSuccess;
    ProfScope ps("bwd_rowdot", st);
    rowdot_kernel<<<nblocks(rows, 8), 256, 0, st>>>(rows, hc, s_q, Dv, dout, out, ty, D);
    return cudaGetLastError();
}

bool bwd_simt_supported(int Dn, int Dr, int Dv) { return Dn <= 32 * PL && Dr <= 32 * PL && Dv <= 32 * PL; }

cudaError_t launch_attn_bwd_simt(const BwdSimtArgs &s, cudaStream_t st) {
    BwdAttn a{};
    a.B = s.B; a.s_q = s.s_q; a.hc = s.hc; a.h0 = s.h0; a.nh = s.nh;
    a.Dn = s.Dn; a.Dr = s.Dr; a.Dv = s.Dv; a.kv = s.kv; a.kv_pad = s.kv_pad;
    a.causal = s.causal; a.q_off = s.q_off; a.scale = s.scale;
    a.q_nope = s.q_nope; a.tq = s.ty; a.qr = s.qr;
    a.K = s.K; a.V = s.V; a.k_b = s.k_b; a.k_h = s.k_h; a.v_b = s.v_b; a.v_h = s.v_h;
    a.kr = s.kr; a.lse = s.lse; a.D = s.D; a.dout = s.dout; a.tdo = s.ty;
    a.dq_nope = s.dq_nope; a.tdq = s.ty; a.dqr = s.dqr;
    a.dK = s.dK; a.dV = s.dV; a.dkr = s.dkr;
    if ((long)s.B * s.nh == 0) return cudaSuccess;
    {
        ProfScope ps("attn_bwd_simt", st);
        if (s.s_q > 0) attn_bwd_dq_simt_kernel<<<dim3(nblocks(s.s_q, 8), s.B * s.nh), 256, 0, st>>>(a);
        if (s.kv > 0) attn_bwd_dkv_simt_kernel<<<dim3(nblocks(s.kv, 8), s.B * s.nh), 256, 0, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_head_sum(int B, int nh, long kv, int Dr, long acc_pitch, const float *part, float *acc,
                            bool accumulate, cudaStream_t st) {
    const long n = (long)B * kv * Dr;
    if (n == 0) return cudaSuccess;
    ProfScope ps("bwd_rows", st);
    head_sum_kernel<<<std::min<long>(nblocks(n, 256), 2048), 256, 0, st>>>(B, nh, kv, Dr, acc_pitch, part, acc,
                                                                           accumulate ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_rope_inv(long rows, int Dr, const float *x, long x_pitch, long pos0, long pos_div, long pos_mod,
                            long pos_end, const float2 *tab, void *y, int ty, long y_pitch, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    ProfScope ps("bwd_rows", st);
    rope_inv_kernel<<<nblocks(rows, 8), 256, 0, st>>>(rows, Dr, x, x_pitch, pos0, pos_div, pos_mod, pos_end, tab, y, ty,
                                                      y_pitch);
    return cudaGetLastError();
}

// Partial dw rows: at most 128, so that the ordered sum over them stays short; each block
// walks s_kv / (parts * RW) rows per warp.
size_t rms_bwd_parts(long s_kv) { return (size_t)std::max<long>(1, std::min<long>(304, (s_kv + RW - 1) / RW)); }

cudaError_t launch_rms_bwd_f32dy(int ty, long n_rows, long s_kv, int Dk, float eps, const void *x, const void *w,
                                 const float *dy, void *dx, float *dw, bool accumulate, float *part,
                                 cudaStream_t st) {
    const unsigned nb = (unsigned)rms_bwd_parts(s_kv);
    const size_t smem = sizeof(float) * RW * Dk;
    cudaError_t e = cudaFuncSetAttribute(rms_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope ps("bwd_rows", st);
    const bool vec = ty == TY_BF16 && (Dk == 256 || Dk == 512 || Dk == 1024) && ((uintptr_t)x & 15) == 0 &&
                     ((uintptr_t)w & 15) == 0 && ((uintptr_t)dy & 15) == 0 && ((uintptr_t)dx & 15) == 0;
    if (s_kv > 0 && vec) {
        const uint4 *xv = (const uint4 *)x, *wv = (const uint4 *)w;
        const float4 *gv = (const float4 *)dy;
        uint4 *dxv = (uint4 *)dx;
        if (Dk == 256) rms_bwd_vec_kernel<1><<<nb, RW * 32, 0, st>>>(n_rows, s_kv, eps, xv, wv, gv, dxv, part);
        if (Dk == 512) rms_bwd_vec_kernel<2><<<nb, RW * 32, 0, st>>>(n_rows, s_kv, eps, xv, wv, gv, dxv, part);
        if (Dk == 1024) rms_bwd_vec_kernel<4><<<nb, RW * 32, 0, st>>>(n_rows, s_kv, eps, xv, wv, gv, dxv, part);
    } else if (s_kv > 0) {
        rms_bwd_kernel<<<nb, RW * 32, smem, st>>>(n_rows, s_kv, Dk, eps, x, w, ty, dy, dx, part);
    }
    part_sum_kernel<<<nblocks(Dk, 32), 1024, 0, st>>>(s_kv > 0 ? (int)nb : 0, Dk, part, dw, accumulate ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace mla
