// SIMT (fp32 FFMA) kernels for the Parallax attention layer.
//
// These serve dtype=fp32 (tensor-core precision would not meet an fp32
// tolerance) and are a reference-quality fallback for bf16 inputs, which are
// widened to fp32 on load.  All arithmetic is fp32.
//
// Layer ("Parallax: Parameterized Local Linear Attention for Language
// Modeling", technical summary, "Core mechanism"; probe u = P_h (q - mu_k)):
//   pass 1      : lse_t, mu_k,t = sum_i p_ti k_i          (online softmax over key tiles)
//   projection  : u_t = P_h (q_t - mu_k,t), gbar_t = mu_k,t . u_t
//   pass 2      : o_t = sum_i p_ti (1 + k_i.u_t - gbar_t) v_i   (p from the stored lse)
// The pass-2 weights p (1 + g - gbar) fold the rank-1 mean term of
// o = mu_v + sum p g v - gbar mu_v into the value contraction, so no mu_v is
// needed.
//
// Backward (chain rule of the lines above, e_ti = do_t . v_i):
//   B1 (query tiles): R_t = sum_i p e k_i,  ebar_t = sum_i p e
//   B2 (rows)       : du = R - ebar mu_k; ddelta = P^T du; dq = ddelta; dmu = -ddelta;
//                     D = do.o - gbar ebar + mu_k.dmu, with do.o = ebar + R.u - gbar ebar
//                     rebuilt from the fp32 sums (sum_i p e (1 + g - gbar), g = k.u), so
//                     the stored (possibly bf16) output is never read
//   dP (rows)       : dP_h = sum_{b,t} du delta^T   (fixed-order two-stage reduction)
//   B3 (key tiles)  : a = p(1+g-gbar), dg = p(e-ebar), ds = p(e(1+g-gbar) - g ebar + k.dmu - D)
//                     dv += a do; dk += c ds q + dg u + p dmu; dq += c ds k (fp32 atomics)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "plx_internal.h"

namespace plx {
namespace {

constexpr int NT = 256;   // threads per CTA (16 x 16 thread grid)
constexpr int BQ = 64;    // query rows per tile
constexpr int BK = 64;    // keys per tile
constexpr int LDS = BK + 1;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Load a [rows x D] tile starting at row r0 of a [T x D] head into padded smem
// (row stride D+1); rows >= T are zero.
template <typename Tin, int D>
__device__ __forceinline__ void load_tile(float* dst, const Tin* src, int r0, int rows, int T) {
    for (int e = threadIdx.x; e < rows * D; e += NT) {
        const int r = e / D, c = e % D;
        const int t = r0 + r;
        dst[r * (D + 1) + c] = t < T ? ldf(src + (size_t)t * D + c) : 0.f;
    }
}

// ------------------------------------------------------------------ pass 1
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_pass1(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                 float* __restrict__ lse, float* __restrict__ mu_k,
                                                 int T, float scale_log2) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NJ = D / 16;
    float* Qs = sm;
    float* Ks = Qs + BQ * LD;
    float* Ss = Ks + BK * LD;
    float* mrow = Ss + BQ * LDS;
    float* lrow = mrow + BQ;
    float* arow = lrow + BQ;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int qt = blockIdx.x;
    const size_t head = blockIdx.y;
    const Tin* Q = q + head * T * D;
    const Tin* K = k + head * T * D;
    const int q0 = qt * BQ;

    load_tile<Tin, D>(Qs, Q, q0, BQ, T);
    if (tid < BQ) { mrow[tid] = -INFINITY; lrow[tid] = 0.f; }
    float acc[4][NJ];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < NJ; j++) acc[i][j] = 0.f;

    const int nkt = min(qt, (T - 1) / BK);
    for (int kt = 0; kt <= nkt; kt++) {
        const int k0 = kt * BK;
        __syncthreads();
        load_tile<Tin, D>(Ks, K, k0, BK, T);
        __syncthreads();
        float s[4][4] = {};
        for (int kk = 0; kk < D; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = Qs[(ty + 16 * i) * LD + kk];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Ks[(tx + 16 * j) * LD + kk];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) s[i][j] = fmaf(a[i], b[j], s[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                const int t = q0 + r, key = k0 + c;
                Ss[r * LDS + c] = (key <= t && key < T) ? s[i][j] * scale_log2 : -INFINITY;
            }
        __syncthreads();
        {
            const int r = tid >> 2, part = tid & 3;
            float* srow = Ss + r * LDS + part * 16;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 16; c++) mx = fmaxf(mx, srow[c]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mold = mrow[r];
            const float mnew = fmaxf(mold, mx);
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 16; c++) {
                const float p = (mnew == -INFINITY) ? 0.f : exp2f(srow[c] - mnew);
                srow[c] = p;
                sum += p;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            const float alpha = (mold == -INFINITY) ? 0.f : exp2f(mold - mnew);
            __syncwarp();
            if (part == 0) {
                mrow[r] = mnew;
                lrow[r] = lrow[r] * alpha + sum;
                arow[r] = alpha;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float al = arow[ty + 16 * i];
#pragma unroll
            for (int j = 0; j < NJ; j++) acc[i][j] *= al;
        }
        for (int c = 0; c < BK; c++) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = Ss[(ty + 16 * i) * LDS + c];
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                const float b = Ks[c * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; i++) acc[i][j] = fmaf(a[i], b, acc[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int r = ty + 16 * i, t = q0 + r;
        if (t < T) {
            const float inv = 1.f / lrow[r];
            const size_t row = head * T + t;
#pragma unroll
            for (int j = 0; j < NJ; j++) mu_k[row * D + tx + 16 * j] = acc[i][j] * inv;
            if (tx == 0) lse[row] = (mrow[r] + log2f(lrow[r])) * LN2;
        }
    }
}

// ------------------------------------------------------------- projection
// u = P_h (q - mu_k), gbar = mu_k . u.  P_h is staged transposed with a
// padded row so that both u = P delta and P^T du read conflict-free.
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_proj(const Tin* __restrict__ q, const float* __restrict__ mu_k,
                                                const float* __restrict__ P, float* __restrict__ U,
                                                float* __restrict__ gbar, int B, int H, int T, int rows_per_cta) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NA = D / 32;
    float* PT = sm;            // PT[b][a] = P[a][b]
    float* dl = PT + D * LD;   // per-warp delta buffer [8][D]
    const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* Ph = P + (size_t)h * D * D;
    for (int e = threadIdx.x; e < D * D; e += NT) {
        const int a = e / D, b = e % D;
        PT[b * LD + a] = Ph[e];
    }
    __syncthreads();
    float* dw = dl + warp * D;
    const int r_begin = blockIdx.x * rows_per_cta;
    const int r_end = min(r_begin + rows_per_cta, B * T);
    for (int r = r_begin + warp; r < r_end; r += NT / 32) {
        const int b = r / T, t = r % T;
        const size_t row = ((size_t)b * H + h) * T + t;
        float mk[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) {
            const int a = lane + 32 * j;
            mk[j] = mu_k[row * D + a];
            dw[a] = ldf(q + row * D + a) - mk[j];
        }
        __syncwarp();
        float u[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) u[j] = 0.f;
        for (int bb = 0; bb < D; bb++) {
            const float db = dw[bb];
#pragma unroll
            for (int j = 0; j < NA; j++) u[j] = fmaf(PT[bb * LD + lane + 32 * j], db, u[j]);
        }
        float g = 0.f;
#pragma unroll
        for (int j = 0; j < NA; j++) {
            U[row * D + lane + 32 * j] = u[j];
            g = fmaf(mk[j], u[j], g);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
        if (lane == 0) gbar[row] = g;
        __syncwarp();
    }
}

// ------------------------------------------------------------------ pass 2
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_pass2(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                 const Tin* __restrict__ v, const float* __restrict__ U,
                                                 const float* __restrict__ gbar, const float* __restrict__ lse,
                                                 Tin* __restrict__ out, int T, float scale_log2) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NJ = D / 16;
    float* Qs = sm;
    float* Us = Qs + BQ * LD;
    float* Ks = Us + BQ * LD;
    float* Vs = Ks + BK * LD;
    float* Ws = Vs + BK * LD;
    float* L2 = Ws + BQ * LDS;
    float* G1 = L2 + BQ;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int qt = blockIdx.x;
    const size_t head = blockIdx.y;
    const int q0 = qt * BQ;
    load_tile<Tin, D>(Qs, q + head * T * D, q0, BQ, T);
    load_tile<float, D>(Us, U + head * T * D, q0, BQ, T);
    if (tid < BQ) {
        const int t = q0 + tid;
        L2[tid] = t < T ? lse[head * T + t] * LOG2E : 0.f;
        G1[tid] = t < T ? 1.f - gbar[head * T + t] : 0.f;
    }
    float acc[4][NJ];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < NJ; j++) acc[i][j] = 0.f;
    const int nkt = min(qt, (T - 1) / BK);
    for (int kt = 0; kt <= nkt; kt++) {
        const int k0 = kt * BK;
        __syncthreads();
        load_tile<Tin, D>(Ks, k + head * T * D, k0, BK, T);
        load_tile<Tin, D>(Vs, v + head * T * D, k0, BK, T);
        __syncthreads();
        float s[4][4] = {}, g[4][4] = {};
        for (int kk = 0; kk < D; kk++) {
            float aq[4], au[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                aq[i] = Qs[(ty + 16 * i) * LD + kk];
                au[i] = Us[(ty + 16 * i) * LD + kk];
            }
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Ks[(tx + 16 * j) * LD + kk];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    s[i][j] = fmaf(aq[i], b[j], s[i][j]);
                    g[i][j] = fmaf(au[i], b[j], g[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                const int t = q0 + r, key = k0 + c;
                float w = 0.f;
                if (key <= t && key < T) {
                    const float p = exp2f(s[i][j] * scale_log2 - L2[r]);
                    w = p * (g[i][j] + G1[r]);
                }
                Ws[r * LDS + c] = w;
            }
        __syncthreads();
        for (int c = 0; c < BK; c++) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = Ws[(ty + 16 * i) * LDS + c];
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                const float bv = Vs[c * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; i++) acc[i][j] = fmaf(a[i], bv, acc[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int t = q0 + ty + 16 * i;
        if (t < T) {
            const size_t row = head * T + t;
#pragma unroll
            for (int j = 0; j < NJ; j++) stf(out + row * D + tx + 16 * j, acc[i][j]);
        }
    }
}

// ---------------------------------------------------------------- bwd B1
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_bwd_b1(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                  const Tin* __restrict__ v, const Tin* __restrict__ dout,
                                                  const float* __restrict__ lse, float* __restrict__ R,
                                                  float* __restrict__ ebar, int T, float scale_log2) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NJ = D / 16;
    float* Qs = sm;
    float* Os = Qs + BQ * LD;  // dO
    float* Ks = Os + BQ * LD;
    float* Vs = Ks + BK * LD;
    float* Ws = Vs + BK * LD;
    float* L2 = Ws + BQ * LDS;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int qt = blockIdx.x;
    const size_t head = blockIdx.y;
    const int q0 = qt * BQ;
    load_tile<Tin, D>(Qs, q + head * T * D, q0, BQ, T);
    load_tile<Tin, D>(Os, dout + head * T * D, q0, BQ, T);
    if (tid < BQ) {
        const int t = q0 + tid;
        L2[tid] = t < T ? lse[head * T + t] * LOG2E : 0.f;
    }
    float acc[4][NJ], es[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < NJ; j++) acc[i][j] = 0.f;
    const int nkt = min(qt, (T - 1) / BK);
    for (int kt = 0; kt <= nkt; kt++) {
        const int k0 = kt * BK;
        __syncthreads();
        load_tile<Tin, D>(Ks, k + head * T * D, k0, BK, T);
        load_tile<Tin, D>(Vs, v + head * T * D, k0, BK, T);
        __syncthreads();
        float s[4][4] = {}, e[4][4] = {};
        for (int kk = 0; kk < D; kk++) {
            float aq[4], ao[4], bk[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                aq[i] = Qs[(ty + 16 * i) * LD + kk];
                ao[i] = Os[(ty + 16 * i) * LD + kk];
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                bk[j] = Ks[(tx + 16 * j) * LD + kk];
                bv[j] = Vs[(tx + 16 * j) * LD + kk];
            }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    s[i][j] = fmaf(aq[i], bk[j], s[i][j]);
                    e[i][j] = fmaf(ao[i], bv[j], e[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                const int t = q0 + r, key = k0 + c;
                float w = 0.f;
                if (key <= t && key < T) w = exp2f(s[i][j] * scale_log2 - L2[r]) * e[i][j];
                Ws[r * LDS + c] = w;
                es[i] += w;
            }
        __syncthreads();
        for (int c = 0; c < BK; c++) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = Ws[(ty + 16 * i) * LDS + c];
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                const float b = Ks[c * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; i++) acc[i][j] = fmaf(a[i], b, acc[i][j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float x = es[i];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        es[i] = x;  // the 16 lanes sharing ty now hold the row sum
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int t = q0 + ty + 16 * i;
        if (t < T) {
            const size_t row = head * T + t;
#pragma unroll
            for (int j = 0; j < NJ; j++) R[row * D + tx + 16 * j] = acc[i][j];
            if (tx == 0) ebar[row] = es[i];
        }
    }
}

// ---------------------------------------------------------------- bwd B2
// Per row: delta, u, gbar, du (overwrites R), ddelta = P^T du, dq_acc = ddelta,
// dmu = -ddelta, D = (ebar + R.u - gbar ebar) - gbar ebar + mu_k.dmu.
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_bwd_b2(const Tin* __restrict__ q, const float* __restrict__ mu_k,
                                                  const float* __restrict__ P, float* __restrict__ R,
                                                  const float* __restrict__ ebar, float* __restrict__ U,
                                                  float* __restrict__ dmu, float* __restrict__ dq_acc,
                                                  float* __restrict__ gbar, float* __restrict__ Dv,
                                                  int B, int H, int T, int rows_per_cta) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NA = D / 32;
    float* PT = sm;
    float* buf = PT + D * LD;  // per-warp [D]
    const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* Ph = P + (size_t)h * D * D;
    for (int e = threadIdx.x; e < D * D; e += NT) {
        const int a = e / D, b = e % D;
        PT[b * LD + a] = Ph[e];
    }
    __syncthreads();
    float* w = buf + warp * D;
    const int r_begin = blockIdx.x * rows_per_cta;
    const int r_end = min(r_begin + rows_per_cta, B * T);
    for (int r = r_begin + warp; r < r_end; r += NT / 32) {
        const int b = r / T, t = r % T;
        const size_t row = ((size_t)b * H + h) * T + t;
        float mk[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) {
            const int a = lane + 32 * j;
            mk[j] = mu_k[row * D + a];
            w[a] = ldf(q + row * D + a) - mk[j];
        }
        __syncwarp();
        float u[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) u[j] = 0.f;
        for (int bb = 0; bb < D; bb++) {
            const float db = w[bb];
#pragma unroll
            for (int j = 0; j < NA; j++) u[j] = fmaf(PT[bb * LD + lane + 32 * j], db, u[j]);
        }
        const float eb = ebar[row];
        float g = 0.f, ru = 0.f, du[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) {
            const int a = lane + 32 * j;
            const float r = R[row * D + a];
            g = fmaf(mk[j], u[j], g);
            ru = fmaf(r, u[j], ru);
            du[j] = r - eb * mk[j];
            U[row * D + a] = u[j];
            R[row * D + a] = du[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            ru += __shfl_xor_sync(0xffffffffu, ru, o);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NA; j++) w[lane + 32 * j] = du[j];
        __syncwarp();
        // ddelta[b] = sum_a P[a][b] du[a] = sum_a PT[b][a] du[a]
        float dd[NA];
#pragma unroll
        for (int j = 0; j < NA; j++) dd[j] = 0.f;
        for (int a = 0; a < D; a++) {
            const float da = w[a];
#pragma unroll
            for (int j = 0; j < NA; j++) dd[j] = fmaf(PT[(lane + 32 * j) * LD + a], da, dd[j]);
        }
        float x = 0.f;
#pragma unroll
        for (int j = 0; j < NA; j++) {
            const int a = lane + 32 * j;
            dq_acc[row * D + a] = dd[j];
            dmu[row * D + a] = -dd[j];
            x = fmaf(mk[j], -dd[j], x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) {
            gbar[row] = g;
            Dv[row] = (eb + ru - g * eb) - g * eb + x;
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ dP
// Stage 1: partial[h][chunk] = sum over the chunk's rows of du delta^T.
template <typename Tin, int D>
__global__ void __launch_bounds__(NT) simt_dp_partial(const Tin* __restrict__ q, const float* __restrict__ mu_k,
                                                      const float* __restrict__ du, float* __restrict__ partial,
                                                      int B, int H, int T, int rows_per_chunk) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NI = D / 16;
    constexpr int RB = 32;  // rows staged at a time
    float* Us = sm;             // du rows  [RB][LD]
    float* Ds = Us + RB * LD;   // delta rows
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int h = blockIdx.y, chunk = blockIdx.x;
    float acc[NI][NI];
#pragma unroll
    for (int i = 0; i < NI; i++)
#pragma unroll
        for (int j = 0; j < NI; j++) acc[i][j] = 0.f;
    const int r_begin = chunk * rows_per_chunk;
    const int r_end = min(r_begin + rows_per_chunk, B * T);
    for (int r0 = r_begin; r0 < r_end; r0 += RB) {
        __syncthreads();
        for (int e = tid; e < RB * D; e += NT) {
            const int rr = e / D, c = e % D, r = r0 + rr;
            float a = 0.f, dlt = 0.f;
            if (r < r_end) {
                const int b = r / T, t = r % T;
                const size_t row = ((size_t)b * H + h) * T + t;
                a = du[row * D + c];
                dlt = ldf(q + row * D + c) - mu_k[row * D + c];
            }
            Us[rr * LD + c] = a;
            Ds[rr * LD + c] = dlt;
        }
        __syncthreads();
        for (int rr = 0; rr < RB; rr++) {
            float a[NI], b[NI];
#pragma unroll
            for (int i = 0; i < NI; i++) a[i] = Us[rr * LD + ty + 16 * i];
#pragma unroll
            for (int j = 0; j < NI; j++) b[j] = Ds[rr * LD + tx + 16 * j];
#pragma unroll
            for (int i = 0; i < NI; i++)
#pragma unroll
                for (int j = 0; j < NI; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    float* dst = partial + ((size_t)h * gridDim.x + chunk) * D * D;
#pragma unroll
    for (int i = 0; i < NI; i++)
#pragma unroll
        for (int j = 0; j < NI; j++) dst[(ty + 16 * i) * D + tx + 16 * j] = acc[i][j];
}

// Stage 2: dP[h] = sum over chunks in index order.
__global__ void simt_dp_reduce(const float* __restrict__ partial, float* __restrict__ dP, int nchunks, int dd) {
    const int h = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= dd) return;
    const float* src = partial + (size_t)h * nchunks * dd + e;
    float s = 0.f;
    for (int c = 0; c < nchunks; c++) s += src[(size_t)c * dd];
    dP[(size_t)h * dd + e] = s;
}

// ---------------------------------------------------------------- bwd B3
template <typename Tin, int D, int BM>
__global__ void __launch_bounds__(NT) simt_bwd_b3(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                  const Tin* __restrict__ v, const Tin* __restrict__ dout,
                                                  const float* __restrict__ lse, const float* __restrict__ U,
                                                  const float* __restrict__ dmu, const float* __restrict__ gbar,
                                                  const float* __restrict__ ebar, const float* __restrict__ Dv,
                                                  float* __restrict__ dq_acc, Tin* __restrict__ dk,
                                                  Tin* __restrict__ dv, int T, float scale, float scale_log2) {
    extern __shared__ float sm[];
    constexpr int LD = D + 1, NJ = D / 16, MI = BM / 16;
    float* Ks = sm;
    float* Vs = Ks + BK * LD;
    float* Qs = Vs + BK * LD;
    float* Us = Qs + BM * LD;
    float* Os = Us + BM * LD;   // dO
    float* Ms = Os + BM * LD;   // dmu
    float* Ps = Ms + BM * LD;   // p
    float* As = Ps + BM * LDS;  // a
    float* Gs = As + BM * LDS;  // dg
    float* Ss = Gs + BM * LDS;  // ds
    float* rl = Ss + BM * LDS;  // per-row: L2, 1-gbar, ebar, gbar, D
    float* r1 = rl + BM;
    float* re = r1 + BM;
    float* rg = re + BM;
    float* rd = rg + BM;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int kt = blockIdx.x;
    const size_t head = blockIdx.y;
    const int k0 = kt * BK;
    const size_t hb = head * T * D;
    load_tile<Tin, D>(Ks, k + hb, k0, BK, T);
    load_tile<Tin, D>(Vs, v + hb, k0, BK, T);
    float dK[4][NJ], dV[4][NJ];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < NJ; j++) { dK[i][j] = 0.f; dV[i][j] = 0.f; }
    const int nq = (T + BM - 1) / BM;
    for (int qt = k0 / BM; qt < nq; qt++) {
        const int q0 = qt * BM;
        __syncthreads();
        load_tile<Tin, D>(Qs, q + hb, q0, BM, T);
        load_tile<float, D>(Us, U + hb, q0, BM, T);
        load_tile<Tin, D>(Os, dout + hb, q0, BM, T);
        load_tile<float, D>(Ms, dmu + hb, q0, BM, T);
        if (tid < BM) {
            const int t = q0 + tid;
            const bool ok = t < T;
            const size_t row = head * T + t;
            rl[tid] = ok ? lse[row] * LOG2E : 0.f;
            rg[tid] = ok ? gbar[row] : 0.f;
            r1[tid] = ok ? 1.f - gbar[row] : 0.f;
            re[tid] = ok ? ebar[row] : 0.f;
            rd[tid] = ok ? Dv[row] : 0.f;
        }
        __syncthreads();
        float s[MI][4] = {}, g[MI][4] = {}, e[MI][4] = {}, y[MI][4] = {};
        for (int kk = 0; kk < D; kk++) {
            float aq[MI], au[MI], ao[MI], am[MI], bk[4], bv[4];
#pragma unroll
            for (int i = 0; i < MI; i++) {
                const int o = (ty + 16 * i) * LD + kk;
                aq[i] = Qs[o]; au[i] = Us[o]; ao[i] = Os[o]; am[i] = Ms[o];
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                bk[j] = Ks[(tx + 16 * j) * LD + kk];
                bv[j] = Vs[(tx + 16 * j) * LD + kk];
            }
#pragma unroll
            for (int i = 0; i < MI; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    s[i][j] = fmaf(aq[i], bk[j], s[i][j]);
                    g[i][j] = fmaf(au[i], bk[j], g[i][j]);
                    e[i][j] = fmaf(ao[i], bv[j], e[i][j]);
                    y[i][j] = fmaf(am[i], bk[j], y[i][j]);
                }
        }
#pragma unroll
        for (int i = 0; i < MI; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int r = ty + 16 * i, c = tx + 16 * j;
                const int t = q0 + r, key = k0 + c;
                float p = 0.f, a = 0.f, dg = 0.f, ds = 0.f;
                if (key <= t && t < T && key < T) {
                    p = exp2f(s[i][j] * scale_log2 - rl[r]);
                    const float w1 = g[i][j] + r1[r];  // 1 + g - gbar
                    a = p * w1;
                    dg = p * (e[i][j] - re[r]);
                    ds = p * (e[i][j] * w1 - g[i][j] * re[r] + y[i][j] - rd[r]);
                }
                const int o = r * LDS + c;
                Ps[o] = p; As[o] = a; Gs[o] = dg; Ss[o] = ds;
            }
        __syncthreads();
        // dV += a^T dO ; dK += c ds^T Q + dg^T U + p^T dmu
        for (int r = 0; r < BM; r++) {
            float pa[4], pp[4], pg[4], ps[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int o = r * LDS + ty + 16 * i;
                pa[i] = As[o]; pp[i] = Ps[o]; pg[i] = Gs[o]; ps[i] = Ss[o] * scale;
            }
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                const int o = r * LD + tx + 16 * j;
                const float xo = Os[o], xq = Qs[o], xu = Us[o], xm = Ms[o];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    dV[i][j] = fmaf(pa[i], xo, dV[i][j]);
                    dK[i][j] = fmaf(ps[i], xq, fmaf(pg[i], xu, fmaf(pp[i], xm, dK[i][j])));
                }
            }
        }
        // dQ += c ds K  (atomics into the fp32 accumulator)
        float dq[MI][NJ];
#pragma unroll
        for (int i = 0; i < MI; i++)
#pragma unroll
            for (int j = 0; j < NJ; j++) dq[i][j] = 0.f;
        for (int c = 0; c < BK; c++) {
            float a[MI];
#pragma unroll
            for (int i = 0; i < MI; i++) a[i] = Ss[(ty + 16 * i) * LDS + c];
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                const float b = Ks[c * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < MI; i++) dq[i][j] = fmaf(a[i], b, dq[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < MI; i++) {
            const int t = q0 + ty + 16 * i;
            if (t < T) {
                float* dst = dq_acc + (head * T + t) * D;
#pragma unroll
                for (int j = 0; j < NJ; j++) atomicAdd(dst + tx + 16 * j, dq[i][j] * scale);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int key = k0 + ty + 16 * i;
        if (key < T) {
            const size_t row = head * T + key;
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                stf(dk + row * D + tx + 16 * j, dK[i][j]);
                stf(dv + row * D + tx + 16 * j, dV[i][j]);
            }
        }
    }
}

template <typename Tout>
__global__ void cast_rows(const float* __restrict__ src, Tout* __restrict__ dst, size_t n) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) stf(dst + i, src[i]);
}

// ----------------------------------------------------------------- launch
constexpr int PROJ_ROWS = 128;
constexpr int DP_ROWS = 256;

template <int D>
size_t smem_pass1() { return sizeof(float) * (2 * 64 * (D + 1) + 64 * LDS + 3 * 64); }
template <int D>
size_t smem_pass2() { return sizeof(float) * (4 * 64 * (D + 1) + 64 * LDS + 2 * 64); }
template <int D>
size_t smem_proj() { return sizeof(float) * (D * (D + 1) + 8 * D); }
template <int D>
size_t smem_b1() { return sizeof(float) * (4 * 64 * (D + 1) + 64 * LDS + 64); }
template <int D>
size_t smem_dp() { return sizeof(float) * (2 * 32 * (D + 1)); }
template <int D, int BM>
size_t smem_b3() { return sizeof(float) * (2 * BK * (D + 1) + 4 * BM * (D + 1) + 4 * BM * LDS + 5 * BM); }

template <typename F>
cudaError_t set_smem(F* f, size_t bytes) {
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

#define PLX_TRY(x)                         \
    do {                                   \
        cudaError_t e_ = (x);              \
        if (e_ != cudaSuccess) return e_;  \
    } while (0)

struct FwdWs {
    float* U;
    float* gbar;
};
FwdWs fwd_ws(void* ws, int B, int H, int T, int d) {
    const size_t nd = (size_t)B * H * T * d;
    char* p = (char*)ws;
    FwdWs w;
    w.U = (float*)p;
    p += align256(nd * 4);
    w.gbar = (float*)p;
    return w;
}

struct BwdWs {
    float *R, *U, *dmu, *dq_acc, *ebar, *gbar, *Dv, *partial;
    int nchunks;
};
BwdWs bwd_ws(void* ws, int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T, nd = n * d;
    char* p = (char*)ws;
    BwdWs w;
    w.R = (float*)p; p += align256(nd * 4);
    w.U = (float*)p; p += align256(nd * 4);
    w.dmu = (float*)p; p += align256(nd * 4);
    w.dq_acc = (float*)p; p += align256(nd * 4);
    w.ebar = (float*)p; p += align256(n * 4);
    w.gbar = (float*)p; p += align256(n * 4);
    w.Dv = (float*)p; p += align256(n * 4);
    w.nchunks = (B * T + DP_ROWS - 1) / DP_ROWS;
    w.partial = (float*)p;
    return w;
}

template <typename Tin, int D>
cudaError_t fwd_impl(const FwdArgs& a) {
    const float scale_log2 = LOG2E / sqrtf((float)D);
    FwdWs w = fwd_ws(a.ws, a.B, a.H, a.T, a.d);
    const dim3 grid((a.T + BQ - 1) / BQ, a.B * a.H);
    PLX_TRY(set_smem(simt_pass1<Tin, D>, smem_pass1<D>()));
    timing_begin(a.stream, "simt_pass1");
    simt_pass1<Tin, D><<<grid, NT, smem_pass1<D>(), a.stream>>>(
        (const Tin*)a.q, (const Tin*)a.k, a.lse, a.mu_k, a.T, scale_log2);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    PLX_TRY(set_smem(simt_proj<Tin, D>, smem_proj<D>()));
    const dim3 pgrid((a.B * a.T + PROJ_ROWS - 1) / PROJ_ROWS, a.H);
    timing_begin(a.stream, "simt_proj");
    simt_proj<Tin, D><<<pgrid, NT, smem_proj<D>(), a.stream>>>(
        (const Tin*)a.q, a.mu_k, a.P, w.U, w.gbar, a.B, a.H, a.T, PROJ_ROWS);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    PLX_TRY(set_smem(simt_pass2<Tin, D>, smem_pass2<D>()));
    timing_begin(a.stream, "simt_pass2");
    simt_pass2<Tin, D><<<grid, NT, smem_pass2<D>(), a.stream>>>(
        (const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v, w.U, w.gbar, a.lse, (Tin*)a.out, a.T, scale_log2);
    timing_end(a.stream);
    return cudaGetLastError();
}

// B2, dP, B3 and the dq cast; expects R and ebar (B1's outputs) in the workspace.
template <typename Tin, int D>
cudaError_t bwd_rest_impl(const BwdArgs& a) {
    constexpr int BM = D == 128 ? 32 : 64;
    const float scale = 1.f / sqrtf((float)D);
    const float scale_log2 = LOG2E * scale;
    BwdWs w = bwd_ws(a.ws, a.B, a.H, a.T, a.d);
    PLX_TRY(set_smem(simt_bwd_b2<Tin, D>, smem_proj<D>()));
    const dim3 pgrid((a.B * a.T + PROJ_ROWS - 1) / PROJ_ROWS, a.H);
    timing_begin(a.stream, "simt_bwd_b2");
    simt_bwd_b2<Tin, D><<<pgrid, NT, smem_proj<D>(), a.stream>>>(
        (const Tin*)a.q, a.mu_k, a.P, w.R, w.ebar, w.U, w.dmu, w.dq_acc,
        w.gbar, w.Dv, a.B, a.H, a.T, PROJ_ROWS);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    PLX_TRY(set_smem(simt_dp_partial<Tin, D>, smem_dp<D>()));
    timing_begin(a.stream, "simt_dp_partial");
    simt_dp_partial<Tin, D><<<dim3(w.nchunks, a.H), NT, smem_dp<D>(), a.stream>>>(
        (const Tin*)a.q, a.mu_k, w.R, w.partial, a.B, a.H, a.T, DP_ROWS);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "simt_dp_reduce");
    simt_dp_reduce<<<dim3((D * D + 255) / 256, a.H), 256, 0, a.stream>>>(w.partial, a.dP, w.nchunks, D * D);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    PLX_TRY(set_smem(simt_bwd_b3<Tin, D, BM>, smem_b3<D, BM>()));
    const dim3 kgrid((a.T + BK - 1) / BK, a.B * a.H);
    timing_begin(a.stream, "simt_bwd_b3");
    simt_bwd_b3<Tin, D, BM><<<kgrid, NT, smem_b3<D, BM>(), a.stream>>>(
        (const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v, (const Tin*)a.dout, a.lse, w.U, w.dmu, w.gbar, w.ebar,
        w.Dv, w.dq_acc, (Tin*)a.dk, (Tin*)a.dv, a.T, scale, scale_log2);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    const size_t nd = (size_t)a.B * a.H * a.T * D;
    timing_begin(a.stream, "simt_cast_dq");
    cast_rows<Tin><<<(unsigned)((nd + 255) / 256), 256, 0, a.stream>>>(w.dq_acc, (Tin*)a.dq, nd);
    timing_end(a.stream);
    return cudaGetLastError();
}

template <typename Tin, int D>
cudaError_t bwd_impl(const BwdArgs& a) {
    const float scale_log2 = LOG2E / sqrtf((float)D);
    BwdWs w = bwd_ws(a.ws, a.B, a.H, a.T, a.d);
    const dim3 grid((a.T + BQ - 1) / BQ, a.B * a.H);
    PLX_TRY(set_smem(simt_bwd_b1<Tin, D>, smem_b1<D>()));
    timing_begin(a.stream, "simt_bwd_b1");
    simt_bwd_b1<Tin, D><<<grid, NT, smem_b1<D>(), a.stream>>>(
        (const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v, (const Tin*)a.dout, a.lse, w.R, w.ebar, a.T, scale_log2);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    return bwd_rest_impl<Tin, D>(a);
}

}  // namespace

size_t simt_fwd_ws_bytes(int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T;
    return align256(n * d * 4) + align256(n * 4);
}

size_t simt_bwd_ws_bytes(int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T, nd = n * d;
    const size_t nchunks = ((size_t)B * T + DP_ROWS - 1) / DP_ROWS;
    return 4 * align256(nd * 4) + 3 * align256(n * 4) + align256((size_t)H * nchunks * d * d * 4);
}

cudaError_t simt_fwd(const FwdArgs& a) {
    if (a.dtype == 0) return a.d == 64 ? fwd_impl<float, 64>(a) : fwd_impl<float, 128>(a);
    return a.d == 64 ? fwd_impl<__nv_bfloat16, 64>(a) : fwd_impl<__nv_bfloat16, 128>(a);
}

cudaError_t simt_bwd_after_b1(const BwdArgs& a) {
    if (a.dtype == 0) return a.d == 64 ? bwd_rest_impl<float, 64>(a) : bwd_rest_impl<float, 128>(a);
    return a.d == 64 ? bwd_rest_impl<__nv_bfloat16, 64>(a) : bwd_rest_impl<__nv_bfloat16, 128>(a);
}

void simt_bwd_ws_b1_outputs(void* ws, int B, int H, int T, int d, float** R, float** ebar) {
    BwdWs w = bwd_ws(ws, B, H, T, d);
    *R = w.R;
    *ebar = w.ebar;
}

size_t simt_dp_partial_bytes(int B, int H, int T, int d) {
    const size_t nchunks = ((size_t)B * T + DP_ROWS - 1) / DP_ROWS;
    return align256((size_t)H * nchunks * d * d * 4);
}

cudaError_t simt_dP(const void* q, const float* mu_k, const float* du, float* partial, float* dP, int B, int H,
                    int T, int d, int dtype, cudaStream_t stream) {
    const int nchunks = (B * T + DP_ROWS - 1) / DP_ROWS;
    auto run = [&](auto tin, auto dd) -> cudaError_t {
        using Tin = decltype(tin);
        constexpr int D = decltype(dd)::value;
        PLX_TRY(set_smem(simt_dp_partial<Tin, D>, smem_dp<D>()));
        timing_begin(stream, "simt_dp_partial");
        simt_dp_partial<Tin, D><<<dim3(nchunks, H), NT, smem_dp<D>(), stream>>>((const Tin*)q, mu_k, du, partial,
                                                                                 B, H, T, DP_ROWS);
        timing_end(stream);
        PLX_TRY(cudaGetLastError());
        timing_begin(stream, "simt_dp_reduce");
        simt_dp_reduce<<<dim3((D * D + 255) / 256, H), 256, 0, stream>>>(partial, dP, nchunks, D * D);
        timing_end(stream);
        return cudaGetLastError();
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    if (dtype == 0) return d == 64 ? run(float{}, I64{}) : run(float{}, I128{});
    return d == 64 ? run(__nv_bfloat16{}, I64{}) : run(__nv_bfloat16{}, I128{});
}

cudaError_t simt_bwd(const BwdArgs& a) {
    if (a.dtype == 0) return a.d == 64 ? bwd_impl<float, 64>(a) : bwd_impl<float, 128>(a);
    return a.d == 64 ? bwd_impl<__nv_bfloat16, 64>(a) : bwd_impl<__nv_bfloat16, 128>(a);
}

}  // namespace plx
