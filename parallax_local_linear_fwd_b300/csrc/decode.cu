// Decode: one new query per (sequence, head) against a KV cache.
//
// Same layer as the prefill path ("Parallax: Parameterized Local Linear
// Attention for Language Modeling", technical summary, "Core mechanism"; the
// paper's own kernel is a decode kernel, "Hardware-aware algorithm"): the
// query at position len - 1 of sequence b attends to keys 0 .. len - 1,
//   p_i = softmax(c q.k_i),  mu_k = sum p_i k_i,  u = P_h (q - mu_k),
//   gbar = mu_k . u,         o = sum_i p_i (1 + k_i.u - gbar) v_i.
// fp32 caches: with one query per head the products are matrix-vector, so
// this is an HBM stream, not a contraction: SIMT fp32 kernels over split-KV
// chunks staged in shared memory with coalesced loads.
//   dec_pass1 : per chunk, scores, chunk max m, l = sum 2^(s - m), a = sum 2^(s - m) k
//   dec_merge : per (b, h), combine the chunks (lse merge) -> lse, mu_k; then
//               u = P_h (q - mu_k) and gbar
//   dec_pass2 : per chunk, w_i = p_i (1 + k_i.u - gbar) (p from the merged lse),
//               partial sum w_i v_i
//   dec_sum   : out = sum of the chunk partials (the weights are already
//               normalised, so the partials simply add)
// Keys are read twice (passes 1 and 2) and values once.
//
// bf16 caches take the one-pass form in decode_tc.cu (each chunk keeps
// M = V^T diag(p) K on the tensor cores, so keys and values are read once).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "plx_internal.h"

namespace plx {
namespace {

// Keys per chunk (one CTA): 128 at d = 64, 64 at d = 128, so that pass 2's
// staged K and V stay near 66 KB and three CTAs share an SM.
__host__ __device__ constexpr int chunk_keys(int D) { return D == 64 ? 128 : 64; }
constexpr int NTD = 128;  // threads per CTA
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Valid key count of sequence b, clamped to [1, Lmax] (lens == nullptr: Lmax).
__device__ __forceinline__ int seq_len(const int* lens, int b, int Lmax) {
    return lens ? min(max(lens[b], 1), Lmax) : Lmax;
}

// Stage rows [r0, r0 + n) of a [Lmax][D] head slice into fp32 shared memory
// with row stride D + 1 (column and row walks are both conflict-free); rows
// past n read as zero.  16-byte vector loads, consecutive threads on
// consecutive 16-byte pieces of a row (coalesced).
__device__ __forceinline__ void widen16(const uint4& x, const __nv_bfloat16*, float (&f)[8], int& nf) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    nf = 8;
}
__device__ __forceinline__ void widen16(const uint4& x, const float*, float (&f)[8], int& nf) {
    f[0] = __uint_as_float(x.x);
    f[1] = __uint_as_float(x.y);
    f[2] = __uint_as_float(x.z);
    f[3] = __uint_as_float(x.w);
    nf = 4;
}

template <typename Tin, int D>
__device__ __forceinline__ void stage_rows(float* dst, const Tin* src, int r0, int n) {
    constexpr int DC = chunk_keys(D);
    constexpr int EPV = 16 / sizeof(Tin);  // elements per 16-byte piece
    constexpr int PPR = D / EPV;           // pieces per row
    constexpr int ITER = DC * PPR / NTD;
    uint4 buf[ITER];
#pragma unroll
    for (int k = 0; k < ITER; k++) {
        const int e = threadIdx.x + k * NTD, r = e / PPR, c = (e % PPR) * EPV;
        buf[k] = r < n ? *(const uint4*)(src + (size_t)(r0 + r) * D + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < ITER; k++) {
        const int e = threadIdx.x + k * NTD, r = e / PPR, c = (e % PPR) * EPV;
        float f[8];
        int nf;
        widen16(buf[k], (const Tin*)nullptr, f, nf);
#pragma unroll
        for (int x = 0; x < EPV; x++) dst[r * (D + 1) + c + x] = f[x];
    }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(NTD) dec_pass1(const Tin* __restrict__ q, const Tin* __restrict__ kc,
                                                 const int* __restrict__ lens, int H, int Lmax, int nsplit,
                                                 float scale_log2, float* __restrict__ part) {
    constexpr int DC = chunk_keys(D);
    extern __shared__ float dsm[];
    float* ks = dsm;                 // [DC][D + 1]
    float* qs = ks + DC * (D + 1);   // [D]
    float* ps = qs + D;              // [NTD] p~ of the chunk (0 past its keys)
    float* red = ps + NTD;           // [2 * NTD / 32] warp partials
    const int bh = blockIdx.y, c = blockIdx.x, b = bh / H;
    const int len = seq_len(lens, b, Lmax);
    const int r0 = c * DC, n = min(DC, len - r0);
    float* out = part + ((size_t)bh * nsplit + c) * (D + 2);
    if (n <= 0) {  // chunk past this sequence's length: an empty partial
        for (int j = threadIdx.x; j < D + 2; j += NTD) out[j] = j == 0 ? -INFINITY : 0.f;
        return;
    }
    const Tin* K = kc + (size_t)bh * Lmax * D;
    for (int j = threadIdx.x; j < D; j += NTD) qs[j] = ldf(q + (size_t)bh * D + j);
    stage_rows<Tin, D>(ks, K, r0, n);
    __syncthreads();
    const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
    float s = -INFINITY;
    if (i < n) {
        float acc = 0.f;
#pragma unroll 8
        for (int j = 0; j < D; j++) acc = fmaf(qs[j], ks[i * (D + 1) + j], acc);
        s = acc * scale_log2;
    }
    float m = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
    for (int w = 1; w < NTD / 32; w++) m = fmaxf(m, red[w]);
    const float p = i < n ? exp2f(s - m) : 0.f;
    ps[i] = p;
    float l = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    __syncthreads();
    if (lane == 0) red[NTD / 32 + warp] = l;
    // a_j = sum_i p~_i k_ij: D columns, NTD / D threads per column over interleaved keys
    constexpr int TPC = NTD / D;  // 2 for D = 64, 1 for D = 128
    const int j = i % D, part_id = i / D;
    float a = 0.f;
    for (int r = part_id; r < n; r += TPC) a = fmaf(ps[r], ks[r * (D + 1) + j], a);
    __syncthreads();
    if (TPC == 2 && part_id == 1) ps[j] = a;  // ps is free now: hand the second half over
    __syncthreads();
    if (part_id == 0) {
        if (TPC == 2) a += ps[j];
        out[2 + j] = a;
    }
    if (i == 0) {
        float lt = 0.f;
        for (int w = 0; w < NTD / 32; w++) lt += red[NTD / 32 + w];
        out[0] = m;
        out[1] = lt;
    }
}

// One CTA per (b, h): merge the chunk partials, then the projection.
template <typename Tin, int D>
__global__ void __launch_bounds__(D) dec_merge(const Tin* __restrict__ q, const float* __restrict__ P,
                                               const float* __restrict__ part, const int* __restrict__ lens, int H,
                                               int Lmax, int nsplit, float* __restrict__ lse,
                                               float* __restrict__ state) {
    constexpr int DC = chunk_keys(D);
    __shared__ float dl[D];
    __shared__ float red[D / 32];
    const int bh = blockIdx.x, h = bh % H, b = bh / H, j = threadIdx.x;
    const int len = seq_len(lens, b, Lmax);
    const int nc = (len + DC - 1) / DC;
    const float* pp = part + (size_t)bh * nsplit * (D + 2);
    float M = -INFINITY;
    for (int c = 0; c < nc; c++) M = fmaxf(M, pp[c * (D + 2)]);
    float l = 0.f, a = 0.f;
    for (int c = 0; c < nc; c++) {
        const float w = exp2f(pp[c * (D + 2)] - M);
        l = fmaf(pp[c * (D + 2) + 1], w, l);
        a = fmaf(pp[c * (D + 2) + 2 + j], w, a);
    }
    const float mu = a / l;
    dl[j] = ldf(q + (size_t)bh * D + j) - mu;
    // P_h staged with coalesced loads, row stride D + 1 (conflict-free row walks)
    extern __shared__ float ps[];
    const float* Ph = P + (size_t)h * D * D;
    for (int e = j; e < D * D; e += D) ps[(e / D) * (D + 1) + e % D] = Ph[e];
    __syncthreads();
    float u = 0.f;  // u_j = sum_b P[j][b] delta_b
#pragma unroll 8
    for (int k = 0; k < D; k++) u = fmaf(ps[j * (D + 1) + k], dl[k], u);
    float g = mu * u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if ((j & 31) == 0) red[j >> 5] = g;
    __syncthreads();
    float* st = state + (size_t)bh * (D + 2);
    st[2 + j] = u;
    if (j == 0) {
        float gt = 0.f;
        for (int w = 0; w < D / 32; w++) gt += red[w];
        const float l2 = M + log2f(l);  // lse in log2 units (scale included)
        st[0] = l2;
        st[1] = gt;
        lse[bh] = l2 * LN2;
    }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(NTD) dec_pass2(const Tin* __restrict__ q, const Tin* __restrict__ kc,
                                                 const Tin* __restrict__ vc, const int* __restrict__ lens, int H,
                                                 int Lmax, int nsplit, float scale_log2,
                                                 const float* __restrict__ state, float* __restrict__ opart) {
    constexpr int DC = chunk_keys(D);
    extern __shared__ float dsm[];
    float* ts = dsm;                 // [DC][D + 1]: K
    float* vs = ts + DC * (D + 1);   // [DC][D + 1]: V
    float* qs = vs + DC * (D + 1);   // [D]
    float* us = qs + D;              // [D]
    float* ws = us + D;              // [NTD] weights of the chunk (0 past its keys)
    const int bh = blockIdx.y, c = blockIdx.x, b = bh / H;
    const int len = seq_len(lens, b, Lmax);
    const int r0 = c * DC, n = min(DC, len - r0);
    float* out = opart + ((size_t)bh * nsplit + c) * D;
    if (n <= 0) {
        for (int j = threadIdx.x; j < D; j += NTD) out[j] = 0.f;
        return;
    }
    const float* st = state + (size_t)bh * (D + 2);
    const float l2 = st[0], g1 = 1.f - st[1];
    for (int j = threadIdx.x; j < D; j += NTD) {
        qs[j] = ldf(q + (size_t)bh * D + j);
        us[j] = st[2 + j];
    }
    stage_rows<Tin, D>(ts, kc + (size_t)bh * Lmax * D, r0, n);
    stage_rows<Tin, D>(vs, vc + (size_t)bh * Lmax * D, r0, n);
    __syncthreads();
    const int i = threadIdx.x;
    float w = 0.f;
    if (i < n) {
        float s = 0.f, g = 0.f;
#pragma unroll 8
        for (int j = 0; j < D; j++) {
            const float kv = ts[i * (D + 1) + j];
            s = fmaf(qs[j], kv, s);
            g = fmaf(us[j], kv, g);
        }
        w = exp2f(fmaf(s, scale_log2, -l2)) * (g + g1);
    }
    ws[i] = w;
    __syncthreads();
    constexpr int TPC = NTD / D;
    const int j = i % D, part_id = i / D;
    float a = 0.f;
    for (int r = part_id; r < n; r += TPC) a = fmaf(ws[r], vs[r * (D + 1) + j], a);
    __syncthreads();
    if (TPC == 2 && part_id == 1) ws[j] = a;
    __syncthreads();
    if (part_id == 0) out[j] = TPC == 2 ? a + ws[j] : a;
}

template <typename Tout, int D>
__global__ void __launch_bounds__(D) dec_sum(const float* __restrict__ opart, const int* __restrict__ lens, int H,
                                             int Lmax, int nsplit, Tout* __restrict__ out) {
    constexpr int DC = chunk_keys(D);
    const int bh = blockIdx.x, j = threadIdx.x;
    const int nc = (seq_len(lens, bh / H, Lmax) + DC - 1) / DC;
    const float* src = opart + (size_t)bh * nsplit * D + j;
    float s = 0.f;
    for (int c = 0; c < nc; c++) s += src[(size_t)c * D];
    stf(out + (size_t)bh * D + j, s);
}

// ================================================================ bf16 streaming form
#define PLX_TRY(x)                         \
    do {                                   \
        cudaError_t e_ = (x);              \
        if (e_ != cudaSuccess) return e_;  \
    } while (0)

template <typename Tin, int D>
cudaError_t decode_impl(const DecodeArgs& a) {
    constexpr int DC = chunk_keys(D);
    const int BH = a.B * a.H;
    const int nsplit = (a.Lmax + DC - 1) / DC;
    const float scale_log2 = LOG2E / sqrtf((float)D);
    float* part = (float*)a.ws;
    float* state = part + align256((size_t)BH * nsplit * (D + 2) * 4) / 4;
    float* opart = state + align256((size_t)BH * (D + 2) * 4) / 4;
    const size_t sm1 = sizeof(float) * (DC * (D + 1) + D + NTD + 2 * NTD / 32);
    const size_t sm2 = sizeof(float) * (2 * DC * (D + 1) + 2 * D + NTD);
    PLX_TRY(cudaFuncSetAttribute(dec_pass1<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1));
    PLX_TRY(cudaFuncSetAttribute(dec_pass2<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2));
    timing_begin(a.stream, "dec_pass1");
    dec_pass1<Tin, D><<<dim3(nsplit, BH), NTD, sm1, a.stream>>>((const Tin*)a.q, (const Tin*)a.k, a.lens, a.H,
                                                                 a.Lmax, nsplit, scale_log2, part);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    const size_t smm = sizeof(float) * D * (D + 1);
    PLX_TRY(cudaFuncSetAttribute(dec_merge<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smm));
    timing_begin(a.stream, "dec_merge");
    dec_merge<Tin, D><<<BH, D, smm, a.stream>>>((const Tin*)a.q, a.P, part, a.lens, a.H, a.Lmax, nsplit, a.lse,
                                                 state);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "dec_pass2");
    dec_pass2<Tin, D><<<dim3(nsplit, BH), NTD, sm2, a.stream>>>((const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v,
                                                                 a.lens, a.H, a.Lmax, nsplit, scale_log2, state,
                                                                 opart);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "dec_sum");
    dec_sum<Tin, D><<<BH, D, 0, a.stream>>>(opart, a.lens, a.H, a.Lmax, nsplit, (Tin*)a.out);
    timing_end(a.stream);
    return cudaGetLastError();
}

}  // namespace

size_t decode_ws_bytes(int B, int H, int Lmax, int d) {
    const size_t DC = chunk_keys(d);
    const size_t BH = (size_t)B * H, nsplit = ((size_t)Lmax + DC - 1) / DC;
    const size_t simt = align256(BH * nsplit * (d + 2) * 4) + align256(BH * (d + 2) * 4) +
                        align256(BH * nsplit * d * 4);
    const size_t onepass = decode_tc_ws_bytes(B, H, Lmax, d);
    return simt > onepass ? simt : onepass;
}

cudaError_t decode(const DecodeArgs& a) {
    if (a.dtype == 0) return a.d == 64 ? decode_impl<float, 64>(a) : decode_impl<float, 128>(a);
    return decode_tc(a);
}

}  // namespace plx
