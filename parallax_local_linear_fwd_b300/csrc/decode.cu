// Decode: one new query per (sequence, head) against a KV cache.
//
// Same layer as the prefill path ("Parallax: Parameterized Local Linear
// Attention for Language Modeling", technical summary, "Core mechanism"; the
// paper's own kernel is a decode kernel, "Hardware-aware algorithm"): the
// query at position len - 1 of sequence b attends to keys 0 .. len - 1,
//   p_i = softmax(c q.k_i),  mu_k = sum p_i k_i,  u = P_h (q - mu_k),
//   gbar = mu_k . u,         o = sum_i p_i (1 + k_i.u - gbar) v_i.
// With one query per head the products are matrix-vector, so this is an HBM
// stream, not a contraction: SIMT fp32 kernels over split-KV chunks staged in
// shared memory with coalesced loads.
//   dec_pass1 : per chunk, scores, chunk max m, l = sum 2^(s - m), a = sum 2^(s - m) k
//   dec_merge : per (b, h), combine the chunks (lse merge) -> lse, mu_k; then
//               u = P_h (q - mu_k) and gbar
//   dec_pass2 : per chunk, w_i = p_i (1 + k_i.u - gbar) (p from the merged lse),
//               partial sum w_i v_i
//   dec_sum   : out = sum of the chunk partials (the weights are already
//               normalised, so the partials simply add)
// Keys are read twice (passes 1 and 2) and values once.
//
// bf16 caches take a streaming form of the same steps (dec2_*): each warp
// owns a range of keys (a multiple of 32, sized on the host so that each
// pass's grid is one wave of resident CTAs) and pulls it through shared
// memory in 32-key sub-chunks with a cp.async pipeline (three stages in pass
// 1, so two sub-chunks are in flight while the warp computes on the third;
// two in pass 2, whose stages hold K and V, so that more warps fit); the
// warp keeps an online softmax (pass 1) or a running weighted sum (pass 2)
// and the CTA folds its warps into one partial.  Pass 2 merges pass 1's
// partials and forms u and gbar in its own prologue, and the last pass-2 CTA
// of each head (a completion counter that pass 1 clears) adds the head's
// partials in CTA order, so the sum is reproducible.
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
template <int D>
struct Dec2 {
    static constexpr int RB = D * 2;        // bytes per key row
    static constexpr int PPR = RB / 16;     // 16-byte pieces per row
    static constexpr int CPL = D / 32;      // value columns per lane
    static constexpr int SUB = 32;          // keys per sub-chunk (one per lane)
    static constexpr int NSTG = 3;          // cp.async stages per warp, pass 1
    static constexpr int NSTG2 = 2;         // pass 2 (K and V): smaller stages let more warps reside
    static constexpr int DW1 = 4;           // warps per CTA, pass 1
    static constexpr int DW2 = D == 64 ? 4 : 2;
    static constexpr int ST1 = SUB * RB;      // pass-1 stage (K)
    static constexpr int ST2 = 2 * SUB * RB;  // pass-2 stage (K then V)
    static constexpr size_t SM1 = (size_t)DW1 * NSTG * ST1 + sizeof(float) * (D + DW1 * (D + 2));
    static constexpr size_t SM2 = (size_t)DW2 * NSTG2 * ST2 + sizeof(float) * (4 * D + 2 + DW2 * D);
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Copy rows [0, nv) of a 32-row sub-chunk (rows past nv are zero-filled) into
// a stage: row r, 16-byte piece p lands at r * RB + ((p ^ (r & 7)) << 4), so
// that lanes reading one piece of 8 consecutive rows hit distinct banks.
template <int D>
__device__ __forceinline__ void dec2_issue(uint32_t stage, const __nv_bfloat16* rows, int nv, int lane) {
    using C = Dec2<D>;
#pragma unroll
    for (int idx = lane; idx < C::SUB * C::PPR; idx += 32) {
        const int r = idx / C::PPR, pc = idx % C::PPR;
        const bool ok = r < nv;
        const char* g = (const char*)rows + (size_t)(ok ? r : 0) * C::RB + pc * 16;
        cp_async16(stage + r * C::RB + ((pc ^ (r & 7)) << 4), g, ok ? 16 : 0);
    }
}

// Dot products of row r of a stage with two shared-memory vectors (x, y).
template <int D, bool TWO>
__device__ __forceinline__ void dec2_dots(const uint8_t* stage, int r, const float* x, const float* y, float& sx,
                                          float& sy) {
    using C = Dec2<D>;
    sx = 0.f;
    sy = 0.f;
#pragma unroll
    for (int pc = 0; pc < C::PPR; pc++) {
        const uint4 w = *(const uint4*)(stage + r * C::RB + ((pc ^ (r & 7)) << 4));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        const float4 xa = *(const float4*)(x + 8 * pc), xb = *(const float4*)(x + 8 * pc + 4);
        const float xs[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            sx = fmaf(xs[2 * e], bf_lo(ws[e]), sx);
            sx = fmaf(xs[2 * e + 1], bf_hi(ws[e]), sx);
        }
        if (TWO) {
            const float4 ya = *(const float4*)(y + 8 * pc), yb = *(const float4*)(y + 8 * pc + 4);
            const float ys[8] = {ya.x, ya.y, ya.z, ya.w, yb.x, yb.y, yb.z, yb.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                sy = fmaf(ys[2 * e], bf_lo(ws[e]), sy);
                sy = fmaf(ys[2 * e + 1], bf_hi(ws[e]), sy);
            }
        }
    }
}

// Column sums of a stage matrix, acc += sum_r wt_r x[r][.], eight columns
// per lane: lane = rg NG + cg owns columns 8 cg .. 8 cg + 7 (one 16-byte
// piece) over rows rg, rg + RG, ... (RG = 32 / NG row groups), so a lane
// reads one piece per row.  The row groups are combined once, at the end of
// the warp's keys (dec2_colsum_finish).
template <int D>
__device__ __forceinline__ void dec2_colsum(const uint8_t* mat, float wt, int lane, float (&acc)[8]) {
    using C = Dec2<D>;
    constexpr int NG = D / 8, RG = 32 / NG;
    const int cg = lane % NG, rg = lane / NG;
#pragma unroll
    for (int i = 0; i < C::SUB / RG; i++) {
        const int r = rg + RG * i;
        const float pr = __shfl_sync(0xffffffffu, wt, r);
        const uint4 w = *(const uint4*)(mat + r * C::RB + ((cg ^ (r & 7)) << 4));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            acc[2 * e] = fmaf(pr, bf_lo(ws[e]), acc[2 * e]);
            acc[2 * e + 1] = fmaf(pr, bf_hi(ws[e]), acc[2 * e + 1]);
        }
    }
}

// Add the row groups of dec2_colsum's accumulators and store the D column
// sums at dst[0 .. D) (4-byte stores: dst need not be 16-byte aligned).
template <int D>
__device__ __forceinline__ void dec2_colsum_finish(float (&acc)[8], int lane, float* dst) {
    constexpr int NG = D / 8;
#pragma unroll
    for (int o = NG; o < 32; o <<= 1)
#pragma unroll
        for (int t = 0; t < 8; t++) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    if (lane < NG) {  // dst need not be 16-byte aligned
#pragma unroll
        for (int t = 0; t < 8; t++) dst[8 * lane + t] = acc[t];
    }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Pass 1: CTA (c, bh) covers keys [c DW1 kpw, (c + 1) DW1 kpw), warp w the
// kpw keys from c DW1 kpw + w kpw; partial {m, l, a[D]} with
// l = sum 2^(s - m), a = sum 2^(s - m) k, s in log2 units.  CTA 0 of each
// head also clears that head's completion counter for pass 2.
template <int D>
__global__ void __launch_bounds__(Dec2<D>::DW1 * 32) dec2_pass1(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ kc,
                                                                const int* __restrict__ lens, int H, int Lmax,
                                                                int kpw, float scale_log2,
                                                                float* __restrict__ part, unsigned* __restrict__ cnt) {
    using C = Dec2<D>;
    extern __shared__ __align__(16) uint8_t dsm2[];
    float* qs = (float*)(dsm2 + (size_t)C::DW1 * C::NSTG * C::ST1);
    float* mg = qs + D;  // [DW1][D + 2] warp partials
    const int bh = blockIdx.y, c = blockIdx.x, b = bh / H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = seq_len(lens, b, Lmax);
    if (c == 0 && threadIdx.x == 0) cnt[bh] = 0u;
    for (int j = threadIdx.x; j < D; j += blockDim.x) qs[j] = __bfloat162float(q[(size_t)bh * D + j]);
    const int kb = (c * C::DW1 + warp) * kpw, ke = min(kb + kpw, len);
    const int nsc = ke > kb ? (ke - kb + C::SUB - 1) / C::SUB : 0;
    const __nv_bfloat16* K = kc + ((size_t)bh * Lmax + (kb < len ? kb : 0)) * D;
    uint8_t* stg = dsm2 + (size_t)warp * C::NSTG * C::ST1;
    const uint32_t stg_a = smem_addr(stg);
#pragma unroll
    for (int i = 0; i < C::NSTG - 1; i++) {
        if (i < nsc) dec2_issue<D>(stg_a + i * C::ST1, K + (size_t)i * C::SUB * D, ke - kb - i * C::SUB, lane);
        cp_async_commit();
    }
    __syncthreads();  // qs
    float m_run = -INFINITY, l_run = 0.f;
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; t++) acc[t] = 0.f;
    for (int sc = 0; sc < nsc; sc++) {
        const int nx = sc + C::NSTG - 1;
        if (nx < nsc)
            dec2_issue<D>(stg_a + (nx % C::NSTG) * C::ST1, K + (size_t)nx * C::SUB * D, ke - kb - nx * C::SUB, lane);
        cp_async_commit();
        cp_async_wait<C::NSTG - 1>();
        __syncwarp();
        const uint8_t* st = stg + (sc % C::NSTG) * C::ST1;
        const bool valid = kb + sc * C::SUB + lane < ke;
        float sx, sy;
        dec2_dots<D, false>(st, lane, qs, qs, sx, sy);
        const float s = valid ? sx * scale_log2 : -INFINITY;
        const float m_new = fmaxf(m_run, warp_max(s));
        const float alpha = exp2f(m_run - m_new);  // m_run = -inf at the start: alpha = 0
        const float p = valid ? exp2f(s - m_new) : 0.f;
        l_run = fmaf(l_run, alpha, warp_sum(p));
#pragma unroll
        for (int t = 0; t < 8; t++) acc[t] *= alpha;
        dec2_colsum<D>(st, p, lane, acc);
        m_run = m_new;
        __syncwarp();  // the stage is refilled by the next iteration's issue
    }
    cp_async_wait<0>();
    float* my = mg + warp * (D + 2);
    if (lane == 0) {
        my[0] = m_run;
        my[1] = l_run;
    }
    dec2_colsum_finish<D>(acc, lane, my + 2);
    __syncthreads();
    float* out = part + ((size_t)bh * gridDim.x + c) * (D + 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::DW1; w++) M = fmaxf(M, mg[w * (D + 2)]);
    for (int j = threadIdx.x; j < D + 2; j += blockDim.x) {
        if (j == 0) {
            out[0] = M;
            continue;
        }
        float x = 0.f;
        if (M > -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::DW1; w++) x = fmaf(mg[w * (D + 2) + j], exp2f(mg[w * (D + 2)] - M), x);
        }
        out[j] = x;
    }
}

// Pass 2: merge pass 1's np1 partials of head bh, u = P_h (q - mu_k), gbar;
// then CTA (c, bh) adds sum_i w_i v_i over its keys (laid out like pass 1's,
// kpw keys per warp) with w_i = 2^(s_i - L) (1 + k_i.u - gbar).  The last CTA
// of a head to finish (completion counter) adds the head's partials in CTA
// order and writes out[bh].
template <int D>
__global__ void __launch_bounds__(Dec2<D>::DW2 * 32) dec2_pass2(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ kc,
                                                                const __nv_bfloat16* __restrict__ vc,
                                                                const int* __restrict__ lens,
                                                                const float* __restrict__ P, int H, int Lmax,
                                                                int np1, int kpw1, int kpw, float scale_log2,
                                                                const float* __restrict__ part,
                                                                float* __restrict__ lse, float* __restrict__ opart,
                                                                unsigned* __restrict__ cnt,
                                                                __nv_bfloat16* __restrict__ out) {
    using C = Dec2<D>;
    constexpr int NT = C::DW2 * 32;
    extern __shared__ __align__(16) uint8_t dsm2[];
    float* qs = (float*)(dsm2 + (size_t)C::DW2 * C::NSTG2 * C::ST2);
    float* us = qs + D;
    float* mus = us + D;
    float* dl = mus + D;
    float* scal = dl + D;  // {L (log2 units), 1 - gbar}
    float* mg = scal + 2;  // [DW2][D]
    __shared__ int s_last;
    const int bh = blockIdx.y, c = blockIdx.x, b = bh / H, h = bh % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = seq_len(lens, b, Lmax);
    const int kb = (c * C::DW2 + warp) * kpw, ke = min(kb + kpw, len);
    const int nsc = ke > kb ? (ke - kb + C::SUB - 1) / C::SUB : 0;
    const __nv_bfloat16* K = kc + ((size_t)bh * Lmax + (kb < len ? kb : 0)) * D;
    const __nv_bfloat16* V = vc + ((size_t)bh * Lmax + (kb < len ? kb : 0)) * D;
    uint8_t* stg = dsm2 + (size_t)warp * C::NSTG2 * C::ST2;
    const uint32_t stg_a = smem_addr(stg);
    // start the key and value stream before the prologue
#pragma unroll
    for (int i = 0; i < C::NSTG2 - 1; i++) {
        if (i < nsc) {
            dec2_issue<D>(stg_a + i * C::ST2, K + (size_t)i * C::SUB * D, ke - kb - i * C::SUB, lane);
            dec2_issue<D>(stg_a + i * C::ST2 + C::SUB * C::RB, V + (size_t)i * C::SUB * D, ke - kb - i * C::SUB,
                          lane);
        }
        cp_async_commit();
    }
    // prologue: merge the head's pass-1 partials (unrolled so that the loads overlap)
    const int nc1 = (len + C::DW1 * kpw1 - 1) / (C::DW1 * kpw1);
    const float* pp = part + (size_t)bh * np1 * (D + 2);
    float M = -INFINITY;
#pragma unroll 8
    for (int i = 0; i < nc1; i++) M = fmaxf(M, pp[(size_t)i * (D + 2)]);
    float l = 0.f;
#pragma unroll 8
    for (int i = 0; i < nc1; i++) l = fmaf(pp[(size_t)i * (D + 2) + 1], exp2f(pp[(size_t)i * (D + 2)] - M), l);
    for (int j = threadIdx.x; j < D; j += NT) {
        float a = 0.f;
#pragma unroll 8
        for (int i = 0; i < nc1; i++)
            a = fmaf(pp[(size_t)i * (D + 2) + 2 + j], exp2f(pp[(size_t)i * (D + 2)] - M), a);
        const float mu = a / l, qj = __bfloat162float(q[(size_t)bh * D + j]);
        qs[j] = qj;
        mus[j] = mu;
        dl[j] = qj - mu;
    }
    __syncthreads();
    // u_j = sum_b P[j][b] delta_b: thread j reads row j of P_h with 16-byte loads
    const float* Ph = P + (size_t)h * D * D;
    for (int j = threadIdx.x; j < D; j += NT) {
        const float4* row = (const float4*)(Ph + (size_t)j * D);
        float x = 0.f;
#pragma unroll
        for (int e = 0; e < D / 4; e++) {
            const float4 pv = row[e];
            x = fmaf(pv.x, dl[4 * e], x);
            x = fmaf(pv.y, dl[4 * e + 1], x);
            x = fmaf(pv.z, dl[4 * e + 2], x);
            x = fmaf(pv.w, dl[4 * e + 3], x);
        }
        us[j] = x;
    }
    __syncthreads();
    if (warp == 0) {
        float g = 0.f;
#pragma unroll
        for (int t = 0; t < C::CPL; t++) g = fmaf(mus[lane + 32 * t], us[lane + 32 * t], g);
        g = warp_sum(g);
        if (lane == 0) {
            const float L = M + log2f(l);
            scal[0] = L;
            scal[1] = 1.f - g;
            if (c == 0) lse[bh] = L * LN2;
        }
    }
    __syncthreads();
    const float L = scal[0], g1 = scal[1];
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; t++) acc[t] = 0.f;
    for (int sc = 0; sc < nsc; sc++) {
        const int nx = sc + C::NSTG2 - 1;
        if (nx < nsc) {
            const uint32_t sa = stg_a + (nx % C::NSTG2) * C::ST2;
            dec2_issue<D>(sa, K + (size_t)nx * C::SUB * D, ke - kb - nx * C::SUB, lane);
            dec2_issue<D>(sa + C::SUB * C::RB, V + (size_t)nx * C::SUB * D, ke - kb - nx * C::SUB, lane);
        }
        cp_async_commit();
        cp_async_wait<C::NSTG2 - 1>();
        __syncwarp();
        const uint8_t* st = stg + (sc % C::NSTG2) * C::ST2;
        const bool valid = kb + sc * C::SUB + lane < ke;
        float sx, sg;
        dec2_dots<D, true>(st, lane, qs, us, sx, sg);
        const float w = valid ? exp2f(fmaf(sx, scale_log2, -L)) * (sg + g1) : 0.f;
        dec2_colsum<D>(st + C::SUB * C::RB, w, lane, acc);
        __syncwarp();
    }
    cp_async_wait<0>();
    dec2_colsum_finish<D>(acc, lane, mg + warp * D);
    __syncthreads();
    float* dst = opart + ((size_t)bh * gridDim.x + c) * D;
    for (int j = threadIdx.x; j < D; j += NT) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < C::DW2; w++) x += mg[w * D + j];
        dst[j] = x;
    }
    // the head's last CTA adds the partials in CTA order
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&cnt[bh], 1u) == gridDim.x - 1;
    __syncthreads();
    if (s_last) {
        __threadfence();
        const float* src = opart + (size_t)bh * gridDim.x * D;
        for (int j = threadIdx.x; j < D; j += NT) {
            float x = 0.f;
            for (unsigned i = 0; i < gridDim.x; i++) x += __ldcg(src + (size_t)i * D + j);
            out[(size_t)bh * D + j] = __float2bfloat16_rn(x);
        }
    }
}

// Keys per warp for a pass: the smallest multiple of 32 for which the grid
// (BH x CTAs per head) fits in one wave of resident CTAs.
int dec2_kpw(int BH, int Lmax, int warps_per_cta, int resident_ctas) {
    for (int kpw = 32;; kpw += 32) {
        const long long per_head = (Lmax + (long long)warps_per_cta * kpw - 1) / ((long long)warps_per_cta * kpw);
        if ((long long)BH * per_head <= resident_ctas || kpw >= Lmax) return kpw;
    }
}

template <int D>
size_t dec2_ws_bytes(size_t BH, int Lmax) {
    using C = Dec2<D>;
    // the largest partial counts: 32 keys per warp
    const size_t np1 = ((size_t)Lmax + C::DW1 * 32 - 1) / (C::DW1 * 32);
    const size_t np2 = ((size_t)Lmax + C::DW2 * 32 - 1) / (C::DW2 * 32);
    return align256(BH * np1 * (D + 2) * 4) + align256(BH * np2 * D * 4) + align256(BH * 4);
}

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

template <int D>
cudaError_t decode2_impl(const DecodeArgs& a) {
    using C = Dec2<D>;
    const int BH = a.B * a.H;
    int dev = 0, sms = 0, occ1 = 0, occ2 = 0;
    PLX_TRY(cudaFuncSetAttribute(dec2_pass1<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SM1));
    PLX_TRY(cudaFuncSetAttribute(dec2_pass2<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SM2));
    PLX_TRY(cudaGetDevice(&dev));
    PLX_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    PLX_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, dec2_pass1<D>, C::DW1 * 32, C::SM1));
    PLX_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, dec2_pass2<D>, C::DW2 * 32, C::SM2));
    const int kpw1 = dec2_kpw(BH, a.Lmax, C::DW1, sms * (occ1 > 0 ? occ1 : 1));
    const int kpw2 = dec2_kpw(BH, a.Lmax, C::DW2, sms * (occ2 > 0 ? occ2 : 1));
    const int np1 = (a.Lmax + C::DW1 * kpw1 - 1) / (C::DW1 * kpw1);
    const int np2 = (a.Lmax + C::DW2 * kpw2 - 1) / (C::DW2 * kpw2);
    const float scale_log2 = LOG2E / sqrtf((float)D);
    const size_t np1_max = ((size_t)a.Lmax + C::DW1 * 32 - 1) / (C::DW1 * 32);
    const size_t np2_max = ((size_t)a.Lmax + C::DW2 * 32 - 1) / (C::DW2 * 32);
    float* part = (float*)a.ws;
    float* opart = part + align256((size_t)BH * np1_max * (D + 2) * 4) / 4;
    unsigned* cnt = (unsigned*)(opart + align256((size_t)BH * np2_max * D * 4) / 4);
    const __nv_bfloat16* q = (const __nv_bfloat16*)a.q;
    timing_begin(a.stream, "dec_pass1");
    dec2_pass1<D><<<dim3(np1, BH), C::DW1 * 32, C::SM1, a.stream>>>(q, (const __nv_bfloat16*)a.k, a.lens, a.H,
                                                                     a.Lmax, kpw1, scale_log2, part, cnt);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "dec_pass2");
    dec2_pass2<D><<<dim3(np2, BH), C::DW2 * 32, C::SM2, a.stream>>>(
        q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.lens, a.P, a.H, a.Lmax, np1, kpw1, kpw2,
        scale_log2, part, a.lse, opart, cnt, (__nv_bfloat16*)a.out);
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
