// Decode, bf16 caches: one pass over the keys and values.
//
// The layer at one new query per (sequence, head) ("Parallax: Parameterized
// Local Linear Attention for Language Modeling", technical summary, "Core
// mechanism"; the paper's own kernel is a decode kernel that runs both
// branches over one KV stream, "Hardware-aware algorithm"):
//   p_i = softmax(c q.k_i),  mu_k = sum p_i k_i,  mu_v = sum p_i v_i,
//   u = P_h (q - mu_k),  gbar = mu_k . u,
//   o = sum_i p_i (1 + k_i.u - gbar) v_i = mu_v + M u - gbar mu_v,
//   M = sum_i p_i v_i k_i^T   (d x d).
// u needs mu_k, which needs every key, so the weights p (1 + k.u - gbar)
// cannot be formed in the same pass as the softmax.  M can: it does not
// depend on u.  So each CTA streams its chunk of keys once and keeps, with
// an online softmax, l = sum p, sum p k, sum p v (registers) and
// M = V^T diag(p) K (a tcgen05 MMA into TMEM, d x d per chunk: 2 d^2 flops
// per key, far below the tensor rate, while the stream is HBM-bound).  A
// second kernel merges the chunks of a head by their log-sum-exp and forms
// u, gbar and o.  Keys and values are read once.
//
//   dec1_chunk<D> : grid (chunks, B H), 128 threads (TPK = D/32 threads per
//                   key, 32 features each), three CTAs per SM.  K and V tiles
//                   of KT = 128 / TPK keys (8 KB each) arrive by TMA (128-byte
//                   swizzle) in NS = 4 stages; lane 0 of the last warp refills
//                   each stage two tiles after its MMA was issued (so its wait
//                   is short) while warp 0 issues the previous tile's MMA.
//                   Per tile: scores, tile max (lazy rescale by 2^8), p, the
//                   register sums, then p k and v are written back in place
//                   as f16 and one thread issues M += V^T (p K) (A = V^T read
//                   MN-major; at d = 64 its second 64-row block is a zero
//                   tile, so M = 128 rows of which the first 64 are used).
//   dec1_merge<D> : grid (B H).  m = max m_c, w_c = 2^(m_c - m), then the
//                   merged sums, u = P_h (q - mu_k), gbar, o and lse.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "plx_internal.h"
#include "tc_ptx.cuh"

namespace plx {
namespace {

using namespace tc;

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_TH = 8.f;  // log2 units: p~ <= 2^8 between rescales

__device__ __forceinline__ float fast_exp2_dec(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bar.red.and over the worker warps (barrier 1): every worker gets the AND
// of everyone's predicate, so all take the same branch after a wait.
__device__ __forceinline__ bool workers_and(bool pred, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int D>
struct Dec1 {
    static constexpr int TPK = D / 32;       // threads per key (32 features each)
    static constexpr int KT = 128 / TPK;     // keys per tile: 64 (d 64) or 32 (d 128)
    static constexpr int NW = 4;             // warps: 128 threads, KT keys x TPK
    static constexpr int NT = 32 * NW;
    static constexpr int MIN_CTAS = 3;       // resident CTAs per SM
    static constexpr int NS = 4;             // K|V stages
    static constexpr int TB = KT * D * 2;    // one K or V tile (bf16 / f16): 8 KB
    static constexpr int ZB = D == 64 ? TB : 0;  // zero tile: rows 64..127 of A at d = 64
    static constexpr int NBAR = 2 * NS + 2;  // full[NS], empty[NS], mma_done, drain
    static constexpr int QS = 34;            // stride of q's 32-feature parts in shared memory (even: float2)
    static constexpr int SMEM = 1024 + NS * 2 * TB + ZB + NBAR * 8 + 16 + 8 * 4 + TPK * QS * 4 + 16;
    static_assert(KT * TPK == NW * 32, "one thread per (key, feature part)");
    static_assert(2 * NW <= 8, "the two tile-parity copies of the warp maxima fit their slot");
    static_assert(MIN_CTAS * (SMEM + 1024) <= 233472, "MIN_CTAS CTAs fit an SM's shared memory");
    static constexpr unsigned TMEM_COLS = D;
    // partial of one chunk: {m, l, pad[2]}, sum p k [D], sum p v [D], M [D][D]
    static constexpr int PART = 4 + 2 * D + D * D;
};

__device__ __forceinline__ int seq_len1(const int* lens, int b, int Lmax) {
    return lens ? min(max(lens[b], 1), Lmax) : Lmax;
}

__device__ __forceinline__ uint32_t swz(int r, int c, int rows) {  // 16-bit tile, 64-column blocks
    return (uint32_t)((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void workers_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int D>
__global__ void __launch_bounds__(Dec1<D>::NT, Dec1<D>::MIN_CTAS) dec1_chunk(const __grid_constant__ CUtensorMap tm_k,
                                                           const __grid_constant__ CUtensorMap tm_v,
                                                           const __nv_bfloat16* __restrict__ q,
                                                           const int* __restrict__ lens, int H, int Lmax,
                                                           int chunk, float scale_log2, float* __restrict__ part,
                                                           unsigned* status) {
    // (q, lens, the caches and part are device pointers; status is the
    // device watchdog word of the calling device)
    using C = Dec1<D>;
    constexpr int NS = C::NS, KT = C::KT, TPK = C::TPK, NW = C::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sKV = sm;                       // stage s: K at 2 s TB, V at (2 s + 1) TB
    uint8_t* sZ = sKV + NS * 2 * C::TB;      // d = 64: zero tile (rows 64..127 of the A operand)
    uint64_t* bars = (uint64_t*)(sZ + C::ZB);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* mma_done = bars + 2 * NS;
    uint64_t* drain = mma_done + 1;
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);
    float* wmax = (float*)(holder + 4);      // [2][NW] tile maxima per worker warp, by tile parity
    float* sq = wmax + 8;                    // [D] the query, fp32

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, b = bh / H;
    const int len = seq_len1(lens, b, Lmax);
    const int k_begin = blockIdx.x * chunk;
    const int k_end = min(k_begin + chunk, len);
    if (k_begin >= k_end) return;  // no keys of this sequence in this chunk (uniform per CTA)
    const int nt = (k_end - k_begin + KT - 1) / KT;
    const Watchdog wd{status, abortf, KID_DECODE, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (C::ZB) {
        for (int i = threadIdx.x; i < C::ZB / 16; i += C::NT) ((uint4*)sZ)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tM = *holder;

    // loads of tile j into stage j % NS (rows past Lmax read as zero)
    auto load_tile = [&](int j) {
        const int s = j % NS;
        mbar_expect_tx(&full[s], 2 * C::TB);
#pragma unroll
        for (int r = 0; r < D / 64; r++) {
            tma_load_3d(sKV + (2 * s) * C::TB + r * KT * 128, &tm_k, r * 64, k_begin + j * KT, bh, &full[s]);
            tma_load_3d(sKV + (2 * s + 1) * C::TB + r * KT * 128, &tm_v, r * 64, k_begin + j * KT, bh, &full[s]);
        }
    };
    // the loader is lane 0 of the last warp, so its refills overlap warp 0's
    // MMA issue at the end of the previous tile
    const bool loader = threadIdx.x == (NW - 1) * 32;
    int issued = 0;  // loader: tiles whose loads are issued
    if (loader) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        for (; issued < 2 && issued < nt; issued++) load_tile(issued);
    }
    {
        // workers: lane = fp * KW + kl, thread = (key r = warp KW + kl of the
        // tile, feature part fp); eight lanes of one part read eight keys'
        // rows, which the swizzle spreads over all banks
        constexpr int KW = 32 / TPK;  // keys per warp
        const int kl = lane % KW, fp = lane / KW;
        const int r = warp * KW + kl;
        const int f0 = fp * 32;  // features [f0, f0 + 32)
        // q in shared memory as fp32 (threads of one feature part read the
        // same words: broadcasts), which keeps 32 registers free
        // (part fp at fp * QS: the parts' words fall in different banks; QS is
        // even so pairs load as float2)
        for (int i = threadIdx.x; i < D; i += NW * 32) sq[(i >> 5) * C::QS + (i & 31)] = __bfloat162float(q[(size_t)bh * D + i]);
        workers_sync(NW * 32);
        const float* qf = sq + fp * C::QS;
        uint64_t ak[16], av[16];  // sum p k, sum p v over this thread's keys, as f32x2 pairs
#pragma unroll
        for (int i = 0; i < 16; i++) ak[i] = av[i] = 0;
        float l = 0.f, m_run = -INFINITY;
        const uint32_t idM = idesc_mma(128, D, true, true);
        // M += V^T (p K) for tile jt: A = V^T (MN-major: features contiguous),
        // B = p K (MN-major), K dimension = the tile's keys in steps of 16.
        // Issued by warp 0 at the next tile's max barrier (or after the loop
        // for the last tile), which every write-back of tile jt precedes, so a
        // tile needs one barrier
        auto issue_mma = [&](int jt) {
            const int st = jt % NS;
            const uint32_t va = smem_u32(sKV + (2 * st + 1) * C::TB), kb = smem_u32(sKV + (2 * st) * C::TB);
            const uint32_t lboA = D == 64 ? (uint32_t)(smem_u32(sZ) - va) : (uint32_t)(KT * 128);
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < KT / 16; kk++)
                    mma_ss(tM, desc_mn_lbo(va, kk, lboA), desc_mnmajor(kb, KT, kk), idM, (jt > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty[st]);
                mma_commit(mma_done);
            }
            __syncwarp();
        };
        bool ok = true;
        for (int j = 0; j < nt; j++) {
            const int s = j % NS;
            // refill: tile j + 2 into the stage of tile j - 2 (NS = 4), whose MMA
            // was issued two tiles ago, so the wait is short; tiles j, j + 1
            // and j + 2 are then loaded or in flight
            static_assert(NS == 4, "the refill distance assumes four stages");
            if (loader && ok && issued < nt && issued == j + 2) {
                if (j < 2 || mbar_wait(&empty[(j - 2) % NS], ((j - 2) / NS) & 1, wd, 1)) {
                    load_tile(issued);
                    issued++;
                } else {
                    ok = false;
                }
            }
            ok = mbar_wait(&full[s], (j / NS) & 1, wd, 2) && ok;
            // every worker takes the same decisions below: agree on ok first
            if (!__all_sync(0xffffffffu, ok)) ok = false;
            uint8_t* sk = sKV + (2 * s) * C::TB;
            uint8_t* sv = sKV + (2 * s + 1) * C::TB;
            const int key = k_begin + j * KT + r;
            const bool valid = key < k_end;
            // scores: this thread's 32 features of key r, summed over the TPK threads of the key
            uint4 kc[4];
            uint64_t dp[4] = {0, 0, 0, 0};  // four independent chains of f32x2 pairs
#pragma unroll
            for (int c = 0; c < 4; c++) {
                kc[c] = *(const uint4*)(sk + swz(r, f0 + 8 * c, KT));
                const uint32_t w[4] = {kc[c].x, kc[c].y, kc[c].z, kc[c].w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float2 qq = *(const float2*)(qf + 8 * c + 2 * e);
                    dp[c] = ffma2(f2(qq.x, qq.y), f2(bf16_lo(w[e]), bf16_hi(w[e])), dp[c]);
                }
            }
            const float2 d01 = uf2(fadd2(fadd2(dp[0], dp[1]), fadd2(dp[2], dp[3])));
            float dot = d01.x + d01.y;
#pragma unroll
            for (int o = KW; o < 32; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const float sc = valid ? dot * scale_log2 : -INFINITY;
            float tmax = sc;
#pragma unroll
            for (int o = 1; o < KW; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            // two copies by tile parity: a warp that runs ahead writes the next
            // tile's maximum while a slower one may still read this tile's
            float* wm = wmax + (j & 1) * NW;
            if (lane == 0) wm[warp] = tmax;
            // the abort decision rides on the same barrier
            if (!workers_and(ok, NW * 32)) {
                ok = false;
                break;
            }
            if (warp == 0 && j >= 1) issue_mma(j - 1);
            float tm = wm[0];
#pragma unroll
            for (int w = 1; w < NW; w++) tm = fmaxf(tm, wm[w]);
            const float m_new = fmaxf(m_run, tm);
            float alpha = 1.f;
            if (m_new > m_run + RESCALE_TH) {  // uniform across the CTA
                alpha = fast_exp2_dec(m_run - m_new);
                m_run = m_new;
                l *= alpha;
                const uint64_t A2 = f2(alpha, alpha);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    ak[i] = fmul2(ak[i], A2);
                    av[i] = fmul2(av[i], A2);
                }
                if (j > 0) {
                    // M *= alpha once the previous tile's MMA has landed (warps 0-3
                    // own TMEM lanes 0-127, thread = row of M)
                    const bool got = mbar_wait(mma_done, (j - 1) & 1, wd, 3);
                    ok = ok && got;  // agreed on at the next tile's barrier
                    if (warp < 4 && __all_sync(0xffffffffu, got)) {
                        tc_fence_after();
                        const uint32_t lrow = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
                        for (int c = 0; c < D / 32; c++) {
                            uint32_t u[32];
                            tmem_ld32(tM + lrow + c * 32, u);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                            tmem_st32(tM + lrow + c * 32, u);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                }
            }
            const float p = valid ? fast_exp2_dec(sc - m_run) : 0.f;
            if (fp == 0) l += p;
            // p k and v in f16, written back in place; the register sums.  A key
            // past the sequence writes zeros (its cache row may hold anything)
            const uint64_t P2 = f2(p, p);
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint32_t off = swz(r, f0 + 8 * c, KT);
                uint4 ko = make_uint4(0, 0, 0, 0), vo = make_uint4(0, 0, 0, 0);
                if (valid) {
                    const uint4 vc = *(const uint4*)(sv + off);
                    const uint32_t kw[4] = {kc[c].x, kc[c].y, kc[c].z, kc[c].w};
                    const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
                    uint32_t kp[4], vp[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const uint64_t pk = fmul2(P2, f2(bf16_lo(kw[e]), bf16_hi(kw[e])));
                        const uint64_t vv = f2(bf16_lo(vw[e]), bf16_hi(vw[e]));
                        ak[4 * c + e] = fadd2(ak[4 * c + e], pk);
                        av[4 * c + e] = ffma2(P2, vv, av[4 * c + e]);
                        const float2 pkf = uf2(pk);
                        kp[e] = pack_f16(pkf.x, pkf.y);
                        vp[e] = pack_f16_sat(bf16_lo(vw[e]), bf16_hi(vw[e]));
                    }
                    ko = make_uint4(kp[0], kp[1], kp[2], kp[3]);
                    vo = make_uint4(vp[0], vp[1], vp[2], vp[3]);
                }
                *(uint4*)(sk + off) = ko;
                *(uint4*)(sv + off) = vo;
            }
            fence_proxy_async_smem();
        }
        // the merge grid may now be scheduled (it waits for this grid's
        // completion before it reads the partials)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // loads issued but not consumed (only after an abort) land before
        // stage 0 is reused below and before the CTA exits
        if (loader)
            for (int jj = issued > NS ? issued - NS : 0; jj < issued; jj++) mbar_wait_drain(&full[jj % NS], (jj / NS) & 1);
        // ---- the chunk's partial (every worker agrees whether it is valid)
        ok = workers_and(ok, NW * 32);
        if (ok && warp == 0) issue_mma(nt - 1);  // the last tile's write-back preceded the barrier above
        float* dst = part + ((size_t)bh * gridDim.x + blockIdx.x) * C::PART;
        // l, sum p k, sum p v: reduce over the keys (lanes of one feature part
        // first, then the worker warps through shared memory, reusing stage 0)
        float akf[32], avf[32];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const float2 a2 = uf2(ak[i]), b2 = uf2(av[i]);
            akf[2 * i] = a2.x;
            akf[2 * i + 1] = a2.y;
            avf[2 * i] = b2.x;
            avf[2 * i + 1] = b2.y;
        }
#pragma unroll
        for (int o = 1; o < KW; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
            for (int i = 0; i < 32; i++) {
                akf[i] += __shfl_xor_sync(0xffffffffu, akf[i], o);
                avf[i] += __shfl_xor_sync(0xffffffffu, avf[i], o);
            }
        }
        // every tile's MMA must be done before stage 0 is reused below
        if (warp == 0) {
            if (elect_one()) mma_commit(drain);
            __syncwarp();
            mbar_wait_drain(drain, 0);
        }
        workers_sync(NW * 32);
        float* red = (float*)sKV;  // [NW][2 D + 1]
        if (ok && kl == 0) {
#pragma unroll
            for (int i = 0; i < 32; i++) {
                red[warp * (2 * D + 1) + f0 + i] = akf[i];
                red[warp * (2 * D + 1) + D + f0 + i] = avf[i];
            }
            if (lane == 0) red[warp * (2 * D + 1) + 2 * D] = l;
        }
        workers_sync(NW * 32);
        for (int e = threadIdx.x; ok && e < 2 * D + 1; e += NW * 32) {
            float x = 0.f;
            for (int w = 0; w < NW; w++) x += red[w * (2 * D + 1) + e];
            if (e < 2 * D) dst[4 + e] = x;
            else dst[1] = x;
        }
        if (threadIdx.x == 0) dst[0] = ok ? m_run : -INFINITY;  // an aborted chunk weighs 0 in the merge
        // M from TMEM: warps 0-3, thread = row m of M (rows past D at d = 64 are the zero block's)
        if (warp < 4 && ok) {
            tc_fence_after();
            const int mrow = warp * 32 + lane;
            const uint32_t lrow = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
            for (int c = 0; c < D / 32; c++) {
                uint32_t u[32];
                tmem_ld32(tM + lrow + c * 32, u);
                tmem_wait_ld();
                if (mrow < D) {
                    float* mr = dst + 4 + 2 * D + (size_t)mrow * D + c * 32;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *(float4*)(mr + i) = make_float4(__uint_as_float(u[i]), __uint_as_float(u[i + 1]),
                                                         __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tM, C::TMEM_COLS);
    }
}

// Merge the chunks of one head (only those holding keys of the sequence)
// and finish the layer: lse, mu_k, mu_v, u = P_h (q - mu_k), gbar = mu_k . u,
// o = mu_v + M u - gbar mu_v.  256 threads; the matrix-vector products (P_h
// and each chunk's M) give four threads to a row (D/4 columns each).  The
// kernel is a chain of short dependent steps, so every load that does not
// depend on an earlier step is issued at the start: this thread's P_h row
// part, q, and its M row parts of the first kPre chunks (4 at d = 64, 1 at
// d = 128, within the register budget), which then arrive
// during the scalar steps instead of after them.
constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) dec1_merge(const __nv_bfloat16* __restrict__ q,
                                                            const int* __restrict__ lens, const float* __restrict__ P,
                                                            const float* part, int H, int Lmax,
                                                            int chunk, int nchunk, float* __restrict__ lse,
                                                            __nv_bfloat16* __restrict__ out) {
    using C = Dec1<D>;
    constexpr int NWM = kMergeThreads / 32;
    constexpr int RPP = kMergeThreads / 4;   // rows per pass, four threads per row
    constexpr int NPASS = (D + RPP - 1) / RPP;
    constexpr int CQ = D / 4;                // columns per thread
    constexpr int kPre = D == 64 ? 4 : 1;    // chunks whose M rows are loaded up front
    __shared__ float s_d[D], s_mk[D], s_mv[D], s_u[D], s_red[NWM], s_w[kPre];
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qr = tid & 3, rr = tid >> 2;   // column quarter, row within a pass
    const int len = seq_len1(lens, b, Lmax);
    const int nc = min(nchunk, (len + chunk - 1) / chunk);
    const float* pb = part + (size_t)bh * nchunk * C::PART;
    // loads that depend on nothing computed here: P_h and q before the chunk
    // kernel has finished (this grid may start early, as its programmatic
    // dependent), the chunks' partials after
    float4 pv[NPASS][CQ / 4], mpre[kPre][NPASS][CQ / 4];
#pragma unroll
    for (int ps = 0; ps < NPASS; ps++) {
        const int a = ps * RPP + rr;
#pragma unroll
        for (int i = 0; i < CQ / 4; i++)
            pv[ps][i] = a < D ? ((const float4*)(P + ((size_t)h * D + a) * D + qr * CQ))[i] : make_float4(0, 0, 0, 0);
    }
    const float qv = tid < D ? __bfloat162float(q[(size_t)bh * D + tid]) : 0.f;
    // the partials are read only past this wait: `part` is not declared
    // __restrict__, so the compiler may not move their loads above it
    asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
    for (int ps = 0; ps < NPASS; ps++) {
        const int a = ps * RPP + rr;
#pragma unroll
        for (int i = 0; i < CQ / 4; i++) {
#pragma unroll
            for (int c = 0; c < kPre; c++)
                mpre[c][ps][i] = (a < D && c < nc)
                                     ? ((const float4*)(pb + (size_t)c * C::PART + 4 + 2 * D + (size_t)a * D + qr * CQ))[i]
                                     : make_float4(0, 0, 0, 0);
        }
    }
    float m = -INFINITY;
    for (int c = 0; c < nc; c++) m = fmaxf(m, pb[(size_t)c * C::PART]);
    float l = 0.f;
    for (int c = 0; c < nc; c++) l = fmaf(exp2f(pb[(size_t)c * C::PART] - m), pb[(size_t)c * C::PART + 1], l);
    const float inv = 1.f / l;
    if (tid < kPre) s_w[tid] = tid < nc ? exp2f(pb[(size_t)tid * C::PART] - m) : 0.f;
    if (tid < D) {
        float mk = 0.f, mv = 0.f;
        for (int c = 0; c < nc; c++) {
            const float* pc = pb + (size_t)c * C::PART;
            const float w = exp2f(pc[0] - m);
            mk = fmaf(w, pc[4 + tid], mk);
            mv = fmaf(w, pc[4 + D + tid], mv);
        }
        s_mk[tid] = mk * inv;
        s_mv[tid] = mv * inv;
        s_d[tid] = qv - mk * inv;  // delta = q - mu_k
    }
    __syncthreads();
    // u = P_h delta
#pragma unroll
    for (int ps = 0; ps < NPASS; ps++) {
        const int a = ps * RPP + rr;
        float x = 0.f;
#pragma unroll
        for (int i = 0; i < CQ / 4; i++) {
            const float* dd = s_d + qr * CQ + 4 * i;
            x = fmaf(pv[ps][i].x, dd[0], fmaf(pv[ps][i].y, dd[1], fmaf(pv[ps][i].z, dd[2], fmaf(pv[ps][i].w, dd[3], x))));
        }
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if (a < D && qr == 0) s_u[a] = x;
    }
    __syncthreads();
    // gbar = mu_k . u
    {
        float g = tid < D ? s_mk[tid] * s_u[tid] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
        if (lane == 0) s_red[warp] = g;
    }
    __syncthreads();
    float gbar = 0.f;
#pragma unroll
    for (int w = 0; w < NWM; w++) gbar += s_red[w];
    // o_e = mu_v,e + (sum_c w_c (M_c u)_e) / l - gbar mu_v,e
#pragma unroll
    for (int ps = 0; ps < NPASS; ps++) {
        const int e = ps * RPP + rr;
        float x = 0.f;
#pragma unroll
        for (int c = 0; c < kPre; c++) {
            float y = 0.f;
#pragma unroll
            for (int i = 0; i < CQ / 4; i++) {
                const float* uu = s_u + qr * CQ + 4 * i;
                const float4 mv4 = mpre[c][ps][i];
                y = fmaf(mv4.x, uu[0], fmaf(mv4.y, uu[1], fmaf(mv4.z, uu[2], fmaf(mv4.w, uu[3], y))));
            }
            x = fmaf(s_w[c], y, x);
        }
        for (int c = kPre; c < nc; c++) {  // chunks beyond the first kPre, loaded here
            const float* pc = pb + (size_t)c * C::PART;
            float y = 0.f;
            if (e < D) {
                const float4* mr = (const float4*)(pc + 4 + 2 * D + (size_t)e * D + qr * CQ);
                float4 mv4[CQ / 4];
#pragma unroll
                for (int i = 0; i < CQ / 4; i++) mv4[i] = mr[i];
#pragma unroll
                for (int i = 0; i < CQ / 4; i++) {
                    const float* uu = s_u + qr * CQ + 4 * i;
                    y = fmaf(mv4[i].x, uu[0], fmaf(mv4[i].y, uu[1], fmaf(mv4[i].z, uu[2], fmaf(mv4[i].w, uu[3], y))));
                }
            }
            x = fmaf(exp2f(pc[0] - m), y, x);
        }
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        if (e < D && qr == 0) out[(size_t)bh * D + e] = __float2bfloat16_rn(s_mv[e] + x * inv - gbar * s_mv[e]);
    }
    if (tid == 0) lse[bh] = (m + __log2f(l)) * LN2;
}


// ------------------------------------------------------- given-probe decode
// The layer in the form the paper states it, with the probe rho supplied by
// the caller ("Parallax: Parameterized Local Linear Attention for Language
// Modeling", technical summary, "Core mechanism": o = o^SA - Sigma_KV rho):
// with r_i = k_i . rho,
//   Sigma_KV rho = sum_i p_i (v_i - mu_v)(k_i - mu_k) . rho
//                = sum_i p_i r_i v_i - (sum_i p_i r_i) mu_v,
// so o = mu_v - sum_i p_i r_i v_i + (sum_i p_i r_i) mu_v, and every term is a
// softmax-weighted sum over the keys: one pass over K and V, as the pages'
// decode kernel runs both branches over one KV stream ("Hardware-aware
// algorithm").  No matrix product remains, so the chunk kernel runs on the
// CUDA cores and keeps, with an online softmax, l = sum p, sum p r, sum p v
// and sum p r v.
// Work split: the keys of all heads form one sequence of KT-key tiles, head
// after head (ntile = ceil(Lmax / KT) tiles per head, G = B H ntile in all).
// CTA c of N takes tiles [c G / N, (c + 1) G / N), so every CTA streams the
// same number of bytes, and with N = MIN_CTAS CTAs per SM so does every SM
// (whole heads per CTA would leave some SMs a third more work than others).
// A CTA writes one partial per head its range touches, into slot c + h
// (distinct for every overlapping pair); a second kernel merges the partials
// of a head by their log-sum-exp.
template <int D>
struct DecP {
    static constexpr int TPK = D / 32;       // threads per key (32 features each)
    static constexpr int KT = 128 / TPK;     // keys per tile
    static constexpr int NW = 4, NT = 32 * NW;
    static constexpr int MIN_CTAS = 3;
    static constexpr int NS = 4;             // K|V stages
    static constexpr int TB = KT * D * 2;    // one K or V tile: 8 KB
    static constexpr int QS = 34;            // stride of a 32-feature part of q and rho in shared memory
    static constexpr int NBAR = NS;          // full[NS]
    static constexpr int RED = NW * (2 * D + 2);  // per-warp sums of one partial
    static constexpr int SMEM = 1024 + NS * 2 * TB + NBAR * 8 + 16 + 2 * NW * 4 + 2 * TPK * QS * 4 + RED * 4 + 16;
    static_assert(MIN_CTAS * (SMEM + 1024) <= 233472, "MIN_CTAS CTAs fit an SM's shared memory");
    static_assert(2 * NW <= 8, "the two tile-parity copies of the warp maxima fit their slot");
    // partial of one (CTA, head): {m, l, sum p r, pad}, sum p v [D], sum p r v [D]
    static constexpr int PART = 4 + 2 * D;
};

template <int D>
__global__ void __launch_bounds__(DecP<D>::NT, DecP<D>::MIN_CTAS)
    decp_chunk(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ rho,
               const int* __restrict__ lens, int H, int Lmax, int ntile, long long G, float scale_log2,
               float* __restrict__ part, unsigned* status) {
    using C = DecP<D>;
    constexpr int NS = C::NS, KT = C::KT, TPK = C::TPK, NW = C::NW, NT = C::NT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sKV = sm;  // stage s: K at 2 s TB, V at (2 s + 1) TB
    uint64_t* full = (uint64_t*)(sKV + NS * 2 * C::TB);
    uint32_t* holder = (uint32_t*)(full + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);
    float* wmax = (float*)(holder + 4);  // [2][NW]: tile max per warp, by tile parity
    float* sq = wmax + 8;                // q, fp32, parts of 32 at stride QS
    float* sr = sq + TPK * C::QS;        // rho likewise
    float* red = sr + TPK * C::QS;       // [NW][2 D + 2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long N = gridDim.x, cta = blockIdx.x;
    const long long g0 = cta * G / N, g1 = (cta + 1) * G / N;  // this CTA's tiles
    const int h0 = (int)(g0 / ntile), h1 = (int)((g1 - 1) / ntile);
    const Watchdog wd{status, abortf, KID_DECODE, wait_limit(status)};
    // the merge may be launched now: it waits for this whole grid to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        *abortf = 0;
        for (int s = 0; s < NS; s++) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // tiles [tb, tv) of head h lie in this CTA's range and hold keys of the sequence
    auto range = [&](int h, int& tb, int& tv) {
        const long long hb = (long long)h * ntile;
        tb = (int)(max(g0, hb) - hb);
        const int te = (int)(min(g1, hb + ntile) - hb);
        const int len = seq_len1(lens, h / H, Lmax);
        tv = max(tb, min(te, (len + KT - 1) / KT));
    };
    int total = 0;  // tiles this CTA streams
    for (int h = h0; h <= h1; h++) {
        int tb, tv;
        range(h, tb, tv);
        total += tv - tb;
    }
    // The loader (lane 0 of the last warp) walks the same tiles, NS ahead of
    // the workers: tile n of the walk goes to stage n % NS.
    const bool loader = threadIdx.x == (NW - 1) * 32;
    int lh = h0, lt = 0, le = 0, issued = 0;
    if (loader) range(lh, lt, le);
    auto load_next = [&]() {
        while (lt >= le) range(++lh, lt, le);  // issued < total: a head with tiles follows
        const int s = issued % NS;
        mbar_expect_tx(&full[s], 2 * C::TB);
#pragma unroll
        for (int r = 0; r < D / 64; r++) {
            tma_load_3d(sKV + (2 * s) * C::TB + r * KT * 128, &tm_k, r * 64, lt * KT, lh, &full[s]);
            tma_load_3d(sKV + (2 * s + 1) * C::TB + r * KT * 128, &tm_v, r * 64, lt * KT, lh, &full[s]);
        }
        lt++;
        issued++;
    };
    if (loader) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        while (issued < NS && issued < total) load_next();
    }
    // lane = fp * KW + kl: thread = (key r of the tile, feature part fp)
    constexpr int KW = 32 / TPK;
    const int kl = lane % KW, fp = lane / KW;
    const int r = warp * KW + kl;
    const int f0 = fp * 32;
    const float* qf = sq + fp * C::QS;
    const float* rf = sr + fp * C::QS;
    bool ok = true;
    int n = 0;  // tiles consumed
    for (int h = h0; h <= h1 && ok; h++) {
        int tb, tv;
        range(h, tb, tv);
        const int len = seq_len1(lens, h / H, Lmax);
        workers_sync(NT);  // every read of the previous head's q, rho and partial sums is done
        for (int i = threadIdx.x; i < D; i += NT) {
            sq[(i >> 5) * C::QS + (i & 31)] = __bfloat162float(q[(size_t)h * D + i]);
            sr[(i >> 5) * C::QS + (i & 31)] = __bfloat162float(rho[(size_t)h * D + i]);
        }
        workers_sync(NT);
        uint64_t av[16], arv[16];  // sum p v, sum p r v over this thread's keys, as f32x2 pairs
#pragma unroll
        for (int i = 0; i < 16; i++) av[i] = arv[i] = 0;
        float l = 0.f, lr = 0.f, m_run = -INFINITY;
        for (int t = tb; t < tv; t++, n++) {
            const int s = n % NS;
            ok = mbar_wait(&full[s], (n / NS) & 1, wd, 2) && ok;
            if (!__all_sync(0xffffffffu, ok)) ok = false;
            const uint8_t* sk = sKV + (2 * s) * C::TB;
            const uint8_t* sv = sKV + (2 * s + 1) * C::TB;
            const int key = t * KT + r;
            const bool valid = key < len;
            // q . k and rho . k over this thread's 32 features, summed over the key's threads
            uint64_t dq[2] = {0, 0}, dr[2] = {0, 0};
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint4 kc = *(const uint4*)(sk + swz(r, f0 + 8 * c, KT));
                const uint32_t w[4] = {kc.x, kc.y, kc.z, kc.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const uint64_t kk = f2(bf16_lo(w[e]), bf16_hi(w[e]));
                    const float2 qq = *(const float2*)(qf + 8 * c + 2 * e);
                    const float2 rr = *(const float2*)(rf + 8 * c + 2 * e);
                    dq[c & 1] = ffma2(f2(qq.x, qq.y), kk, dq[c & 1]);
                    dr[c & 1] = ffma2(f2(rr.x, rr.y), kk, dr[c & 1]);
                }
            }
            const float2 q01 = uf2(fadd2(dq[0], dq[1])), r01 = uf2(fadd2(dr[0], dr[1]));
            float dot = q01.x + q01.y, rk = r01.x + r01.y;
#pragma unroll
            for (int o = KW; o < 32; o <<= 1) {
                dot += __shfl_xor_sync(0xffffffffu, dot, o);
                rk += __shfl_xor_sync(0xffffffffu, rk, o);
            }
            const float sc = valid ? dot * scale_log2 : -INFINITY;
            float tmax = sc;
#pragma unroll
            for (int o = 1; o < KW; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            // two copies by tile parity: a warp that runs ahead writes the next
            // tile's maximum while a slower one may still read this tile's
            float* wm = wmax + (n & 1) * NW;
            if (lane == 0) wm[warp] = tmax;
            // every worker has finished tile n - 1 past this barrier: its stage
            // takes tile n - 1 + NS
            if (!workers_and(ok, NT)) {
                ok = false;
                break;
            }
            if (loader && n >= 1 && issued < total && issued == n - 1 + NS) {
                fence_proxy_async_smem();
                load_next();
            }
            float tm = wm[0];
#pragma unroll
            for (int w = 1; w < NW; w++) tm = fmaxf(tm, wm[w]);
            const float m_new = fmaxf(m_run, tm);
            if (m_new > m_run + RESCALE_TH) {  // uniform across the CTA
                const float alpha = fast_exp2_dec(m_run - m_new);
                m_run = m_new;
                l *= alpha;
                lr *= alpha;
                const uint64_t A2 = f2(alpha, alpha);
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    av[i] = fmul2(av[i], A2);
                    arv[i] = fmul2(arv[i], A2);
                }
            }
            const float p = valid ? fast_exp2_dec(sc - m_run) : 0.f;
            const float pr = valid ? p * rk : 0.f;  // a key past the sequence adds nothing (its row may hold anything)
            if (fp == 0) {
                l += p;
                lr += pr;
            }
            const uint64_t P2 = f2(p, p), PR2 = f2(pr, pr);
#pragma unroll
            for (int c = 0; c < 4 && valid; c++) {  // a row past the sequence may hold NaN: not read
                const uint4 vc = *(const uint4*)(sv + swz(r, f0 + 8 * c, KT));
                const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const uint64_t vv = f2(bf16_lo(vw[e]), bf16_hi(vw[e]));
                    av[4 * c + e] = ffma2(P2, vv, av[4 * c + e]);
                    arv[4 * c + e] = ffma2(PR2, vv, arv[4 * c + e]);
                }
            }
        }
        if (!ok) break;
        // the partial of (this CTA, head h): sums over the KW key threads of
        // each warp by a reduce-scatter (each round a lane keeps half of its
        // values and adds the partner's copy of that half: 64 - 64 / KW
        // shuffles in all), then over the warps in shared memory.  Value j of
        // the 64 (sum p v of feature f0 + j, then sum p r v) ends in lane
        // kl = j / (64 / KW).
        float x[64];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const float2 a2 = uf2(av[i]), b2 = uf2(arv[i]);
            x[2 * i] = a2.x;
            x[2 * i + 1] = a2.y;
            x[32 + 2 * i] = b2.x;
            x[32 + 2 * i + 1] = b2.y;
        }
#pragma unroll
        for (int o = KW / 2, hs = 32; o >= 1; o >>= 1, hs >>= 1) {
            const bool upper = (kl & o) != 0;  // this lane keeps the upper half
#pragma unroll
            for (int i = 0; i < hs; i++) {
                const float send = upper ? x[i] : x[i + hs];
                const float keep = upper ? x[i + hs] : x[i];
                x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
#pragma unroll
        for (int o = 1; o < KW; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            lr += __shfl_xor_sync(0xffffffffu, lr, o);
        }
        {
            constexpr int PER = 64 / KW;  // values per lane after the reduce-scatter
            float* rw = red + warp * (2 * D + 2);
#pragma unroll
            for (int i = 0; i < PER; i++) {
                const int j = PER * kl + i;
                rw[(j < 32 ? f0 + j : D + f0 + j - 32)] = x[i];
            }
            if (lane == 0) {
                rw[2 * D] = l;
                rw[2 * D + 1] = lr;
            }
        }
        workers_sync(NT);
        float* dst = part + (size_t)(cta + h) * C::PART;
        for (int e = threadIdx.x; e < 2 * D + 2; e += NT) {
            float x = 0.f;
            for (int w = 0; w < NW; w++) x += red[w * (2 * D + 2) + e];
            if (e < 2 * D) dst[4 + e] = x;
            else dst[1 + (e - 2 * D)] = x;  // l, then sum p r
        }
        if (threadIdx.x == 0) dst[0] = m_run;
    }
    // an aborted CTA's partials weigh 0 in the merge
    if (!ok && threadIdx.x == 0)
        for (int h = h0; h <= h1; h++) part[(size_t)(cta + h) * C::PART] = -INFINITY;
    // loads issued but not consumed (only after an abort) land before the CTA exits
    if (loader)
        for (int jj = issued > NS ? issued - NS : 0; jj < issued; jj++) mbar_wait_drain(&full[jj % NS], (jj / NS) & 1);
}

// Merge the partials of one head: m = max m_c, weights 2^(m_c - m), then
// o = mu_v - (sum p r v) / l + ((sum p r) / l) mu_v and lse.  One thread per
// feature.  The partials of head h are those of CTAs c(h ntile) .. c(h ntile +
// ntile - 1), where c(g) = ((g + 1) N - 1) / G is the CTA whose range holds tile g.
template <int D>
__global__ void __launch_bounds__(D) decp_merge(const float* part, int ntile, long long G, int N,
                                                float* __restrict__ lse, __nv_bfloat16* __restrict__ out) {
    using C = DecP<D>;
    // the partials are read only past this wait: `part` is not declared
    // __restrict__, so the compiler may not move their loads above it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bh = blockIdx.x, e = threadIdx.x;
    const long long ga = (long long)bh * ntile, gb = ga + ntile - 1;
    const int ca = (int)(((ga + 1) * N - 1) / G), cb = (int)(((gb + 1) * N - 1) / G);
    // every load of a partial is issued before any of them is used: a few
    // partials per head, so the merge costs one round trip
    constexpr int MAXP = 8;
    float pm[MAXP], pl[MAXP], plr[MAXP], ppv[MAXP], pprv[MAXP];
    float m = -INFINITY, l = 0.f, lr = 0.f, pv = 0.f, prv = 0.f;
    for (int c0 = ca; c0 <= cb; c0 += MAXP) {
#pragma unroll
        for (int i = 0; i < MAXP; i++) {
            const float* pc = part + (size_t)(c0 + i + bh) * C::PART;
            const bool in = c0 + i <= cb;
            pm[i] = in ? pc[0] : -INFINITY;
            pl[i] = in ? pc[1] : 0.f;
            plr[i] = in ? pc[2] : 0.f;
            ppv[i] = in ? pc[4 + e] : 0.f;
            pprv[i] = in ? pc[4 + D + e] : 0.f;
        }
        float mm = m;
#pragma unroll
        for (int i = 0; i < MAXP; i++) mm = fmaxf(mm, pm[i]);
        const float a = m == -INFINITY ? 0.f : exp2f(m - mm);  // rescale what is summed so far
        l *= a;
        lr *= a;
        pv *= a;
        prv *= a;
#pragma unroll
        for (int i = 0; i < MAXP; i++) {
            if (pm[i] == -INFINITY) continue;  // no keys of this head in that CTA
            const float w = exp2f(pm[i] - mm);
            l = fmaf(w, pl[i], l);
            lr = fmaf(w, plr[i], lr);
            pv = fmaf(w, ppv[i], pv);
            prv = fmaf(w, pprv[i], prv);
        }
        m = mm;
    }
    const float inv = 1.f / l;
    const float mv = pv * inv;
    out[(size_t)bh * D + e] = __float2bfloat16_rn(mv - prv * inv + lr * inv * mv);
    if (e == 0) lse[bh] = (m + __log2f(l)) * LN2;
}

// ----------------------------------------------------------------- host
#define PLX_TRY(x)                         \
    do {                                   \
        cudaError_t e_ = (x);              \
        if (e_ != cudaSuccess) return e_;  \
    } while (0)

// Chunks per head: at most kMaxCtas / (B H) (so the partials' workspace is
// bounded without knowing the device), at most one per 64 keys.
constexpr int kMaxCtas = 1024;

size_t dec1_nchunk_max(size_t BH, int Lmax) {
    const size_t by_keys = ((size_t)Lmax + 63) / 64;
    const size_t by_ctas = BH >= (size_t)kMaxCtas ? 1 : (kMaxCtas + BH - 1) / BH;
    return by_keys < by_ctas ? by_keys : by_ctas;
}

// Per device, once: the SM count; the kernel's shared-memory attributes are
// set at the same time.  Resident CTAs per SM are the kernel's design point
// (MIN_CTAS: its launch bounds keep the registers within it, and MIN_CTAS
// times its shared memory fits an SM), not an occupancy query.
struct Dec1Dev {
    int sms = 0, occ = 0;
};
template <int D>
cudaError_t dec1_device(Dec1Dev* out) {
    static Dec1Dev cache[64];
    static std::mutex mu;
    int dev = 0;
    PLX_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        using C = Dec1<D>;
        Dec1Dev x;
        PLX_TRY(cudaFuncSetAttribute(dec1_chunk<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        PLX_TRY(cudaFuncSetAttribute(dec1_chunk<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared));
        PLX_TRY(cudaDeviceGetAttribute(&x.sms, cudaDevAttrMultiProcessorCount, dev));
        x.occ = C::MIN_CTAS;
        cache[dev] = x;
    }
    *out = cache[dev];
    return cudaSuccess;
}

template <int D>
cudaError_t decode_tc_impl(const DecodeArgs& a) {
    using C = Dec1<D>;
    const int BH = a.B * a.H;
    Dec1Dev dv;
    PLX_TRY(dec1_device<D>(&dv));
    // one wave of resident CTAs: chunks per head, rounded to whole 64-key tiles
    const size_t cap = dec1_nchunk_max(BH, a.Lmax);
    size_t per_head = (size_t)dv.sms * dv.occ / BH;
    if (per_head < 1) per_head = 1;
    if (per_head > cap) per_head = cap;
    int chunk = (int)((a.Lmax + per_head - 1) / per_head);
    chunk = (chunk + C::KT - 1) / C::KT * C::KT;
    const int nchunk = (a.Lmax + chunk - 1) / chunk;
    CUtensorMap mk, mv;
    if (!tc_make_map(&mk, a.k, D, a.Lmax, BH, C::KT) || !tc_make_map(&mv, a.v, D, a.Lmax, BH, C::KT))
        return cudaErrorInvalidValue;
    const float scale_log2 = LOG2E / sqrtf((float)D);
    float* part = (float*)a.ws;
    timing_begin(a.stream, "dec_chunk");
    dec1_chunk<D><<<dim3(nchunk, BH), C::NT, C::SMEM, a.stream>>>(mk, mv, (const __nv_bfloat16*)a.q, a.lens, a.H,
                                                                   a.Lmax, chunk, scale_log2, part, a.status);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "dec_merge");
    {  // programmatic dependent launch: the merge's launch and its P_h and q
       // loads overlap the chunk kernel's last CTAs
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(BH);
        cfg.blockDim = dim3(kMergeThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        PLX_TRY(cudaLaunchKernelEx(&cfg, dec1_merge<D>, (const __nv_bfloat16*)a.q, (const int*)a.lens,
                                   (const float*)a.P, (const float*)part, a.H, a.Lmax, chunk, nchunk, a.lse,
                                   (__nv_bfloat16*)a.out));
    }
    timing_end(a.stream);
    return cudaGetLastError();
}


// ---- given-probe decode
template <int D>
cudaError_t decode_probe_impl(const DecodeArgs& a) {
    using C = DecP<D>;
    const int BH = a.B * a.H;
    static int sms_cache[64];
    static std::mutex mu;
    int dev = 0;
    PLX_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sms_cache[dev] == 0) {
            PLX_TRY(cudaFuncSetAttribute(decp_chunk<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
            PLX_TRY(cudaFuncSetAttribute(decp_chunk<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared));
            PLX_TRY(cudaDeviceGetAttribute(&sms_cache[dev], cudaDevAttrMultiProcessorCount, dev));
        }
        sms = sms_cache[dev];
    }
    // the tiles of all heads split evenly over one wave of resident CTAs
    const int ntile = (a.Lmax + C::KT - 1) / C::KT;
    const long long G = (long long)BH * ntile;
    const int N = (int)std::min<long long>(std::min<long long>((long long)sms * C::MIN_CTAS, G), kMaxCtas);
    CUtensorMap mk, mv;
    if (!tc_make_map(&mk, a.k, D, a.Lmax, BH, C::KT) || !tc_make_map(&mv, a.v, D, a.Lmax, BH, C::KT))
        return cudaErrorInvalidValue;
    const float scale_log2 = LOG2E / sqrtf((float)D);
    float* part = (float*)a.ws;
    timing_begin(a.stream, "decp_chunk");
    decp_chunk<D><<<N, C::NT, C::SMEM, a.stream>>>(mk, mv, (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.rho,
                                                   a.lens, a.H, a.Lmax, ntile, G, scale_log2, part, a.status);
    timing_end(a.stream);
    PLX_TRY(cudaGetLastError());
    timing_begin(a.stream, "decp_merge");
    {  // programmatic dependent launch: the chunk kernel releases it at its start
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(BH);
        cfg.blockDim = dim3(D);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        PLX_TRY(cudaLaunchKernelEx(&cfg, decp_merge<D>, (const float*)part, ntile, G, N, a.lse,
                                   (__nv_bfloat16*)a.out));
    }
    timing_end(a.stream);
    return cudaGetLastError();
}
}  // namespace

size_t decode_tc_ws_bytes(int B, int H, int Lmax, int d) {
    const size_t BH = (size_t)B * H;
    const size_t part = d == 64 ? (size_t)Dec1<64>::PART : (size_t)Dec1<128>::PART;
    return align256(BH * dec1_nchunk_max(BH, Lmax) * part * sizeof(float));
}

cudaError_t decode_tc(const DecodeArgs& a) {
    if (a.dtype != 1 || !tc_available()) return cudaErrorNotSupported;
    return a.d == 64 ? decode_tc_impl<64>(a) : decode_tc_impl<128>(a);
}

size_t decode_probe_ws_bytes(int B, int H, int Lmax, int d) {
    (void)Lmax;
    const size_t BH = (size_t)B * H;
    const size_t part = d == 64 ? (size_t)DecP<64>::PART : (size_t)DecP<128>::PART;
    return align256((kMaxCtas + BH) * part * sizeof(float));  // slots c + h, c < kMaxCtas
}

cudaError_t decode_probe(const DecodeArgs& a) {
    if (a.dtype != 1 || !tc_available() || !a.rho) return cudaErrorNotSupported;
    return a.d == 64 ? decode_probe_impl<64>(a) : decode_probe_impl<128>(a);
}

}  // namespace plx
