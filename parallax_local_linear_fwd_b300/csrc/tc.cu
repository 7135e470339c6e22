// Tensor-core (tcgen05 / TMEM / TMA) kernels for the Parallax attention layer,
// sm_103a.  Inputs are bf16; every MMA operand is f16 with fp32 accumulation:
// the inputs convert to f16 exactly (within its range), and the operands the
// path itself rounds (P~, u, the pass-2 and backward weights) keep three more
// mantissa bits than bf16 would, which the stated output tolerance needs.
//
// Layer ("Parallax: Parameterized Local Linear Attention for Language
// Modeling", technical summary, "Core mechanism" and "Hardware-aware
// algorithm"; probe u = P_h (q - mu_k)):
//   pass 1 (tc_pass1_pp): S = c Q K^T on a key tile, online softmax,
//                       Mu += P~ K; emits lse and mu_k = Mu / l; then the
//   projection        : u = P_h (q - mu_k) rounded to f16, gbar = mu_k . u.
//   pass 2 (tc_dual at d = 64, tc_dual_w at d = 128): S = c Q K^T and
//                       G = U K^T on the SAME key tile in shared memory (both
//                       branches read one KV stream); weights p (1 + g - gbar)
//                       with p from the stored lse; O += W V.
//   backward B1 (tc_dual / tc_dual_pp, second mode): S = c Q K^T and
//                       E = dO V^T; weights p e; R += W K and ebar = sum p e.
//   backward B2 (tc_b2, tc_rows): the row math, the dP_h partials.
//   backward B3 (tc_bwd_b3_q64 at d = 64, tc_bwd_b3 at d = 128): dK, dV, dQ.
//
// Warp roles in the tensor-core kernels: warp 0 issues TMA loads, warp 1 owns
// TMEM and issues MMAs (one elected thread; some kernels give a second warp
// the accumulation MMAs), and warpgroups of four warps move scores between
// TMEM and registers (one TMEM lane = one row) and write results.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <functional>
#include <mutex>

#include "plx_internal.h"
#include "tc_ptx.cuh"

namespace plx {
namespace {

using namespace tc;

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
// Online-softmax rescale threshold (log2 units): the running max is only
// moved when a row max exceeds it by more than this, so p~ <= 2^8.
constexpr float RESCALE_TH = 8.f;

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Launch order of (tile, head) work items: heads in groups of kHeadGroup, and
// within a group the longest tiles first (rank 0 = most work).  CTAs that run
// at the same time then share a few heads' K/V (and dQ rows) in L2 instead of
// streaming every head's, while the causal triangle still starts heavy-first.
constexpr int kHeadGroup = 8;
__device__ __forceinline__ void work_item(int item, int BH, int ntiles, int* rank, int* bh) {
    const int per_group = kHeadGroup * ntiles;
    const int g = item / per_group;
    const int gsize = min(kHeadGroup, BH - g * kHeadGroup);
    const int r = item - g * per_group;
    *rank = r / gsize;
    *bh = g * kHeadGroup + r % gsize;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Byte offset of the 16-byte chunk holding columns [c, c + 8) of row r in a
// swizzled 16-bit tile of `rows` rows (column blocks of 64).
__device__ __forceinline__ uint32_t sw_off(int r, int c, int rows) {
    return (uint32_t)((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}

// ======================================================= pass 1, two query tiles
// Pass 1 with one CTA per SM holding two adjacent query
// tiles, a = 2m and b = 2m + 1, which read the same key tiles (b one more):
// every K tile is loaded once for both, and warpgroup 0 (warps 2-5) runs
// tile a's softmax while warpgroup 1 (warps 6-9) runs tile b's, so the
// tensor core works on one tile while the other's weights are formed.  The
// MMA thread issues, per key tile j:
//   Mu_a += P~_a(j) K,  S_a(j+1),  Mu_b += P~_b(j) K,  S_b(j+1)
// The projection U = delta P_h^T of both tiles runs once every key MMA is
// done: delta_a (hi, lo) goes to K stages 0, 1 and delta_b to stages 2, 3,
// and P_h (f16, one head, both tiles) sits in a slot of its own, written by
// the converter warps once the first key stages are converted.
// Q and K arrive as the bf16 inputs and are converted to f16 in shared
// memory: each softmax warpgroup converts its Q tile once (and writes its q
// rows in f16 for pass 2); warps 10-11 convert each K tile as soon as it
// lands, up to NS tiles ahead of its MMAs, and produce the other f16 copies
// pass 2 reads: this CTA's own two K tiles (keys [256 m, 256 m + 256), by a
// TMA store of the converted tile) and V rows [256 m, 256 m + 256).
// TMEM: tile x at column 256 x: S [0,128) (P~ aliases [0,64); U after the
// loop), Mu [128, 128 + D).
template <int D>
struct P1PP {
    static constexpr int BM = 128, BN = 128, NT = 384;
    static constexpr int NS = D == 64 ? 6 : 4;  // K stages, shared by both tiles
    static constexpr int QB = BM * D * 2;
    static constexpr int KB = BN * D * 2;
    static constexpr int PB = D * D * 2;  // P_h in f16
    // q_full, k_full[NS], k_empty[NS], k16[NS], q16[2], s_full[2], p_full[2],
    // o_done[2], kfree, cdone, ph_full, proj_ready[2], proj_done[2], drain, v_full
    static constexpr int NBAR = 1 + 3 * NS + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 2 + 2 + 1 + 1;
    static constexpr int SMEM = 1024 + 2 * QB + NS * KB + PB + NBAR * 8 + 16;
    static constexpr unsigned TMEM_COLS = 512;
    static_assert(NS >= 4 && KB == QB, "the projection of each tile takes two K stages");
    static_assert(SMEM <= 232448, "one CTA per SM must fit");
};

template <int D>
__global__ void __launch_bounds__(P1PP<D>::NT, 1)
    tc_pass1_pp(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_k16, const __grid_constant__ CUtensorMap tm_mu,
                const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_q16,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_v16,
                const float* __restrict__ P, float* __restrict__ lse, float* __restrict__ gbar,
                int T, int H, int BH, int npairs, float scale_log2, int* item_ctr, unsigned* status) {
    // (item_ctr, when given: the work counter of the persistent pass 2 that
    // follows on the same stream, set to zero here)
    using C = P1PP<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sQ = sm;                // tile x at x QB
    uint8_t* sK = sQ + 2 * C::QB;    // stage s at s KB
    uint8_t* sP = sK + NS * C::KB;   // P_h (f16, K-major [a][b]): the projections' B operand
    uint64_t* bars = (uint64_t*)(sP + C::PB);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + NS;     // the MMA thread and the converter leader
    uint64_t* k16 = k_empty + NS;        // stage s holds K in f16
    uint64_t* q16r = k16 + NS;           // [2] tile x's Q in f16
    uint64_t* s_full = q16r + 2;         // [2]
    uint64_t* p_full = s_full + 2;       // [2]
    uint64_t* o_done = p_full + 2;       // [2]
    uint64_t* kfree = o_done + 2;        // every MMA reading a K stage has completed (one phase)
    uint64_t* cdone = kfree + 1;         // the converters' K stores have read their stages (one phase)
    uint64_t* ph_full = cdone + 1;       // P_h staged in f16 (one phase)
    uint64_t* proj_ready = ph_full + 1;  // [2] delta_x staged
    uint64_t* proj_done = proj_ready + 2;  // [2] U_x in TMEM
    uint64_t* drain = proj_done + 2;
    uint64_t* v_full = drain + 1;        // the pair's V rows (bf16) are in K stages 0-1 (one phase)
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    work_item(blockIdx.x, BH, npairs, &rank, &bh);
    const int m = npairs - 1 - rank;  // longest pairs first
    const int q0a = 2 * m * C::BM, q0b = q0a + C::BM;
    const int nkta = min(q0a + C::BM - 1, T - 1) / C::BN + 1;
    const int nktb = q0b < T ? min(q0b + C::BM - 1, T - 1) / C::BN + 1 : 0;
    const int nk = nktb > nkta ? nktb : nkta;
    const int ntiles = nktb > 0 ? 2 : 1;
    const Watchdog wd{status, abortf, KID_TC_PASS1, wait_limit(status)};
    if (item_ctr && blockIdx.x == 0 && threadIdx.x == 0) *item_ctr = 0;
    // pass 2, launched as a programmatic dependent, may be scheduled once
    // every CTA of this grid has started (it waits for this grid's completion
    // before it reads anything written here)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 2);
            mbar_init(&k16[s], 1);
        }
        for (int x = 0; x < 2; x++) {
            mbar_init(&q16r[x], 128);
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 128);
            mbar_init(&o_done[x], 1);
            mbar_init(&proj_ready[x], 128);
            mbar_init(&proj_done[x], 1);
        }
        mbar_init(kfree, 1);
        mbar_init(cdone, 1);
        mbar_init(ph_full, 1);
        mbar_init(drain, 1);
        mbar_init(v_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_k16);
            mbar_expect_tx(q_full, ntiles * C::QB);
            for (int x = 0; x < ntiles; x++) {
#pragma unroll
                for (int r = 0; r < D / 64; r++)
                    tma_load_3d(sQ + x * C::QB + r * C::BM * 128, &tm_q, r * 64, x ? q0b : q0a, bh, q_full);
            }
            int issued = 0;
            for (int j = 0; j < nk; j++) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(&k_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&k_full[s], C::KB);
#pragma unroll
                for (int r = 0; r < D / 64; r++)
                    tma_load_3d(sK + s * C::KB + r * C::BN * 128, &tm_k, r * 64, j * C::BN, bh, &k_full[s]);
                issued = j + 1;
            }
            // Every load issued must land before the CTA may exit.
            mbar_wait_drain(q_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&k_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1) {
        // The whole warp runs the issue loop (warp-uniform descriptors); the
        // elected lane issues every tcgen05 instruction, in order.
        const uint32_t idS = idesc_mma(128, C::BN, false, false);
        const uint32_t idM = idesc_mma(128, D, false, true);
        auto scores = [&](int x, int j) {  // S_x(j) = Q_x K_j^T
            const uint32_t qaddr = smem_u32(sQ + x * C::QB), kaddr = smem_u32(sK + (j % NS) * C::KB);
            const uint32_t tS = tmem + 256 * x;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tS, desc_kmajor(qaddr, C::BM, kk), desc_kmajor(kaddr, C::BN, kk), idS, kk > 0);
                mma_commit(&s_full[x]);
            }
            __syncwarp();
        };
        auto accumulate = [&](int x, int j) {  // Mu_x += P~_x(j) K_j (K read MN-major)
            const uint32_t kaddr = smem_u32(sK + (j % NS) * C::KB);
            const uint32_t tS = tmem + 256 * x, tMu = tS + 128;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; kk++)
                    mma_ts(tMu, tS + kk * 8, desc_mnmajor(kaddr, C::BN, kk), idM, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&o_done[x]);
            }
            __syncwarp();
        };
        // every operand in f16: the Q tiles and key tile 0 converted
        bool ok = __all_sync(0xffffffffu, mbar_wait(&q16r[0], 0, wd, 2)) &&
                  (nktb == 0 || __all_sync(0xffffffffu, mbar_wait(&q16r[1], 0, wd, 2))) &&
                  __all_sync(0xffffffffu, mbar_wait(&k16[0], 0, wd, 3));
        if (ok) {
            tc_fence_after();
            scores(0, 0);
            if (nktb > 0) scores(1, 0);
        }
        for (int j = 0; ok && j < nk; j++) {
            // S_x(j + 1) aliases P~_x(j): the accumulation reading it is issued
            // first, and MMAs issued by one thread run in order
            if (j < nkta) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&p_full[0], j & 1, wd, 5)))) break;
                tc_fence_after();
                accumulate(0, j);
            }
            if (j + 1 < nk) {  // key tile j + 1, converted to f16
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&k16[(j + 1) % NS], ((j + 1) / NS) & 1, wd, 3))))
                    break;
                tc_fence_after();
                if (j + 1 < nkta) scores(0, j + 1);
            }
            if (j < nktb) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&p_full[1], j & 1, wd, 6)))) break;
                tc_fence_after();
                accumulate(1, j);
            }
            if (elect_one()) mma_commit(&k_empty[j % NS]);  // every MMA reading key tile j is issued
            __syncwarp();
            if (j + 1 < nktb) scores(1, j + 1);
        }
        if (ok) {
            if (elect_one()) mma_commit(kfree);
            __syncwarp();
            // projections U_x = delta_x P_h^T (delta = hi + lo, P_h in f16 in its
            // slot): M = 128 rows, N = D, K = D, into S_x's columns
            const uint32_t idP = idesc_mma(128, D, false, false);
            const uint32_t pb = smem_u32(sP);
            for (int x = 0; x < ntiles; x++) {
                if (!__all_sync(0xffffffffu, mbar_wait(ph_full, 0, wd, 9))) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&proj_ready[x], 0, wd, 10))) break;
                tc_fence_after();
                const uint32_t dhi = smem_u32(sK + (2 * x) * C::KB), dlo = smem_u32(sK + (2 * x + 1) * C::KB);
                const uint32_t tS = tmem + 256 * x;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tS, desc_kmajor(dhi, C::BM, kk), desc_kmajor(pb, D, kk), idP, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tS, desc_kmajor(dlo, C::BM, kk), desc_kmajor(pb, D, kk), idP, 1u);
                    mma_commit(&proj_done[x]);
                }
                __syncwarp();
            }
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else if (warp >= 10) {
        // converters (warps 10-11): K tile j to f16 in place as soon as it
        // lands; P_h to f16 once the first stages are done (tile NS arrives
        // only after tile 0's scores complete); then this pair's V rows,
        // while the softmax warpgroups finish
        const int ct = threadIdx.x - 320;  // 0..63
        const int ph_at = min(nk, NS) - 1;
        bool ok = true;
        for (int j = 0; j < nk; j++) {
            const int s = j % NS;
            ok = mbar_wait(&k_full[s], (j / NS) & 1, wd, 13);
            if (!named_bar_and(3, 64, ok)) {
                ok = false;
                break;
            }
            uint4* tile = (uint4*)(sK + s * C::KB);
#pragma unroll 4
            for (int c = ct; c < C::KB / 16; c += 64) {
                const uint4 x = tile[c];
                tile[c] = make_uint4(pack_f16_sat(bf16_lo(x.x), bf16_hi(x.x)), pack_f16_sat(bf16_lo(x.y), bf16_hi(x.y)),
                                     pack_f16_sat(bf16_lo(x.z), bf16_hi(x.z)), pack_f16_sat(bf16_lo(x.w), bf16_hi(x.w)));
            }
            fence_proxy_async_smem();
            named_bar_sync(3, 64);
            if (ct == 0) {
                mbar_arrive(&k16[s]);
                // this pair's own key tiles go to the f16 copy pass 2 reads
                if ((j >> 1) == m && j * C::BN < T) {
#pragma unroll
                    for (int r = 0; r < D / 64; r++)
                        tma_store_3d(&tm_k16, r * 64, j * C::BN, bh, sK + s * C::KB + r * C::BN * 128);
                    bulk_commit();
                    bulk_wait_read_all();  // the stage may be reloaded once the store has read it
                }
                mbar_arrive(&k_empty[s]);
            }
            if (j == ph_at) {
                // P_h (fp32, row a = output index) as the K-major B operand of
                // both projections: rows = a, K = b
                const float* Ph = P + (size_t)(bh % H) * D * D;
#pragma unroll 8
                for (int id = ct; id < D * D / 8; id += 64) {
                    const int pa = id / (D / 8), pb0 = (id % (D / 8)) * 8;
                    const float4 x0 = *(const float4*)(Ph + pa * D + pb0);
                    const float4 x1 = *(const float4*)(Ph + pa * D + pb0 + 4);
                    *(uint4*)(sP + sw_off(pa, pb0, D)) = make_uint4(pack_f16(x0.x, x0.y), pack_f16(x0.z, x0.w),
                                                                    pack_f16(x1.x, x1.y), pack_f16(x1.z, x1.w));
                }
                fence_proxy_async_smem();
                named_bar_sync(3, 64);
                if (ct == 0) mbar_arrive(ph_full);
            }
        }
        if (ct == 0) {
            bulk_wait_all();
            if (ok) mbar_arrive(cdone);  // the K stages may now take delta
        }
        // V rows [q0a, q0a + 256) of head bh in f16, through K stages 0-1 once
        // both projections have read their delta tiles there: one tensor load
        // per 128 x 64 box, conversion in place, one tensor store per box
        if (ok) ok = mbar_wait(&proj_done[0], 0, wd, 16);
        if (ok && ntiles > 1) ok = mbar_wait(&proj_done[1], 0, wd, 16);
        ok = named_bar_and(3, 64, ok);
        if (ok) {
            const int vt = min(2, (T - q0a + C::BM - 1) / C::BM);  // 128-row V tiles of this pair
            if (ct == 0) {
                mbar_expect_tx(v_full, vt * C::KB);
                for (int rt = 0; rt < vt; rt++)
#pragma unroll
                    for (int r = 0; r < D / 64; r++)
                        tma_load_3d(sK + rt * C::KB + r * C::BN * 128, &tm_v, r * 64, q0a + rt * C::BM, bh, v_full);
            }
            ok = named_bar_and(3, 64, mbar_wait(v_full, 0, wd, 17));
            if (ok) {
                uint4* tile = (uint4*)sK;
#pragma unroll 4
                for (int c = ct; c < vt * C::KB / 16; c += 64) {
                    const uint4 x = tile[c];
                    tile[c] = make_uint4(pack_f16_sat(bf16_lo(x.x), bf16_hi(x.x)), pack_f16_sat(bf16_lo(x.y), bf16_hi(x.y)),
                                         pack_f16_sat(bf16_lo(x.z), bf16_hi(x.z)), pack_f16_sat(bf16_lo(x.w), bf16_hi(x.w)));
                }
                fence_proxy_async_smem();
                named_bar_sync(3, 64);
                if (ct == 0) {
                    for (int rt = 0; rt < vt; rt++)
#pragma unroll
                        for (int r = 0; r < D / 64; r++)
                            tma_store_3d(&tm_v16, r * 64, q0a + rt * C::BM, bh, sK + rt * C::KB + r * C::BN * 128);
                    bulk_commit();
                }
            } else if (ct == 0) {
                mbar_wait_drain(v_full, 0);  // the loads land before the CTA exits
            }
        }
        if (ct == 0) bulk_wait_all();
    } else if (warp >= 2) {
        // softmax / epilogue warpgroup x: thread <-> query row (TMEM lane)
        const int x = (warp - 2) >> 2;
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const int q0 = x ? q0b : q0a;
        const int t = q0 + row;
        const int my_nkt = x ? nktb : nkta;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        const uint32_t tS = tmem + 256 * x, tMu = tS + 128;
        uint8_t* sQx = sQ + x * C::QB;
        float m_use = -INFINITY, l = 0.f;
        bool ok = my_nkt > 0;
        if (ok) {
            // this thread's q row to f16, in place in the Q tile (the MMA operand)
            ok = mbar_wait(q_full, 0, wd, 14);
            if (__all_sync(0xffffffffu, ok)) {
#pragma unroll 4
                for (int c = 0; c < D / 8; c++) {
                    const uint32_t off = sw_off(row, 8 * c, C::BM);
                    const uint4 x8 = *(const uint4*)(sQx + off);
                    const uint4 h8 = make_uint4(pack_f16_sat(bf16_lo(x8.x), bf16_hi(x8.x)),
                                                pack_f16_sat(bf16_lo(x8.y), bf16_hi(x8.y)),
                                                pack_f16_sat(bf16_lo(x8.z), bf16_hi(x8.z)),
                                                pack_f16_sat(bf16_lo(x8.w), bf16_hi(x8.w)));
                    *(uint4*)(sQx + off) = h8;
                }
                fence_proxy_async_smem();
                mbar_arrive(&q16r[x]);
                // the f16 tile, once all its rows are converted, to the copy
                // pass 2 reads: one tensor store per 64 columns
                if (qd == 0 && lane == 0 && mbar_wait(&q16r[x], 0, wd, 18)) {
#pragma unroll
                    for (int r = 0; r < D / 64; r++) tma_store_3d(&tm_q16, r * 64, q0, bh, sQx + r * (C::BM * 128));
                    bulk_commit();
                }
            } else {
                ok = false;
            }
        }
        for (int j = 0; j < my_nkt; j++) {
            ok = mbar_wait(&s_full[x], j & 1, wd, 6);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * C::BN;
            const int lim = (k0 + C::BN - 1 > q0) ? t - k0 : C::BN;  // key k0 + c valid iff c <= lim
            // the row's whole score tile in registers: one TMEM round trip
            uint32_t v[C::BN];
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) tmem_ld32(tS + lrow + c * 32, *reinterpret_cast<uint32_t(*)[32]>(v + c * 32));
            tmem_wait_ld();
            if (lim < C::BN) {  // the diagonal tile only: masked keys score -inf (weight 0)
#pragma unroll
                for (int i = 0; i < C::BN; i++)
                    if (i > lim) v[i] = __float_as_uint(-INFINITY);
            }
            float mx;
            {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < C::BN; i += 8)
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        m4[u] = fmax3(m4[u], __uint_as_float(v[i + 2 * u]), __uint_as_float(v[i + 2 * u + 1]));
                mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
            }
            mx *= scale_log2;
            const float m_new = fmaxf(m_use, mx);
            const bool need = m_new > m_use + RESCALE_TH;
            float alpha = 1.f;
            if (need) {
                alpha = fast_exp2(m_use - m_new);
                m_use = m_new;
            }
            l *= alpha;
            const uint64_t SL2 = f2(scale_log2, scale_log2), NM2 = f2(-m_use, -m_use);
            uint64_t sum2 = f2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {  // keys 2i, 2i + 1: one f32x2 op each (2^-inf = 0)
                    const uint32_t* vv = v + c * 32 + 2 * i;
                    const float2 xx = uf2(ffma2(f2(__uint_as_float(vv[0]), __uint_as_float(vv[1])), SL2, NM2));
                    const float p0 = fast_exp2(xx.x), p1 = fast_exp2(xx.y);
                    sum2 = fadd2(sum2, f2(p0, p1));
                    pk[i] = pack_f16(p0, p1);
                }
                tmem_st16(tS + lrow + c * 16, pk);
            }
            const float2 sp = uf2(sum2);
            l += sp.x + sp.y;
            // rescale the accumulator to the moved maximum; the previous tile's
            // P~ K has completed (this tile's scores were issued after it)
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                ok = mbar_wait(&o_done[x], (j - 1) & 1, wd, 7);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    tmem_wait_st();
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; c++) {
                    uint32_t u[32];
                    tmem_ld32(tMu + lrow + c * 32, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                    tmem_st32(tMu + lrow + c * 32, u);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }
        // the last P~ K of this tile, then every MMA that reads a K stage
        if (ok) ok = mbar_wait(&o_done[x], (my_nkt - 1) & 1, wd, 8);
        if (ok) ok = mbar_wait(kfree, 0, wd, 11);
        if (ok) ok = mbar_wait(cdone, 0, wd, 15);
        // The four warps agree on ok before the projection (whose steps
        // synchronise on a named barrier): an abort anywhere skips it.
        ok = named_bar_and(1 + x, 128, ok);
        // one thread of the warpgroup issues its tensor stores (mu_k, U)
        const bool leader = qd == 0 && lane == 0;
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            const size_t grow = (size_t)bh * T + t;
            uint8_t* sDhi = sK + (2 * x) * C::KB;
            uint8_t* sDlo = sK + (2 * x + 1) * C::KB;
            // delta = q - mu_k (mu_k = Mu / l) split into f16 hi + lo, written
            // as the K-major A tile of the projection; this thread's q row is
            // read in full here, before its own mu_k row overwrites it below
#pragma unroll 1
            for (int c = 0; c < D / 32; c++) {
                uint32_t u[32];
                tmem_ld32(tMu + lrow + c * 32, u);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; g++) {
                    const uint32_t off = sw_off(row, c * 32 + g * 8, C::BM);
                    const uint4 qv = *(const uint4*)(sQx + off);  // f16 q
                    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float d0 = f16_lo(qw[e]) - __uint_as_float(u[g * 8 + 2 * e]) * inv;
                        const float d1 = f16_hi(qw[e]) - __uint_as_float(u[g * 8 + 2 * e + 1]) * inv;
                        hi[e] = pack_f16(d0, d1);
                        lo[e] = pack_f16(d0 - f16_lo(hi[e]), d1 - f16_hi(hi[e]));
                    }
                    *(uint4*)(sDhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *(uint4*)(sDlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&proj_ready[x]);
            // mu_k (output, fp32) through tile x's Q slot while the projection
            // runs: 32-column boxes (128-byte swizzle), as many per round as
            // the slot holds (D / 64), one tensor store per box; row t of a
            // box lies in row t of the Q tile's own bytes, so each thread
            // overwrites only its q row
            constexpr int BPR = C::QB / (C::BM * 128);  // boxes per round
            static_assert(BPR >= 1 && (D / 32) % BPR == 0, "the Q slot holds whole boxes");
#pragma unroll 1
            for (int r2 = 0; r2 < D / 32 / BPR; r2++) {
                // the previous tensor store from the slot (the f16 q copy, then
                // the previous round) has read it
                if (leader) bulk_wait_read_all();
                named_bar_sync(1 + x, 128);
#pragma unroll 1
                for (int b2 = 0; b2 < BPR; b2++) {
                    uint32_t u[32];
                    tmem_ld32(tMu + lrow + (r2 * BPR + b2) * 32, u);
                    tmem_wait_ld();
                    uint8_t* box = sQx + b2 * (C::BM * 128) + row * 128;
#pragma unroll
                    for (int y = 0; y < 8; y++)
                        *(uint4*)(box + ((y ^ (row & 7)) << 4)) =
                            make_uint4(__float_as_uint(__uint_as_float(u[4 * y]) * inv),
                                       __float_as_uint(__uint_as_float(u[4 * y + 1]) * inv),
                                       __float_as_uint(__uint_as_float(u[4 * y + 2]) * inv),
                                       __float_as_uint(__uint_as_float(u[4 * y + 3]) * inv));
                }
                fence_proxy_async_smem();
                named_bar_sync(1 + x, 128);
                if (leader) {
#pragma unroll
                    for (int b2 = 0; b2 < BPR; b2++)
                        tma_store_3d(&tm_mu, (r2 * BPR + b2) * 32, q0, bh, sQx + b2 * (C::BM * 128));
                    bulk_commit();
                }
            }
            ok = mbar_wait(&proj_done[x], 0, wd, 12);
            // the U stores below meet on the named barrier: agree first
            ok = named_bar_and(1 + x, 128, ok);
            if (ok) {
                tc_fence_after();
                if (leader) bulk_wait_read_all();  // the mu_k stores have read the Q slot
                named_bar_sync(1 + x, 128);
                float g = 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; c++) {
                    uint32_t vu[32], vm[32];
                    tmem_ld32(tS + lrow + c * 32, vu);
                    tmem_ld32(tMu + lrow + c * 32, vm);
                    tmem_wait_ld();
                    uint32_t uh[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        uh[i] = pack_f16(__uint_as_float(vu[2 * i]), __uint_as_float(vu[2 * i + 1]));
                        g = fmaf(__uint_as_float(vm[2 * i]) * inv, f16_lo(uh[i]), g);
                        g = fmaf(__uint_as_float(vm[2 * i + 1]) * inv, f16_hi(uh[i]), g);
                    }
                    // U (f16) in the Q tile's own layout, then one tensor store per 64 columns
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        *(uint4*)(sQx + sw_off(row, c * 32 + 8 * i, C::BM)) =
                            make_uint4(uh[4 * i], uh[4 * i + 1], uh[4 * i + 2], uh[4 * i + 3]);
                }
                fence_proxy_async_smem();
                named_bar_sync(1 + x, 128);
                if (leader) {
#pragma unroll
                    for (int r = 0; r < D / 64; r++) tma_store_3d(&tm_u, r * 64, q0, bh, sQx + r * (C::BM * 128));
                    bulk_commit();
                }
                if (t < T) {
                    lse[grow] = (m_use + __log2f(l)) * LN2;
                    gbar[grow] = g;
                }
            }
        }
        // the tensor stores have read shared memory (and completed) before the CTA exits
        if (leader) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ====================================================== f16 operand copies
// The MMAs take f16 operands: a bf16 input converts to f16 exactly when its
// magnitude lies in f16's normal range (larger magnitudes saturate to the
// largest finite f16; tiny ones keep an absolute error below 2^-25).
struct CvtJob {
    const uint4* src[4];
    uint4* dst[4];
};

__global__ void __launch_bounds__(256) tc_to_f16(CvtJob job, size_t n8) {
    const uint4* __restrict__ src = job.src[blockIdx.y];
    uint4* __restrict__ dst = job.dst[blockIdx.y];
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 x = src[i];
        dst[i] = make_uint4(pack_f16_sat(bf16_lo(x.x), bf16_hi(x.x)), pack_f16_sat(bf16_lo(x.y), bf16_hi(x.y)),
                            pack_f16_sat(bf16_lo(x.z), bf16_hi(x.z)), pack_f16_sat(bf16_lo(x.w), bf16_hi(x.w)));
    }
}

// The dual-score pass's accumulator to global memory through shared memory,
// by the four-warp group that owns TMEM lanes 0-127 (thread = row): MODE 0
// writes out (bf16) in the A1 slot's 16-bit tile layout, MODE 1 writes R
// (fp32) in 32-column boxes (128-byte swizzle) over the A1 and A2 slots, which
// lie back to back; both slots are free once the accumulation has completed.
// The group meets on named barrier `bar`, then `leader` issues one tensor
// store per box (rows past T are not written).
template <int D, int MODE>
__device__ __forceinline__ void dual_store_acc(uint32_t tAcc, uint32_t lrow, int row, uint8_t* slot, int bar,
                                               bool leader, const CUtensorMap* tm_out, int q0, int bh) {
    constexpr int BM = 128;
#pragma unroll 1
    for (int c = 0; c < D / 32; c++) {
        uint32_t v[32];
        tmem_ld32(tAcc + lrow + c * 32, v);
        tmem_wait_ld();
        if (MODE == 0) {
#pragma unroll
            for (int i = 0; i < 4; i++)
                *(uint4*)(slot + sw_off(row, c * 32 + 8 * i, BM)) =
                    make_uint4(pack_bf16(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1])),
                               pack_bf16(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3])),
                               pack_bf16(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5])),
                               pack_bf16(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7])));
        } else {
            uint8_t* box = slot + c * (BM * 128) + row * 128;
#pragma unroll
            for (int y = 0; y < 8; y++)
                *(uint4*)(box + ((y ^ (row & 7)) << 4)) = make_uint4(v[4 * y], v[4 * y + 1], v[4 * y + 2], v[4 * y + 3]);
        }
    }
    fence_proxy_async_smem();
    named_bar_sync(bar, 128);
    if (leader) {
        if (MODE == 0) {
#pragma unroll
            for (int r = 0; r < D / 64; r++) tma_store_3d(tm_out, r * 64, q0, bh, slot + r * (BM * 128));
        } else {
#pragma unroll
            for (int c = 0; c < D / 32; c++) tma_store_3d(tm_out, c * 32, q0, bh, slot + c * (BM * 128));
        }
        bulk_commit();
        bulk_wait_all();  // the slot stays valid until the stores have read it
    }
}

// ======================================================== dual-score pass
// MODE 0 (forward pass 2): X = U K^T, W = p (x + 1 - gbar), Acc += W V, out = Acc.
// MODE 1 (backward B1)   : X = dO V^T, W = p x,           Acc += W K, R = Acc,
//                          ebar = sum_i W (fp32, before rounding).
// The weights W have TMEM columns of their own, so the MMA thread issues the
// next key tile's S and X as soon as the elementwise warps have read this
// tile's (before they have formed W), and the accumulation of W after them:
// the scores of tile j + 1 run while tile j's weights are formed.
template <int D>
struct DualCfg {
    static constexpr int BM = 128, BN = 64;
    static constexpr int NS = D == 64 ? 4 : 1;  // K+V stages
    static constexpr int AB = BM * D * 2;       // one A tile (Q, U or dO)
    static constexpr int KB = BN * D * 2;       // one K or V tile
    static constexpr int NBAR = 1 + 2 * NS + 4 + 2;  // + sx_free, w_free
    static constexpr int NT = 224;  // TMA warp, S|X MMA warp, 4 elementwise warps, accumulation MMA warp
    static constexpr int SMEM = 1024 + 2 * AB + NS * 2 * KB + NBAR * 8 + 16;
    static constexpr unsigned TMEM_COLS = 256;  // S [0,64), X [64,128), W [128,160), Acc [160,160+D)
};

template <int D, int MODE>
__global__ void __launch_bounds__(DualCfg<D>::NT, 2)
    tc_dual(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
            const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
            const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ lse,
            const float* __restrict__ gbar, float* __restrict__ ebar_out, int T, int BH, int ntq, float scale_log2,
            unsigned* status) {
    using C = DualCfg<D>;
    constexpr int NS = C::NS;
    static_assert(D == 64, "the TMEM plan holds S, X, W and Acc for d = 64");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sA1 = sm;
    uint8_t* sA2 = sA1 + C::AB;
    uint8_t* sKV = sA2 + C::AB;  // stage s: K at s * 2KB, V at s * 2KB + KB
    uint64_t* bars = (uint64_t*)(sKV + NS * 2 * C::KB);
    uint64_t* a_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = bars + 1 + NS;
    uint64_t* s_full = bars + 1 + 2 * NS;
    uint64_t* w_full = s_full + 1;
    uint64_t* acc_done = s_full + 2;
    uint64_t* drain = s_full + 3;
    uint64_t* sx_free = s_full + 4;  // the elementwise warps have read S and X of the tile (128 arrivals)
    uint64_t* w_free = s_full + 5;   // the accumulation has read W of the tile
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    work_item(blockIdx.x, BH, ntq, &rank, &bh);
    const int qt = ntq - 1 - rank;
    const int q0 = qt * C::BM;
    const int nkt = min(q0 + C::BM - 1, T - 1) / C::BN + 1;
    const Watchdog wd{status, abortf, MODE == 0 ? (unsigned)KID_TC_PASS2 : (unsigned)KID_TC_BWD_B1, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(a_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 2);  // a commit from each issuing warp
        }
        mbar_init(s_full, 1);
        mbar_init(w_full, 128);
        mbar_init(acc_done, 1);
        mbar_init(drain, 2);
        mbar_init(sx_free, 128);
        mbar_init(w_free, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t tS = tmem, tX = tmem + 64, tW = tmem + 128, tAcc = tmem + 160;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_a1);
            prefetch_tmap(&tm_a2);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(a_full, 2 * C::AB);
#pragma unroll
            for (int r = 0; r < D / 64; r++) {
                tma_load_3d(sA1 + r * C::BM * 128, &tm_a1, r * 64, q0, bh, a_full);
                tma_load_3d(sA2 + r * C::BM * 128, &tm_a2, r * 64, q0, bh, a_full);
            }
            int issued = 0;
            for (int j = 0; j < nkt; j++) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(&kv_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&kv_full[s], 2 * C::KB);
                uint8_t* st = sKV + s * 2 * C::KB;
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    tma_load_3d(st + r * C::BN * 128, &tm_k, r * 64, j * C::BN, bh, &kv_full[s]);
                    tma_load_3d(st + C::KB + r * C::BN * 128, &tm_v, r * 64, j * C::BN, bh, &kv_full[s]);
                }
                issued = j + 1;
            }
            mbar_wait_drain(a_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&kv_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1 || warp == C::NT / 32 - 1) {
        // Two issuing warps: warp 1 issues S and X, the last warp the
        // accumulation, so one warp's barrier waits overlap the other's MMAs.
        // Neither overwrites what the other's MMAs read: S and X are released
        // by the elementwise warps (sx_free), W by the accumulation (w_free),
        // a K|V stage once both warps have committed their last read of it.
        // In each warp the elected lane (lane 0 of the converged warp) issues
        // all of its tcgen05 instructions, in order.
        const uint32_t a1 = smem_u32(sA1), a2 = smem_u32(sA2);
        if (warp == 1) {
            const uint32_t idS = idesc_mma(128, C::BN, false, false);
            bool ok = __all_sync(0xffffffffu, mbar_wait(a_full, 0, wd, 2));
            for (int j = 0; ok && j < nkt; j++) {
                const int s = j % NS;
                if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[s], (j / NS) & 1, wd, 3))) break;
                // tile j - 1's S and X are in registers: tile j's may overwrite them
                if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(sx_free, (j - 1) & 1, wd, 9))) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sKV + s * 2 * C::KB);
                const uint32_t xb = MODE == 0 ? kaddr : kaddr + C::KB;  // B of the second score product
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tS, desc_kmajor(a1, C::BM, kk), desc_kmajor(kaddr, C::BN, kk), idS, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tX, desc_kmajor(a2, C::BM, kk), desc_kmajor(xb, C::BN, kk), idS, kk > 0);
                    mma_commit(s_full);
                    mma_commit(&kv_empty[s]);  // this warp's last read of the stage
                }
                __syncwarp();
            }
        } else {
            const uint32_t idA = idesc_mma(128, D, false, true);
            for (int j = 0; j < nkt; j++) {
                const int s = j % NS;
                if (!__all_sync(0xffffffffu, mbar_wait(w_full, j & 1, wd, 5))) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sKV + s * 2 * C::KB);
                const uint32_t ab = MODE == 0 ? kaddr + C::KB : kaddr;  // B of the accumulation
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; kk++)
                        mma_ts(tAcc, tW + kk * 8, desc_mnmajor(ab, C::BN, kk), idA, (j > 0 || kk > 0) ? 1u : 0u);
                    if (j == nkt - 1) mma_commit(acc_done);  // one phase: the epilogue's only wait
                    mma_commit(w_free);
                    mma_commit(&kv_empty[s]);  // this warp's last read of the stage
                }
                __syncwarp();
            }
        }
        if (elect_one()) mma_commit(drain);  // one arrival per issuing warp
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const int t = q0 + row;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        const bool valid = t < T;
        const float L2 = valid ? lse[(size_t)bh * T + t] * LOG2E : 0.f;
        const float g1 = (MODE == 0 && valid) ? 1.f - gbar[(size_t)bh * T + t] : 0.f;
        const uint64_t SL2 = f2(scale_log2, scale_log2), NL2 = f2(-L2, -L2), G1 = f2(g1, g1);
        uint64_t rs2 = f2(0.f, 0.f);  // row sum of the rounded weights, as an (even, odd) pair
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            ok = mbar_wait(s_full, j & 1, wd, 6);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * C::BN;
            const int lim = (k0 + C::BN - 1 > q0) ? t - k0 : C::BN;
            const bool need_mask = lim < C::BN;
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) {
                uint32_t vs[32], vx[32];
                tmem_ld32(tS + lrow + c * 32, vs);
                tmem_ld32(tX + lrow + c * 32, vx);
                tmem_wait_ld();
                if (c == C::BN / 32 - 1) {  // S and X of the tile are in registers
                    tc_fence_before();
                    mbar_arrive(sx_free);
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {  // keys 2i, 2i + 1 of the chunk, one f32x2 op each
                    const int cc = c * 32 + 2 * i;
                    const float2 xs = uf2(ffma2(f2(__uint_as_float(vs[2 * i]), __uint_as_float(vs[2 * i + 1])),
                                                SL2, NL2));
                    float p0 = fast_exp2(xs.x), p1 = fast_exp2(xs.y);
                    if (need_mask) {
                        if (cc > lim) p0 = 0.f;
                        if (cc + 1 > lim) p1 = 0.f;
                    }
                    const uint64_t xv = f2(__uint_as_float(vx[2 * i]), __uint_as_float(vx[2 * i + 1]));
                    const float2 w = uf2(MODE == 0 ? fmul2(f2(p0, p1), fadd2(xv, G1)) : fmul2(f2(p0, p1), xv));
                    pk[i] = pack_f16(w.x, w.y);
                    // ebar sums the rounded weights the MMA sees, so that
                    // R - ebar mu_k = sum_i w_i (k_i - mu_k) holds for them.
                    if (MODE == 1) rs2 = fadd2(rs2, f2(f16_lo(pk[i]), f16_hi(pk[i])));
                }
                if (c == 0 && j > 0) {  // the previous tile's accumulation has read W
                    ok = mbar_wait(w_free, (j - 1) & 1, wd, 10);
                    tc_fence_after();
                }
                tmem_st16(tW + lrow + c * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(w_full);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
        }
        if (ok) ok = mbar_wait(acc_done, 0, wd, 8);
        // the group meets on a named barrier in the store below: agree first
        ok = named_bar_and(1, 128, ok);
        if (ok) {
            {
                tc_fence_after();
                dual_store_acc<D, MODE>(tAcc, lrow, row, sA1, 1, qd == 0 && lane == 0, &tm_out, q0, bh);
                if (MODE == 1 && valid) {
                    const float2 r2 = uf2(rs2);
                    ebar_out[(size_t)bh * T + t] = r2.x + r2.y;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================ dual-score pass, two query tiles
// The d = 128 form of tc_dual, used for B1 (the second mode); pass 2 at
// d = 128 runs tc_dual_w below.  Two 128-row A tiles (Q and U, or Q and dO)
// take 64 KB of shared memory per query tile, so two independent CTAs per SM
// leave room for one K|V stage each, and every key tile's load latency is
// exposed.  Here one CTA per SM holds two adjacent query tiles, a = 2m and
// b = 2m + 1, which read the same key tiles (b one 128-key block further):
// three K|V stages serve both, and each key tile is loaded once for the two.
// Warpgroup 0 (warps 2-5) forms tile a's weights and warpgroup 1 (warps 6-9)
// tile b's, so the tensor core works on one tile while the other tile's
// weights are formed.  The MMA thread issues, per key tile j:
//   Acc_a += W_a(j) V,  S_a(j+1) | X_a(j+1),  Acc_b += W_b(j) V,  S_b(j+1) | X_b(j+1)
// TMEM: tile x at column 256 x: S [0,64) (W aliases [0,32)), X [64,128),
// Acc [128,256).
template <int D>
struct DualPP {
    static constexpr int BM = 128, BN = 64, NT = 320;
    static constexpr int NS = 3;             // K+V stages, shared by both tiles
    static constexpr int AB = BM * D * 2;    // one A tile (Q, U or dO)
    static constexpr int KB = BN * D * 2;    // one K or V tile
    static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 2 + 1;
    static constexpr int SMEM = 1024 + 4 * AB + NS * 2 * KB + NBAR * 8 + 16;
    static constexpr unsigned TMEM_COLS = 512;
    static_assert(SMEM <= 232448, "one CTA per SM must fit");
};

template <int D, int MODE>
__global__ void __launch_bounds__(DualPP<D>::NT, 1)
    tc_dual_pp(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ lse,
               const float* __restrict__ gbar, float* __restrict__ ebar_out, int T, int BH, int npairs,
               float scale_log2, unsigned* status) {
    using C = DualPP<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sA = sm;                   // tile x: A1 at 2x AB, A2 at (2x + 1) AB
    uint8_t* sKV = sA + 4 * C::AB;      // stage s: K at s * 2KB, V at s * 2KB + KB
    uint64_t* bars = (uint64_t*)(sKV + NS * 2 * C::KB);
    uint64_t* a_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = kv_full + NS;
    uint64_t* s_full = kv_empty + NS;   // [2]
    uint64_t* w_full = s_full + 2;      // [2]
    uint64_t* acc_done = w_full + 2;    // [2]
    uint64_t* drain = acc_done + 2;
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    work_item(blockIdx.x, BH, npairs, &rank, &bh);
    const int m = npairs - 1 - rank;  // longest pairs first
    // tile a (x = 0) is always inside the sequence; tile b (x = 1) may lie past T
    const int q0a = 2 * m * C::BM, q0b = q0a + C::BM;
    const int nkta = min(q0a + C::BM - 1, T - 1) / C::BN + 1;
    const int nktb = q0b < T ? min(q0b + C::BM - 1, T - 1) / C::BN + 1 : 0;
    const int nk = nktb > nkta ? nktb : nkta;
    const int ntiles = nktb > 0 ? 2 : 1;
    const Watchdog wd{status, abortf, MODE == 0 ? (unsigned)KID_TC_PASS2 : (unsigned)KID_TC_BWD_B1, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(a_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int x = 0; x < 2; x++) {
            mbar_init(&s_full[x], 1);
            mbar_init(&w_full[x], 128);
            mbar_init(&acc_done[x], 1);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_a1);
            prefetch_tmap(&tm_a2);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(a_full, ntiles * 2 * C::AB);
            for (int x = 0; x < ntiles; x++) {
                const int qx = x ? q0b : q0a;
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    tma_load_3d(sA + (2 * x) * C::AB + r * C::BM * 128, &tm_a1, r * 64, qx, bh, a_full);
                    tma_load_3d(sA + (2 * x + 1) * C::AB + r * C::BM * 128, &tm_a2, r * 64, qx, bh, a_full);
                }
            }
            int issued = 0;
            for (int j = 0; j < nk; j++) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(&kv_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&kv_full[s], 2 * C::KB);
                uint8_t* st = sKV + s * 2 * C::KB;
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    tma_load_3d(st + r * C::BN * 128, &tm_k, r * 64, j * C::BN, bh, &kv_full[s]);
                    tma_load_3d(st + C::KB + r * C::BN * 128, &tm_v, r * 64, j * C::BN, bh, &kv_full[s]);
                }
                issued = j + 1;
            }
            mbar_wait_drain(a_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&kv_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1) {
        // The whole warp runs the issue loop (warp-uniform descriptors); the
        // elected lane issues every tcgen05 instruction, in order.
        const uint32_t idS = idesc_mma(128, C::BN, false, false);
        const uint32_t idA = idesc_mma(128, D, false, true);
        auto scores = [&](int x, int j) {  // S_x(j) = A1_x K_j^T, X_x(j) = A2_x (K or V)_j^T
            const uint32_t kaddr = smem_u32(sKV + (j % NS) * 2 * C::KB);
            const uint32_t xb = MODE == 0 ? kaddr : kaddr + C::KB;
            const uint32_t a1 = smem_u32(sA + (2 * x) * C::AB), a2 = smem_u32(sA + (2 * x + 1) * C::AB);
            const uint32_t tS = tmem + 256 * x, tX = tS + 64;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tS, desc_kmajor(a1, C::BM, kk), desc_kmajor(kaddr, C::BN, kk), idS, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tX, desc_kmajor(a2, C::BM, kk), desc_kmajor(xb, C::BN, kk), idS, kk > 0);
                mma_commit(&s_full[x]);
            }
            __syncwarp();
        };
        auto accumulate = [&](int x, int j) {  // Acc_x += W_x(j) (V or K)_j
            const uint32_t kaddr = smem_u32(sKV + (j % NS) * 2 * C::KB);
            const uint32_t ab = MODE == 0 ? kaddr + C::KB : kaddr;
            const uint32_t tS = tmem + 256 * x, tAcc = tS + 128;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; kk++)
                    mma_ts(tAcc, tS + kk * 8, desc_mnmajor(ab, C::BN, kk), idA, (j > 0 || kk > 0) ? 1u : 0u);
                if (j == (x ? nktb : nkta) - 1) mma_commit(&acc_done[x]);  // one phase: the epilogue's only wait
            }
            __syncwarp();
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(a_full, 0, wd, 2)) &&
                  __all_sync(0xffffffffu, mbar_wait(&kv_full[0], 0, wd, 3));
        if (ok) {
            tc_fence_after();
            scores(0, 0);
            if (nktb > 0) scores(1, 0);
        }
        for (int j = 0; ok && j < nk; j++) {
            // S_x(j + 1) aliases W_x(j): the accumulation that reads W_x(j)
            // is issued first, and MMAs issued by one thread run in order
            if (j < nkta) {
                if (!__all_sync(0xffffffffu, mbar_wait(&w_full[0], j & 1, wd, 5))) break;
                tc_fence_after();
                accumulate(0, j);
            }
            if (j + 1 < nk) {
                if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[(j + 1) % NS], ((j + 1) / NS) & 1, wd, 3))) break;
                tc_fence_after();
                if (j + 1 < nkta) scores(0, j + 1);
            }
            if (j < nktb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&w_full[1], j & 1, wd, 6))) break;
                tc_fence_after();
                accumulate(1, j);
            }
            // every MMA that reads key tile j has been issued
            if (elect_one()) mma_commit(&kv_empty[j % NS]);
            __syncwarp();
            if (j + 1 < nktb) scores(1, j + 1);
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int x = (warp - 2) >> 2;  // query tile of this warpgroup
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const int q0 = x ? q0b : q0a;
        const int t = q0 + row;
        const int my_nkt = x ? nktb : nkta;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        const uint32_t tS = tmem + 256 * x, tX = tS + 64, tAcc = tS + 128;
        const bool valid = t < T;
        const float L2 = valid ? lse[(size_t)bh * T + t] * LOG2E : 0.f;
        const float g1 = (MODE == 0 && valid) ? 1.f - gbar[(size_t)bh * T + t] : 0.f;
        const uint64_t SL2 = f2(scale_log2, scale_log2), NL2 = f2(-L2, -L2), G1 = f2(g1, g1);
        uint64_t rs2 = f2(0.f, 0.f);  // row sum of the rounded weights, as an (even, odd) pair
        bool ok = my_nkt > 0;
        for (int j = 0; j < my_nkt; j++) {
            ok = mbar_wait(&s_full[x], j & 1, wd, 7);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * C::BN;
            const int lim = (k0 + C::BN - 1 > q0) ? t - k0 : C::BN;
            const bool need_mask = lim < C::BN;
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) {
                uint32_t vs[32], vx[32];
                tmem_ld32(tS + lrow + c * 32, vs);
                tmem_ld32(tX + lrow + c * 32, vx);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {  // keys 2i, 2i + 1 of the chunk, one f32x2 op each
                    const int cc = c * 32 + 2 * i;
                    const float2 xs = uf2(ffma2(f2(__uint_as_float(vs[2 * i]), __uint_as_float(vs[2 * i + 1])),
                                                SL2, NL2));
                    float p0 = fast_exp2(xs.x), p1 = fast_exp2(xs.y);
                    if (need_mask) {
                        if (cc > lim) p0 = 0.f;
                        if (cc + 1 > lim) p1 = 0.f;
                    }
                    const uint64_t xv = f2(__uint_as_float(vx[2 * i]), __uint_as_float(vx[2 * i + 1]));
                    const float2 w = uf2(MODE == 0 ? fmul2(f2(p0, p1), fadd2(xv, G1)) : fmul2(f2(p0, p1), xv));
                    pk[i] = pack_f16(w.x, w.y);
                    if (MODE == 1) rs2 = fadd2(rs2, f2(f16_lo(pk[i]), f16_hi(pk[i])));
                }
                tmem_st16(tS + lrow + c * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&w_full[x]);
        }
        if (ok) ok = mbar_wait(&acc_done[x], 0, wd, 8);
        // the group meets on a named barrier in the store below: agree first
        // (a group whose tile lies past T has no work and takes no part)
        if (my_nkt > 0) ok = named_bar_and(1 + x, 128, ok);
        if (ok) {
            {
                tc_fence_after();
                dual_store_acc<D, MODE>(tAcc, lrow, row, sA + (2 * x) * C::AB, 1 + x, qd == 0 && lane == 0, &tm_out,
                                        q0, bh);
                if (MODE == 1 && valid) {
                    const float2 r2 = uf2(rs2);
                    ebar_out[(size_t)bh * T + t] = r2.x + r2.y;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================================ given probe
// The one-pass form with a probe rho supplied as input ("Parallax: Parameterized
// Local Linear Attention for Language Modeling", technical summary, "Core
// mechanism": o = o^SA - Sigma_KV rho, the probe from a learned projection of
// the layer input; "Hardware-aware algorithm": both branches on one KV stream).
// With r_i = k_i . rho and the softmax p:
//   Sigma_KV rho = sum_i p_i r_i v_i - rbar mu_v,   rbar = sum_i p_i r_i,
//   o = mu_v (1 + rbar) - sum_i p_i r_i v_i.
// Per key tile: S = Q K^T and R = rho K^T on the same K tile, online softmax,
// O1 += P~ V and O2 += (P~ o R) V with both weight tiles in TMEM; l and rbar
// sum the rounded weights the MMAs see, so constant values give that value
// exactly.  8 d MMA flops per causal pair, one pass.
template <int D>
struct ProbeCfg {
    static constexpr int BM = 128, BN = 64, NT = 192;
    static constexpr int NS = D == 64 ? 4 : 3;  // K+V stages
    static constexpr int AB = BM * D * 2;
    static constexpr int KB = BN * D * 2;
    static constexpr int NBAR = 1 + 2 * NS + 4;
    static constexpr int SMEM = 1024 + 2 * AB + NS * 2 * KB + NBAR * 8 + 16;
    // S [0,64) (P~ aliases [0,32)), R [64,128) (P~ o R aliases [64,96)), O1 [128,128+D), O2 [128+D, 128+2D)
    static constexpr unsigned TMEM_COLS = D == 64 ? 256 : 512;
    static constexpr int MIN_BLOCKS = D == 64 ? 2 : 1;
};

template <int D>
__global__ void __launch_bounds__(ProbeCfg<D>::NT, ProbeCfg<D>::MIN_BLOCKS)
    tc_probe_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int T, int BH, int ntq,
                    float scale_log2, unsigned* status) {
    using C = ProbeCfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sQ = sm;
    uint8_t* sR = sQ + C::AB;
    uint8_t* sKV = sR + C::AB;
    uint64_t* bars = (uint64_t*)(sKV + NS * 2 * C::KB);
    uint64_t* a_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = kv_full + NS;
    uint64_t* s_full = kv_empty + NS;
    uint64_t* p_full = s_full + 1;
    uint64_t* o_done = s_full + 2;
    uint64_t* drain = s_full + 3;
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int rank, bh;
    work_item(blockIdx.x, BH, ntq, &rank, &bh);
    const int qt = ntq - 1 - rank;
    const int q0 = qt * C::BM;
    const int nkt = min(q0 + C::BM - 1, T - 1) / C::BN + 1;
    const Watchdog wd{status, abortf, KID_TC_PROBE, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(a_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 128);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t tS = tmem, tR = tmem + 64, tO1 = tmem + 128, tO2 = tmem + 128 + D;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(a_full, 2 * C::AB);
#pragma unroll
            for (int r = 0; r < D / 64; r++) {
                tma_load_3d(sQ + r * C::BM * 128, &tm_q, r * 64, q0, bh, a_full);
                tma_load_3d(sR + r * C::BM * 128, &tm_r, r * 64, q0, bh, a_full);
            }
            int issued = 0;
            for (int j = 0; j < nkt; j++) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(&kv_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&kv_full[s], 2 * C::KB);
                uint8_t* st = sKV + s * 2 * C::KB;
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    tma_load_3d(st + r * C::BN * 128, &tm_k, r * 64, j * C::BN, bh, &kv_full[s]);
                    tma_load_3d(st + C::KB + r * C::BN * 128, &tm_v, r * 64, j * C::BN, bh, &kv_full[s]);
                }
                issued = j + 1;
            }
            mbar_wait_drain(a_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&kv_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1) {
        // The whole warp runs the issue loop, so the descriptors stay
        // warp-uniform; the elected lane (lane 0 of the converged warp) issues
        // every tcgen05 instruction, so one thread issues all MMAs, in order.
        const uint32_t idS = idesc_mma(128, C::BN, false, false);
        const uint32_t idO = idesc_mma(128, D, false, true);
        const uint32_t qa = smem_u32(sQ), ra = smem_u32(sR);
        if (__all_sync(0xffffffffu, mbar_wait(a_full, 0, wd, 2))) {
            for (int j = 0; j < nkt; j++) {
                const int s = j % NS;
                if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[s], (j / NS) & 1, wd, 3))) break;
                // S and R alias the previous tile's weights; tcgen05.mma ops issued by
                // one thread execute in issue order, so no wait for those MMAs here.
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sKV + s * 2 * C::KB), vaddr = kaddr + C::KB;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) {
                        const uint64_t kd = desc_kmajor(kaddr, C::BN, kk);
                        mma_ss(tS, desc_kmajor(qa, C::BM, kk), kd, idS, kk > 0);
                        mma_ss(tR, desc_kmajor(ra, C::BM, kk), kd, idS, kk > 0);
                    }
                    mma_commit(s_full);
                }
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(p_full, j & 1, wd, 5))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; kk++) {
                        const uint64_t vd = desc_mnmajor(vaddr, C::BN, kk);
                        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                        mma_ts(tO1, tS + kk * 8, vd, idO, acc);
                        mma_ts(tO2, tR + kk * 8, vd, idO, acc);
                    }
                    mma_commit(o_done);
                    mma_commit(&kv_empty[s]);
                }
                __syncwarp();
            }
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const int t = q0 + row;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        float m_use = -INFINITY, l = 0.f, rs = 0.f;
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            ok = mbar_wait(s_full, j & 1, wd, 6);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * C::BN;
            const int lim = (k0 + C::BN - 1 > q0) ? t - k0 : C::BN;  // key k0 + c valid iff c <= lim
            // the row's whole score tile in registers: one TMEM round trip
            uint32_t v[C::BN];
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) tmem_ld32(tS + lrow + c * 32, *reinterpret_cast<uint32_t(*)[32]>(v + c * 32));
            tmem_wait_ld();
            if (lim < C::BN) {  // the diagonal tile only: masked keys score -inf (weight 0)
#pragma unroll
                for (int i = 0; i < C::BN; i++)
                    if (i > lim) v[i] = __float_as_uint(-INFINITY);
            }
            float mx;
            {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < C::BN; i += 8)
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        m4[u] = fmax3(m4[u], __uint_as_float(v[i + 2 * u]), __uint_as_float(v[i + 2 * u + 1]));
                mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
            }
            mx *= scale_log2;
            const float m_new = fmaxf(m_use, mx);
            const bool need = m_new > m_use + RESCALE_TH;
            float alpha = 1.f;
            if (need) {
                alpha = fast_exp2(m_use - m_new);
                m_use = m_new;
            }
            l *= alpha;
            rs *= alpha;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                ok = mbar_wait(o_done, (j - 1) & 1, wd, 7);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 2 * D / 32; c++) {  // O1 and O2 are contiguous
                    uint32_t v[32];
                    tmem_ld32(tO1 + lrow + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st32(tO1 + lrow + c * 32, v);
                }
            }
            const uint64_t SL2 = f2(scale_log2, scale_log2), NM2 = f2(-m_use, -m_use);
            const bool need_mask = lim < C::BN;
            uint64_t l2 = f2(0.f, 0.f), rs2 = f2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < C::BN / 32; c++) {
                uint32_t vs[32], vr[32];
                tmem_ld32(tS + lrow + c * 32, vs);
                tmem_ld32(tR + lrow + c * 32, vr);
                tmem_wait_ld();
                uint32_t pk[16], wk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {  // keys 2i, 2i + 1: one f32x2 op each
                    const int cc = c * 32 + 2 * i;
                    const float2 x =
                        uf2(ffma2(f2(__uint_as_float(vs[2 * i]), __uint_as_float(vs[2 * i + 1])), SL2, NM2));
                    float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                    if (need_mask) {
                        if (cc > lim) p0 = 0.f;
                        if (cc + 1 > lim) p1 = 0.f;
                    }
                    const uint64_t p2 = f2(p0, p1);
                    const float2 w = uf2(fmul2(p2, f2(__uint_as_float(vr[2 * i]), __uint_as_float(vr[2 * i + 1]))));
                    pk[i] = pack_f16(p0, p1);
                    wk[i] = pack_f16(w.x, w.y);
                    l2 = fadd2(l2, f2(f16_lo(pk[i]), f16_hi(pk[i])));
                    rs2 = fadd2(rs2, f2(f16_lo(wk[i]), f16_hi(wk[i])));
                }
                tmem_st16(tS + lrow + c * 16, pk);
                tmem_st16(tR + lrow + c * 16, wk);
            }
            {
                const float2 a2 = uf2(l2), b2 = uf2(rs2);
                l += a2.x + a2.y;
                rs += b2.x + b2.y;
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok) {
            ok = mbar_wait(o_done, (nkt - 1) & 1, wd, 8);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float inv = 1.f / l, g = 1.f + rs * inv;
#pragma unroll 1
                for (int c = 0; c < D / 32; c++) {
                    uint32_t v1[32], v2[32];
                    tmem_ld32(tO1 + lrow + c * 32, v1);
                    tmem_ld32(tO2 + lrow + c * 32, v2);
                    tmem_wait_ld();
                    if (t < T) {
                        uint4* dst = (uint4*)(out + ((size_t)bh * T + t) * D + c * 32);
                        uint32_t o[16];
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            const float a0 = (__uint_as_float(v1[2 * i]) * g - __uint_as_float(v2[2 * i])) * inv;
                            const float a1 =
                                (__uint_as_float(v1[2 * i + 1]) * g - __uint_as_float(v2[2 * i + 1])) * inv;
                            o[i] = pack_bf16(a0, a1);
                        }
#pragma unroll
                        for (int i = 0; i < 4; i++) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
                }
                if (t < T) lse[(size_t)bh * T + t] = (m_use + __log2f(l)) * LN2;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================================= row math
// Per-row work around the attention passes, as register-tiled fp32 products
// over blocks of 64 rows of one head (rows = the B*T queries of head h):
//   MODE 0 (forward projection): u = P_h (q - mu_k), U = f16(u),
//          gbar = mu_k . U (from the rounded U, so that sum_i p_i (g_i - gbar)
//          vanishes for the values pass 2's MMA sees).
//   MODE 1 (backward B2): the same u, du = R - ebar mu_k, ddelta = P_h^T du,
//          dq_acc = ddelta, z = f16(dmu - ebar U) with dmu = -ddelta (B3's
//          operand in place of dmu: k . z = y - ebar g), the row scalars B3 needs
//          {-lse log2 e, 1 - mu_k . U, -ebar, -D} (stored by query pairs) with
//          D = do.o - gbar ebar + mu_k . dmu and do.o = ebar + R.u - gbar ebar
//          (rebuilt from B1's fp32 sums, gbar = mu_k . u in fp32), and this
//          CTA's partial dP_h = sum_rows du delta^T.
// Thread (ty, tx) of 16 x 16 owns rows 4ty..4ty+3 and columns NC tx..NC tx+NC-1.
template <int D>
struct RowCfg {
    static constexpr int RB = 64, NT = 256;
    static constexpr int LDT = RB + 4;  // stride of the transposed row tiles
    static constexpr int LDP = D + 4;   // stride of the P tiles
    static constexpr int NC = D / 16;   // output columns per thread
    static constexpr int NA = D / 16;   // dP rows (a) per thread
    static constexpr int ROWS_PER_CTA = 512;
    static constexpr int CPT = D / 4;  // columns per thread in the load phase (4 threads per row)
    // mu_k is kept row-major in shared memory unless that would not fit
    static constexpr bool mu_in_smem(int mode) { return D == 64 || mode == 0; }
    static constexpr size_t smem(int mode) {
        return sizeof(float) * ((mode ? 2 : 1) * (size_t)D * LDP + (mode ? 2 : 1) * (size_t)D * LDT +
                                (mu_in_smem(mode) ? (size_t)RB * LDP : 0));
    }
};

template <int D, int MODE>
__global__ void __launch_bounds__(256) tc_rows(const __nv_bfloat16* __restrict__ q, const float* __restrict__ mu_k,
                                               const float* __restrict__ P, const float* __restrict__ lse,
                                               const float* __restrict__ R, const float* __restrict__ ebar,
                                               __half* __restrict__ U, float* __restrict__ gbar,
                                               __half* __restrict__ dmu, float* __restrict__ dq_acc,
                                               float* __restrict__ rowpack, float* __restrict__ dp_partial,
                                               int B, int H, int T) {
    using C = RowCfg<D>;
    constexpr int NC = C::NC, NA = C::NA, LDT = C::LDT, LDP = C::LDP, RB = C::RB;
    extern __shared__ float rsm[];
    float* PT = rsm;                                    // PT[b][a] = P[a][b]
    float* PM = PT + D * LDP;                           // PM[a][b] = P[a][b]      (MODE 1)
    float* XT = MODE ? PM + D * LDP : PT + D * LDP;     // XT[b][r] = delta[r][b]
    float* YT = XT + D * LDT;                           // YT[a][r] = du[r][a]     (MODE 1)
    float* MS = MODE ? YT + D * LDT : YT;               // MS[r][c] = mu_k (when it fits)
    constexpr bool kMu = C::mu_in_smem(MODE);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int h = blockIdx.y;
    const float* Ph = P + (size_t)h * D * D;
    for (int e = tid; e < D * D; e += C::NT) {
        const float v = Ph[e];
        PT[(e % D) * LDP + e / D] = v;
        if (MODE) PM[(e / D) * LDP + e % D] = v;
    }
    const int nrows = B * T;
    const int r_begin = blockIdx.x * C::ROWS_PER_CTA;
    const int r_end = min(r_begin + C::ROWS_PER_CTA, nrows);
    float dp[NA][NA];
#pragma unroll
    for (int i = 0; i < NA; i++)
#pragma unroll
        for (int j = 0; j < NA; j++) dp[i][j] = 0.f;

    // Block loads: 4 threads per row, CPT consecutive columns each, 16-byte
    // loads into registers (fetch), then transposed into shared memory (put).
    // At d = 64 the next block's loads are issued as soon as the current
    // block is in shared memory, so they complete under this block's math.
    constexpr int CPT = C::CPT;
    constexpr bool kPrefetch = D == 64;
    struct Rows {
        uint4 qv[CPT / 8];
        float4 m[CPT / 4];
        float4 rv[MODE ? CPT / 4 : 1];
        float eb;
        bool ok;
    };
    const int rr = tid >> 2, c0 = (tid & 3) * CPT;
    auto fetch = [&](int r0_, Rows& x) {
        const int r = r0_ + rr;
        x.ok = r < r_end;
        if (!x.ok) return;
        const size_t base = (((size_t)(r / T) * H + h) * T + r % T) * D + c0;
        x.eb = MODE ? ebar[base / D] : 0.f;
#pragma unroll
        for (int k = 0; k < CPT / 8; k++) x.qv[k] = *(const uint4*)&q[base + 8 * k];
#pragma unroll
        for (int k = 0; k < CPT / 4; k++) x.m[k] = *(const float4*)&mu_k[base + 4 * k];
        if (MODE) {
#pragma unroll
            for (int k = 0; k < CPT / 4; k++) x.rv[k] = *(const float4*)&R[base + 4 * k];
        }
    };
    auto put = [&](const Rows& x) {
        if (x.ok) {
#pragma unroll
            for (int k = 0; k < CPT; k += 8) {
                const uint32_t qw[4] = {x.qv[k / 8].x, x.qv[k / 8].y, x.qv[k / 8].z, x.qv[k / 8].w};
                float m[8], rv[8];
                *(float4*)&m[0] = x.m[k / 4];
                *(float4*)&m[4] = x.m[k / 4 + 1];
                if (MODE) {
                    *(float4*)&rv[0] = x.rv[k / 4];
                    *(float4*)&rv[4] = x.rv[k / 4 + 1];
                }
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const float qf = (e & 1) ? bf16_hi(qw[e >> 1]) : bf16_lo(qw[e >> 1]);
                    XT[(c0 + k + e) * LDT + rr] = qf - m[e];
                    if (MODE) YT[(c0 + k + e) * LDT + rr] = rv[e] - x.eb * m[e];
                }
                if (kMu) {
                    *(float4*)&MS[rr * LDP + c0 + k] = *(float4*)&m[0];
                    *(float4*)&MS[rr * LDP + c0 + k + 4] = *(float4*)&m[4];
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < CPT; k++) {
                XT[(c0 + k) * LDT + rr] = 0.f;
                if (MODE) YT[(c0 + k) * LDT + rr] = 0.f;
            }
        }
    };
    Rows nxt;
    if (kPrefetch) fetch(r_begin, nxt);
    for (int r0 = r_begin; r0 < r_end; r0 += RB) {
        __syncthreads();
        if (kPrefetch) {
            put(nxt);
            if (r0 + RB < r_end) fetch(r0 + RB, nxt);
        } else {
            Rows cur;
            fetch(r0, cur);
            put(cur);
        }
        __syncthreads();
        // u = P delta for the thread's 4 rows x NC columns
        float u[4][NC];
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < NC; j++) u[i][j] = 0.f;
#pragma unroll 4
        for (int b = 0; b < D; b++) {
            const float4 x = *(const float4*)&XT[b * LDT + 4 * ty];
            const float xs[4] = {x.x, x.y, x.z, x.w};
            float pv[NC];
#pragma unroll
            for (int j = 0; j < NC; j += 4) *(float4*)&pv[j] = *(const float4*)&PT[b * LDP + NC * tx + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < NC; j++) u[i][j] = fmaf(xs[i], pv[j], u[i][j]);
        }
        float dd[4][NC];
        if (MODE) {
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < NC; j++) dd[i][j] = 0.f;
#pragma unroll 4
            for (int a = 0; a < D; a++) {
                const float4 y = *(const float4*)&YT[a * LDT + 4 * ty];
                const float ys[4] = {y.x, y.y, y.z, y.w};
                float pv[NC];
#pragma unroll
                for (int j = 0; j < NC; j += 4) *(float4*)&pv[j] = *(const float4*)&PM[a * LDP + NC * tx + j];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < NC; j++) dd[i][j] = fmaf(ys[i], pv[j], dd[i][j]);
            }
        }
        // per-row outputs
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int r = r0 + 4 * ty + i;
            const bool valid = r < r_end;
            const size_t row = valid ? ((size_t)(r / T) * H + h) * T + r % T : 0;
            const size_t off = row * D + NC * tx;
            float m[NC], rr_[NC];
            float gr = 0.f, gb = 0.f, ru = 0.f, xx = 0.f;
            uint32_t uh[NC / 2];
#pragma unroll
            for (int j = 0; j < NC; j += 2) uh[j / 2] = pack_f16(u[i][j], u[i][j + 1]);
            if (valid) {
#pragma unroll
                for (int j = 0; j < NC; j += 4)
                    *(float4*)&m[j] = kMu ? *(const float4*)&MS[(4 * ty + i) * LDP + NC * tx + j]
                                          : *(const float4*)&mu_k[off + j];
                if (MODE) {
#pragma unroll
                    for (int j = 0; j < NC; j += 4) *(float4*)&rr_[j] = *(const float4*)&R[off + j];
                }
#pragma unroll
                for (int j = 0; j < NC; j += 2) {
                    gr = fmaf(m[j], f16_lo(uh[j / 2]), gr);
                    gr = fmaf(m[j + 1], f16_hi(uh[j / 2]), gr);
                }
                if (MODE) {
#pragma unroll
                    for (int j = 0; j < NC; j++) {
                        gb = fmaf(m[j], u[i][j], gb);
                        ru = fmaf(rr_[j], u[i][j], ru);
                        xx = fmaf(m[j], -dd[i][j], xx);
                    }
                }
                if (NC == 4)
                    *(uint2*)&U[off] = make_uint2(uh[0], uh[1]);
                else
                    *(uint4*)&U[off] = make_uint4(uh[0], uh[1], uh[2], uh[3]);
                if (MODE) {
                    const float eb = ebar[row];
                    uint32_t mh[NC / 2];
#pragma unroll
                    for (int j = 0; j < NC; j += 2)
                        mh[j / 2] = pack_f16(fmaf(-eb, f16_lo(uh[j / 2]), -dd[i][j]),
                                             fmaf(-eb, f16_hi(uh[j / 2]), -dd[i][j + 1]));
                    if (NC == 4)
                        *(uint2*)&dmu[off] = make_uint2(mh[0], mh[1]);
                    else
                        *(uint4*)&dmu[off] = make_uint4(mh[0], mh[1], mh[2], mh[3]);
#pragma unroll
                    for (int j = 0; j < NC; j += 4)
                        *(float4*)&dq_acc[off + j] = make_float4(dd[i][j], dd[i][j + 1], dd[i][j + 2], dd[i][j + 3]);
                }
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                gr += __shfl_xor_sync(0xffffffffu, gr, o);
                if (MODE) {
                    gb += __shfl_xor_sync(0xffffffffu, gb, o);
                    ru += __shfl_xor_sync(0xffffffffu, ru, o);
                    xx += __shfl_xor_sync(0xffffffffu, xx, o);
                }
            }
            if (valid && tx == 0) {
                if (MODE == 0) {
                    gbar[row] = gr;
                } else {
                    const float eb = ebar[row];
                    const float doo = eb + ru - gb * eb;
                    // paired layout: pair t / 2 of head bh holds
                    // {-L_even, -L_odd, g1_even, g1_odd, -ebar_even, -ebar_odd, -D_even, -D_odd}
                    const int tt = r % T, half = tt & 1;
                    float* pr = rowpack + (((size_t)(r / T) * H + h) * ((T + 1) / 2) + tt / 2) * 8 + half;
                    pr[0] = -lse[row] * LOG2E;
                    pr[2] = 1.f - gr;
                    pr[4] = -eb;
                    pr[6] = -(doo - gb * eb + xx);
                }
            }
        }
        if (MODE) {
            // dP_h partial: dp[a][b] += sum over the block's rows du[r][a] delta[r][b],
            // a = ty + 16 ii, b = tx + 16 jj (strided ownership: a half-warp reads 16
            // consecutive transposed rows, which the row stride spreads over all banks)
#pragma unroll 2
            for (int r = 0; r < RB; r += 4) {
                float4 ya[NA], xb[NA];
#pragma unroll
                for (int ii = 0; ii < NA; ii++) ya[ii] = *(const float4*)&YT[(ty + 16 * ii) * LDT + r];
#pragma unroll
                for (int jj = 0; jj < NA; jj++) xb[jj] = *(const float4*)&XT[(tx + 16 * jj) * LDT + r];
#pragma unroll
                for (int ii = 0; ii < NA; ii++)
#pragma unroll
                    for (int jj = 0; jj < NA; jj++)
                        dp[ii][jj] = fmaf(ya[ii].x, xb[jj].x,
                                          fmaf(ya[ii].y, xb[jj].y,
                                               fmaf(ya[ii].z, xb[jj].z, fmaf(ya[ii].w, xb[jj].w, dp[ii][jj]))));
            }
        }
    }
    if (MODE) {
        float* dst = dp_partial + ((size_t)h * gridDim.x + blockIdx.x) * D * D;
#pragma unroll
        for (int ii = 0; ii < NA; ii++)
#pragma unroll
            for (int jj = 0; jj < NA; jj++) dst[(ty + 16 * ii) * D + tx + 16 * jj] = dp[ii][jj];
    }
}

// ============================================================ B2 on the tensor cores (d = 64)
// The row math of B2 (same outputs as tc_rows<64, 1>) with its three
// products on the tensor cores, per tile of 128 rows of head h:
//   U = delta P_h^T and ddelta = du P_h, with delta and du split into f16
//   hi + lo halves against P_h in f16 (the forward's projection: delta is
//   formed from the same f16 copy of q, so U equals the forward's);
//   dP_h partial += du^T delta over a chunk of 512 rows as one M = 128
//   product whose A stacks [du | delta] along M (rows 0..63 of the result
//   are du^T delta), in three passes hi.hi + lo.hi + hi.lo.
// Two persistent CTAs per SM each walk a contiguous range of the (head,
// chunk) list tile by tile and write each chunk's partial when the chunk
// ends.  Global memory is read and written in row-contiguous order: thread
// item (row, quad) covers columns [4 quad, 4 quad + 4) of one row, sixteen
// consecutive threads one whole row.  The products leave U and ddelta in
// TMEM, one row per lane; they go through shared memory (fp32, in the space
// of the finished MMA operand tiles) back to the (row, quad) layout, where
// the row dot products are summed across the row's sixteen threads.
struct B2T {
    static constexpr int D = 64, BM = 128, NT = 256, TILES = 4;  // 512 rows per chunk
    static constexpr int TB = BM * D * 2;                         // one f16 [128][64] tile
    static constexpr int PB = D * D * 2;                          // P_h in f16
    static constexpr int LDF = D + 4;                             // row stride of the fp32 U / ddelta tiles
    static constexpr int XB = BM * LDF * 4;
    static constexpr int OPS = (4 * TB > 2 * XB ? 4 * TB : 2 * XB + 1023) / 1024 * 1024;
    static constexpr int ITEMS = BM * (D / 4) / NT;               // (row, quad) items per thread per tile
    // tiles in this order: [du_hi | delta_hi] and [du_lo | delta_lo] sit TB
    // apart, as the two 64-row M blocks of the dP product's A operand
    static constexpr int SMEM = 1024 + OPS + PB + 2 * BM * 4 + 64;
    static constexpr unsigned TMEM_COLS = 256;  // U [0,64), ddelta [64,128), dP [128,192)
};
static_assert(B2T::BM * B2T::TILES == RowCfg<64>::ROWS_PER_CTA, "dP partial layout shared with tc_rows");
static_assert(B2T::ITEMS == 8, "the item loops are written for 8 items per thread");

// One tile of B2's walk: item = h * nchunks + chunk, rows [r0, r_end) of the
// chunk's rows [chunk * 512, min(chunk * 512 + 512, B T)).
struct B2Tile {
    int item, r0, r_end;
};

__global__ void __launch_bounds__(B2T::NT, 2) tc_b2(const __half* __restrict__ q16, const float* __restrict__ mu_k,
                                                 const float* __restrict__ P, const float* __restrict__ lse,
                                                 const float* __restrict__ R, const float* __restrict__ ebar,
                                                 __half* __restrict__ U, __half* __restrict__ dmu,
                                                 float* __restrict__ dq_acc, float* __restrict__ rowpack,
                                                 float* __restrict__ dp_partial, int B, int H, int T, int nchunks,
                                                 unsigned* status) {
    using C = B2T;
    constexpr int D = C::D, LDF = C::LDF, RPC = C::BM * C::TILES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sUH = sm;
    uint8_t* sDH = sUH + C::TB;
    uint8_t* sUL = sDH + C::TB;
    uint8_t* sDL = sUL + C::TB;
    float* sXU = (float*)sm;                   // after the products: U (fp32) [128][LDF]
    float* sXD = (float*)(sm + C::XB);         // and ddelta
    uint8_t* sP = sm + C::OPS;
    float* sEb = (float*)(sP + C::PB);         // the tile's ebar
    float* sL = sEb + C::BM;                   // and lse
    uint64_t* bars = (uint64_t*)(sL + C::BM);  // [0] the tile's MMAs are done, [1] teardown drain
    uint32_t* holder = (uint32_t*)(bars + 2);
    volatile int* abortf = (volatile int*)(holder + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
    const int rit = quad * 32 + lane;             // row in the tile = TMEM lane
    const int nrows = B * T;
    const int nitems = H * nchunks;
    const int it_begin = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int it_end = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);
    const Watchdog wd{status, abortf, KID_TC_BWD_B2, wait_limit(status)};
    if (tid == 0) {
        *abortf = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder, tU = tmem, tDD = tmem + 64, tDP = tmem + 128;
    const uint32_t lrow = (uint32_t)(quad * 32) << 16;
    const int c0 = 32 * half;  // this thread's TMEM columns [c0, c0 + 32)
    const int qd = tid & 15;   // item column quad: columns [4 qd, 4 qd + 4)
    const uint32_t idN = idesc_mma(128, D, false, false);  // U: A and B K-major
    const uint32_t idNb = idesc_mma(128, D, false, true);  // ddelta: B = P_h read MN-major
    const uint32_t idPd = idesc_mma(128, D, true, true);   // dP: A = [du | delta], B = delta, both MN-major

    auto first_tile = [&](int item) -> B2Tile {
        const int chunk = item % nchunks;
        return B2Tile{item, chunk * RPC, min(chunk * RPC + RPC, nrows)};
    };
    auto next_tile = [&](const B2Tile& c) -> B2Tile {
        if (c.r0 + C::BM < c.r_end) return B2Tile{c.item, c.r0 + C::BM, c.r_end};
        return c.item + 1 < it_end ? first_tile(c.item + 1) : B2Tile{-1, 0, 0};
    };
    // item k of this thread: row (k * NT + tid) / 16 of the tile, quad qd
    auto item_row = [&](const B2Tile& c, int k, int& rl, size_t& row) -> bool {
        rl = (k * C::NT + tid) >> 4;
        const int r = c.r0 + rl;
        const bool valid = r < c.r_end;
        const int h = c.item / nchunks;
        row = valid ? ((size_t)(r / T) * H + h) * T + r % T : 0;
        return valid;
    };

    bool ok = true;
    int head = -1, ntile = 0;
    B2Tile cur = it_begin < it_end ? first_tile(it_begin) : B2Tile{-1, 0, 0};
    while (cur.item >= 0) {
        const int h = cur.item / nchunks;
        const bool chunk_first = cur.r0 % RPC == 0;
        const bool chunk_last = cur.r0 + C::BM >= cur.r_end;
        if (h != head) {
            // P_h in f16 as a K-major [a][b] tile: the B operand of U (N = a,
            // K = b) and, read MN-major, of ddelta (N = b, K = a); the previous
            // tile's products have completed
            const float* Ph = P + (size_t)h * D * D;
            for (int id = tid; id < D * D / 8; id += C::NT) {
                const int pa = id / (D / 8), pb0 = (id % (D / 8)) * 8;
                const float4 x0 = *(const float4*)(Ph + pa * D + pb0);
                const float4 x1 = *(const float4*)(Ph + pa * D + pb0 + 4);
                *(uint4*)(sP + sw_off(pa, pb0, D)) = make_uint4(pack_f16(x0.x, x0.y), pack_f16(x0.z, x0.w),
                                                                pack_f16(x1.x, x1.y), pack_f16(x1.z, x1.w));
            }
            head = h;
        }
        // delta = q - mu_k and du = R - ebar mu_k as f16 hi + lo, K-major
        // rows; ebar and lse of each row kept for the epilogue
#pragma unroll 1
        for (int kb = 0; kb < C::ITEMS; kb += 4) {
        uint2 pq[4];
        float4 pm[4], pr[4];
        float pe[4], pl[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            int rl;
            size_t row;
            pq[e] = make_uint2(0, 0);
            pm[e] = pr[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            pe[e] = pl[e] = 0.f;
            if (item_row(cur, kb + e, rl, row)) {
                pq[e] = *(const uint2*)(q16 + row * D + 4 * qd);
                pm[e] = *(const float4*)(mu_k + row * D + 4 * qd);
                pr[e] = *(const float4*)(R + row * D + 4 * qd);
                pe[e] = ebar[row];
                if (qd == 0) pl[e] = lse[row];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {
            int rl;
            size_t row;
            const bool valid = item_row(cur, kb + e, rl, row);
            const float m[4] = {pm[e].x, pm[e].y, pm[e].z, pm[e].w};
            const float x[4] = {pr[e].x, pr[e].y, pr[e].z, pr[e].w};
            const uint32_t qw[2] = {pq[e].x, pq[e].y};
            uint32_t dh[2], dl[2], uh[2], ul[2];
#pragma unroll
            for (int w = 0; w < 2; w++) {
                const float d0 = f16_lo(qw[w]) - m[2 * w];
                const float d1 = f16_hi(qw[w]) - m[2 * w + 1];
                dh[w] = pack_f16(d0, d1);
                dl[w] = pack_f16(d0 - f16_lo(dh[w]), d1 - f16_hi(dh[w]));
                const float u0 = x[2 * w] - pe[e] * m[2 * w];
                const float u1 = x[2 * w + 1] - pe[e] * m[2 * w + 1];
                uh[w] = pack_f16(u0, u1);
                ul[w] = pack_f16(u0 - f16_lo(uh[w]), u1 - f16_hi(uh[w]));
            }
            if (!valid) dh[0] = dh[1] = dl[0] = dl[1] = uh[0] = uh[1] = ul[0] = ul[1] = 0u;
            if (qd == 0) {
                sEb[rl] = pe[e];
                sL[rl] = pl[e];
            }
            const uint32_t off = sw_off(rl, (4 * qd) & ~7, C::BM) + ((qd & 1) << 3);
            *(uint2*)(sDH + off) = make_uint2(dh[0], dh[1]);
            *(uint2*)(sDL + off) = make_uint2(dl[0], dl[1]);
            *(uint2*)(sUH + off) = make_uint2(uh[0], uh[1]);
            *(uint2*)(sUL + off) = make_uint2(ul[0], ul[1]);
        }
        }
        fence_proxy_async_smem();
        tc_fence_before();  // the previous tile's TMEM reads come before these MMAs
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            if (elect_one()) {
                const uint32_t dh = smem_u32(sDH), dl = smem_u32(sDL), uh = smem_u32(sUH), ul = smem_u32(sUL);
                const uint32_t pb = smem_u32(sP);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tU, desc_kmajor(dh, C::BM, kk), desc_kmajor(pb, D, kk), idN, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tU, desc_kmajor(dl, C::BM, kk), desc_kmajor(pb, D, kk), idN, 1u);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tDD, desc_kmajor(uh, C::BM, kk), desc_mnmajor(pb, D, kk), idNb, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++)
                    mma_ss(tDD, desc_kmajor(ul, C::BM, kk), desc_mnmajor(pb, D, kk), idNb, 1u);
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; kk++)
                    mma_ss(tDP, desc_mn_lbo(uh, kk, C::TB), desc_mnmajor(dh, C::BM, kk), idPd,
                           (!chunk_first || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; kk++)
                    mma_ss(tDP, desc_mn_lbo(ul, kk, C::TB), desc_mnmajor(dh, C::BM, kk), idPd, 1u);
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; kk++)
                    mma_ss(tDP, desc_mn_lbo(uh, kk, C::TB), desc_mnmajor(dl, C::BM, kk), idPd, 1u);
                mma_commit(&bars[0]);
            }
            __syncwarp();
        }
        ok = __syncthreads_and(mbar_wait(&bars[0], ntile & 1, wd, 1)) != 0;
        if (!ok) break;
        tc_fence_after();
        // U and ddelta, one row per TMEM lane, to shared memory (the operand
        // tiles were read by the completed products)
        {
            uint32_t vu[32], vd[32];
            tmem_ld32(tU + lrow + c0, vu);
            tmem_ld32(tDD + lrow + c0, vd);
            tmem_wait_ld();
            float* xu = sXU + rit * LDF + c0;
            float* xd = sXD + rit * LDF + c0;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                *(uint4*)(xu + i) = make_uint4(vu[i], vu[i + 1], vu[i + 2], vu[i + 3]);
                *(uint4*)(xd + i) = make_uint4(vd[i], vd[i + 1], vd[i + 2], vd[i + 3]);
            }
        }
        // the chunk's dP_h partial: rows a = TMEM lanes 0..63 (quadrants 0
        // and 1), columns split between the two halves
        if (chunk_last && quad < 2) {
            const int chunk = cur.item % nchunks;
            float* dst = dp_partial + ((size_t)h * nchunks + chunk) * D * D + (size_t)rit * D + c0;
            uint32_t v[32];
            tmem_ld32(tDP + lrow + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *(float4*)(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                  __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
        __syncthreads();
        // per item: U (f16), z = dmu - ebar U (f16, dmu = -ddelta), dq_acc =
        // ddelta, and the row sums gr = mu_k . f16(U), gb = mu_k . U, ru = R . U,
        // xx = mu_k . dmu
#pragma unroll 2
        for (int kb = 0; kb < C::ITEMS; kb += 4) {
            float4 mv[4], rv[4];
            bool valid[4];
            int rl[4];
            size_t row[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                valid[e] = item_row(cur, kb + e, rl[e], row[e]);
                mv[e] = rv[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (valid[e]) {
                    mv[e] = *(const float4*)(mu_k + row[e] * D + 4 * qd);
                    rv[e] = *(const float4*)(R + row[e] * D + 4 * qd);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float4 u4 = *(const float4*)(sXU + rl[e] * LDF + 4 * qd);
                const float4 d4 = *(const float4*)(sXD + rl[e] * LDF + 4 * qd);
                const uint32_t uh0 = pack_f16(u4.x, u4.y), uh1 = pack_f16(u4.z, u4.w);
                float gr = mv[e].x * f16_lo(uh0);
                gr = fmaf(mv[e].y, f16_hi(uh0), gr);
                gr = fmaf(mv[e].z, f16_lo(uh1), gr);
                gr = fmaf(mv[e].w, f16_hi(uh1), gr);
                float gb = mv[e].x * u4.x;
                gb = fmaf(mv[e].y, u4.y, gb);
                gb = fmaf(mv[e].z, u4.z, gb);
                gb = fmaf(mv[e].w, u4.w, gb);
                float ru = rv[e].x * u4.x;
                ru = fmaf(rv[e].y, u4.y, ru);
                ru = fmaf(rv[e].z, u4.z, ru);
                ru = fmaf(rv[e].w, u4.w, ru);
                float xx = mv[e].x * -d4.x;
                xx = fmaf(mv[e].y, -d4.y, xx);
                xx = fmaf(mv[e].z, -d4.z, xx);
                xx = fmaf(mv[e].w, -d4.w, xx);
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) {  // the row's sixteen threads (lanes 16-aligned)
                    gr += __shfl_xor_sync(0xffffffffu, gr, o);
                    gb += __shfl_xor_sync(0xffffffffu, gb, o);
                    ru += __shfl_xor_sync(0xffffffffu, ru, o);
                    xx += __shfl_xor_sync(0xffffffffu, xx, o);
                }
                if (valid[e]) {
                    const size_t base = row[e] * D + 4 * qd;
                    *(float4*)(dq_acc + base) = d4;
                    *(uint2*)(U + base) = make_uint2(uh0, uh1);
                    const float eb = sEb[rl[e]];
                    *(uint2*)(dmu + base) =
                        make_uint2(pack_f16(fmaf(-eb, f16_lo(uh0), -d4.x), fmaf(-eb, f16_hi(uh0), -d4.y)),
                                   pack_f16(fmaf(-eb, f16_lo(uh1), -d4.z), fmaf(-eb, f16_hi(uh1), -d4.w)));
                    if (qd == 0) {
                        // paired row scalars {-L_e, -L_o, g1_e, g1_o, -ebar_e, -ebar_o, -D_e, -D_o}
                        const float doo = eb + ru - gb * eb;
                        const int r = cur.r0 + rl[e], tt = r % T, hp = tt & 1;
                        float* prow = rowpack + (((size_t)(r / T) * H + h) * ((T + 1) / 2) + tt / 2) * 8 + hp;
                        prow[0] = -sL[rl[e]] * LOG2E;
                        prow[2] = 1.f - gr;
                        prow[4] = -eb;
                        prow[6] = -(doo - gb * eb + xx);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // the fp32 tiles are read before the next tile's operands overwrite them
        cur = next_tile(cur);
        ntile++;
    }
    // teardown: every MMA issued must complete before the CTA releases TMEM
    if (warp == 0) {
        if (elect_one()) mma_commit(&bars[1]);
        __syncwarp();
        mbar_wait_drain(&bars[1], 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// dP[h] = sum of the CTA partials in chunk order (fixed order: reproducible).
__global__ void __launch_bounds__(256) tc_dp_reduce(const float4* __restrict__ partial, float4* __restrict__ dP,
                                                    int nchunks, int dd4) {
    const int h = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= dd4) return;
    const float4* src = partial + (size_t)h * nchunks * dd4 + e;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < nchunks; c++) {
        const float4 v = src[(size_t)c * dd4];
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
    }
    dP[(size_t)h * dd4 + e] = s;
}

// ============================================================ backward B3
// CTA = one tile of 128 keys of one head; queries stream in sub-chunks of 64.
// Per sub-chunk (TMEM lanes = keys i, columns = queries t):
//   [S^T | G^T | Y^T] = K [Q | U | z]^T     (one N = 192 MMA: K is read once)
//   E^T = V dO^T
//   p = exp(c s - lse_t), w1 = 1 + g - gbar_t, a = p w1, pe = p e,
//   ds = c p (e w1 + y - D_t)      (y = k . z = k . dmu - g ebar_t)
//   dV += a dO, dK += pe U + ds Q + p z        (A operands f16 in TMEM)
// The dK sum is p (e - ebar_t) U + ds Q + p dmu written with z = dmu - ebar_t U,
// which B2 stores in place of dmu: the ebar_t terms leave the per-element step.
// and per 128 queries dQ += ds^T K (A = ds from shared memory), added into the
// fp32 dq accumulator with vector reductions.  Two warpgroups split the
// elementwise work by query columns.
template <int D>
struct B3Cfg {
    static constexpr int BK = 128, BQ = 64, QT = 128;
    static constexpr int NT = 320;              // TMA warp, MMA warp, 2 x 4 elementwise warps
    static constexpr int NS = D == 64 ? 2 : 1;  // sub-chunk stages
    static constexpr int KB = BK * D * 2;       // K or V tile
    static constexpr int QUM_B = 3 * BQ * 128;  // one 64-column block of the stacked [Q|U|dmu] rows
    static constexpr int DO_OFF = (D / 64) * QUM_B;
    static constexpr int ROWS_OFF = DO_OFF + BQ * D * 2;
    static constexpr int STAGE = ROWS_OFF + BQ * 16;
    static constexpr int DSB = BK * QT * 2;     // ds, f16 [keys][128 queries]
    static constexpr int NBAR = 1 + 2 * NS + 6;
    static constexpr int SMEM = 1024 + 2 * KB + DSB + NS * STAGE + NBAR * 8 + 16;
    static constexpr unsigned TMEM_COLS = 512;
    // TMEM columns: S^T [0,64), G^T [64,128), Y^T [128,192), E^T [192,256),
    // dV [256, 256+D), dK [256+D, 256+2D); dQ reuses [128, 128+D).
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}


// The elementwise step for 16 queries (one 16-column chunk) of one key row,
// two queries per f32x2 instruction.  rp points at the chunk's first query
// pair: {-L_e, -L_o, g1_e, g1_o, -ebar_e, -ebar_o, -D_e, -D_o} per pair, with
// L = lse log2 e and g1 = 1 - gbar (-ebar is not needed here: see z above).
template <bool MASK>
__device__ __forceinline__ void b3_chunk(const uint32_t (&vs)[16], const uint32_t (&vg)[16], const uint32_t (&vy)[16],
                                         const uint32_t (&ve)[16], const float* rp, int qlo, float scale,
                                         float scale_log2, uint32_t (&o1)[16], uint32_t (&o2)[16]) {
    const uint64_t SL2 = f2(scale_log2, scale_log2), SC = f2(scale, scale);
#pragma unroll
    for (int q2 = 0; q2 < 8; q2++) {
        const float4 ra = *(const float4*)(rp + 8 * q2);
        const float4 rb = *(const float4*)(rp + 8 * q2 + 4);
        const uint64_t nL = f2(ra.x, ra.y), g1 = f2(ra.z, ra.w), nD = f2(rb.z, rb.w);
        const uint64_t sv = f2(__uint_as_float(vs[2 * q2]), __uint_as_float(vs[2 * q2 + 1]));
        const uint64_t g = f2(__uint_as_float(vg[2 * q2]), __uint_as_float(vg[2 * q2 + 1]));
        const uint64_t y = f2(__uint_as_float(vy[2 * q2]), __uint_as_float(vy[2 * q2 + 1]));
        const uint64_t e = f2(__uint_as_float(ve[2 * q2]), __uint_as_float(ve[2 * q2 + 1]));
        const float2 x = uf2(ffma2(sv, SL2, nL));  // c s - L (log2 units)
        float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
        if (MASK) {
            if (2 * q2 < qlo) p0 = 0.f;
            if (2 * q2 + 1 < qlo) p1 = 0.f;
        }
        const uint64_t p = f2(p0, p1);
        const uint64_t w1 = fadd2(g, g1);                    // 1 + g - gbar
        const float2 a = uf2(fmul2(p, w1));                  // p w1
        const float2 pe = uf2(fmul2(p, e));                  // p e
        uint64_t tt = fadd2(y, nD);                          // k.z - D
        tt = ffma2(e, w1, tt);                               // + e w1
        const float2 ds = uf2(fmul2(fmul2(p, SC), tt));      // c p (...)
        o1[q2] = pack_f16(a.x, a.y);
        o1[8 + q2] = pack_f16(pe.x, pe.y);
        o2[q2] = pack_f16(ds.x, ds.y);
        o2[8 + q2] = pack_f16(p0, p1);
    }
}

template <int D>
__global__ void __launch_bounds__(B3Cfg<D>::NT, 1)
    tc_bwd_b3(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_u,
              const __grid_constant__ CUtensorMap tm_dmu, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_rows, float* __restrict__ dq_acc,
              __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int T, int BH, int nkt, float scale,
              float scale_log2, unsigned* status) {
    using C = B3Cfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sK = sm;
    uint8_t* sV = sK + C::KB;
    uint8_t* sDS = sV + C::KB;
    uint8_t* sSt = sDS + C::DSB;  // stage s: [Q|U|dmu] blocks, dO, row scalars
    uint64_t* bars = (uint64_t*)(sSt + NS * C::STAGE);
    uint64_t* kv_full = bars;
    uint64_t* st_full = bars + 1;
    uint64_t* st_empty = bars + 1 + NS;
    uint64_t* sc_full = bars + 1 + 2 * NS;
    uint64_t* op_full = sc_full + 1;
    uint64_t* acc_done = sc_full + 2;
    uint64_t* dq_full = sc_full + 3;
    uint64_t* dq_free = sc_full + 4;
    uint64_t* drain = sc_full + 5;
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int kt, bh;
    work_item(blockIdx.x, BH, nkt, &kt, &bh);  // key tiles with the most queries first
    const int k0 = kt * C::BK;
    // sub-chunk j covers queries [k0 + 64 j, k0 + 64 j + 64); pairs j = 2m, 2m + 1
    // form the m-th 128-query tile of the dQ product
    const int nsub = (T - k0 + C::BQ - 1) / C::BQ;
    const Watchdog wd{status, abortf, KID_TC_BWD_B3, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(kv_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&st_full[s], 1);
            mbar_init(&st_empty[s], 1);
        }
        mbar_init(sc_full, 1);
        mbar_init(op_full, 256);
        mbar_init(acc_done, 1);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 256);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    // ds buffer starts at zero: a query tile cut by T leaves its upper half
    // unwritten, and the dQ MMA must not read uninitialised bits.
    for (int i = threadIdx.x; i < C::DSB / 16; i += C::NT) ((uint4*)sDS)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t tS = tmem, tG = tmem + 64, tY = tmem + 128, tE = tmem + 192;
    const uint32_t tDV = tmem + 256, tDK = tmem + 256 + D, tDQ = tmem + 128;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(kv_full, 2 * C::KB);
#pragma unroll
            for (int r = 0; r < D / 64; r++) {
                tma_load_3d(sK + r * C::BK * 128, &tm_k, r * 64, k0, bh, kv_full);
                tma_load_3d(sV + r * C::BK * 128, &tm_v, r * 64, k0, bh, kv_full);
            }
            int issued = 0;
            for (int j = 0; j < nsub; j++) {
                const int s = j % NS;
                const int t0 = k0 + j * C::BQ;
                if (j >= NS && !mbar_wait(&st_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&st_full[s], C::STAGE);
                uint8_t* st = sSt + s * C::STAGE;
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    uint8_t* blk = st + r * C::QUM_B;
                    tma_load_3d(blk, &tm_q, r * 64, t0, bh, &st_full[s]);
                    tma_load_3d(blk + C::BQ * 128, &tm_u, r * 64, t0, bh, &st_full[s]);
                    tma_load_3d(blk + 2 * C::BQ * 128, &tm_dmu, r * 64, t0, bh, &st_full[s]);
                    tma_load_3d(st + C::DO_OFF + r * C::BQ * 128, &tm_do, r * 64, t0, bh, &st_full[s]);
                }
                tma_load_3d(st + C::ROWS_OFF, &tm_rows, 0, t0 / 2, bh, &st_full[s]);
                issued = j + 1;
            }
            mbar_wait_drain(kv_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&st_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1) {
        // The whole warp runs the issue loop, so the descriptors stay
        // warp-uniform; the elected lane (lane 0 of the converged warp) issues
        // every tcgen05 instruction, so one thread issues all MMAs, in order.
        const uint32_t idS3 = idesc_mma(128, 3 * C::BQ, false, false);  // [S|G|Y]^T: N = 192 queries x3
        const uint32_t idS = idesc_mma(128, C::BQ, false, false);       // E^T
        const uint32_t idA = idesc_mma(128, D, false, true);            // dV, dK: A in TMEM, B MN-major
        const uint32_t idQ = idesc_mma(128, D, true, true);             // dQ: A = ds MN-major, B = K MN-major
        const uint32_t kaddr = smem_u32(sK), vaddr = smem_u32(sV), dsaddr = smem_u32(sDS);
        if (__all_sync(0xffffffffu, mbar_wait(kv_full, 0, wd, 2))) {
            for (int j = 0; j < nsub; j++) {
                const int s = j % NS;
                if (!__all_sync(0xffffffffu, mbar_wait(&st_full[s], (j / NS) & 1, wd, 3))) break;
                // the scores overwrite the previous sub-chunk's weight operands;
                // tcgen05.mma ops issued by one thread execute in issue order
                if (j > 0 && (j & 1) == 0 && !__all_sync(0xffffffffu, mbar_wait(dq_free, ((j >> 1) - 1) & 1, wd, 5))) break;
                tc_fence_after();
                const uint32_t st = smem_u32(sSt + s * C::STAGE);
                const uint32_t ado = st + C::DO_OFF;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) {
                        mma_ss(tS, desc_kmajor(kaddr, C::BK, kk), desc_kmajor(st, 3 * C::BQ, kk), idS3, kk > 0);
                        mma_ss(tE, desc_kmajor(vaddr, C::BK, kk), desc_kmajor(ado, C::BQ, kk), idS, kk > 0);
                    }
                    mma_commit(sc_full);
                }
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(op_full, j & 1, wd, 6))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < C::BQ / 16; kk++) {
                        const uint32_t first = (j == 0 && kk == 0) ? 0u : 1u;
                        mma_ts(tDV, tS + 16 * kk, desc_mn_lbo(ado, kk, C::BQ * 128), idA, first);
                        mma_ts(tDK, tS + 16 * kk + 8, desc_mn_lbo(st + C::BQ * 128, kk, C::QUM_B), idA, first);
                        mma_ts(tDK, tG + 16 * kk, desc_mn_lbo(st, kk, C::QUM_B), idA, 1u);
                        mma_ts(tDK, tG + 16 * kk + 8, desc_mn_lbo(st + 2 * C::BQ * 128, kk, C::QUM_B), idA, 1u);
                    }
                    if (j == nsub - 1) mma_commit(acc_done);  // one phase: the epilogue's only wait
                    mma_commit(&st_empty[s]);
                    if ((j & 1) == 1 || j == nsub - 1) {
#pragma unroll
                        for (int kk = 0; kk < C::BK / 16; kk++)
                            mma_ss(tDQ, desc_mnmajor(dsaddr, C::BK, kk), desc_mnmajor(kaddr, C::BK, kk), idQ, kk > 0);
                        mma_commit(dq_full);
                    }
                }
                __syncwarp();
            }
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int wg = (warp - 2) >> 2;  // warpgroup: query columns [32 wg, 32 wg + 32)
        const int qd = warp & 3;
        const int i = qd * 32 + lane;  // key row (and, for dQ, query row) of this thread
        const int key = k0 + i;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        bool ok = true;
        for (int j = 0; j < nsub && ok; j++) {
            const int s = j % NS;
            const int t0 = k0 + j * C::BQ;
            ok = mbar_wait(sc_full, j & 1, wd, 7);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* rows = (const float*)(sSt + s * C::STAGE + C::ROWS_OFF);  // 8 floats per query pair
            uint8_t* dsrow = sDS + (j & 1) * (C::BK * 128) + i * 128;
            const bool need_mask = t0 < k0 + C::BK || t0 + C::BQ > T;
#pragma unroll 1
            for (int c = 2 * wg; c < 2 * wg + 2; c++) {
                uint32_t vs[16], vg[16], vy[16], ve[16];
                tmem_ld16(tS + lrow + 16 * c, vs);
                tmem_ld16(tG + lrow + 16 * c, vg);
                tmem_ld16(tY + lrow + 16 * c, vy);
                tmem_ld16(tE + lrow + 16 * c, ve);
                tmem_wait_ld();
                uint32_t o1[16], o2[16];  // o1: a | pe, o2: ds | p (f16 pairs)
                if (need_mask) {
                    // query t = t0 + 16 c + qq is valid iff key <= t and t < T
                    const int qlo = max(key - (t0 + 16 * c), 0);
                    const int qhi = T - (t0 + 16 * c);
                    b3_chunk<true>(vs, vg, vy, ve, rows + 64 * c, qhi <= 0 ? 16 : qlo, scale, scale_log2, o1, o2);
                    if (qhi < 16) {
#pragma unroll
                        for (int x = 0; x < 8; x++) {
                            const uint32_t keep = (2 * x + 1 < qhi) ? 0xFFFFFFFFu : (2 * x < qhi ? 0xFFFFu : 0u);
                            o1[x] &= keep;
                            o1[8 + x] &= keep;
                            o2[x] &= keep;
                            o2[8 + x] &= keep;
                        }
                    }
                } else {
                    b3_chunk<false>(vs, vg, vy, ve, rows + 64 * c, 0, scale, scale_log2, o1, o2);
                }
                tmem_st16(tS + lrow + 16 * c, o1);
                tmem_st16(tG + lrow + 16 * c, o2);
                // ds row segment (16 queries = 32 bytes) into the swizzled
                // [keys][queries] buffer: 16-byte chunks 2c and 2c + 1.
                *(uint4*)(dsrow + (((2 * c) ^ (i & 7)) << 4)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                *(uint4*)(dsrow + (((2 * c + 1) ^ (i & 7)) << 4)) = make_uint4(o2[4], o2[5], o2[6], o2[7]);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(op_full);
            if ((j & 1) == 1 || j == nsub - 1) {
                // dQ of the 128-query tile m = j / 2: thread = query row i,
                // warpgroup wg adds columns [wg D/2, wg D/2 + D/2)
                ok = mbar_wait(dq_full, (j >> 1) & 1, wd, 8);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int t = k0 + (j >> 1) * C::QT + i;
#pragma unroll 1
                for (int c = 0; c < D / 64; c++) {
                    const int col = wg * (D / 2) + 32 * c;
                    uint32_t v[32];
                    tmem_ld32(tDQ + lrow + col, v);
                    tmem_wait_ld();
                    if (t < T) {
                        float* dst = dq_acc + ((size_t)bh * T + t) * D + col;
#pragma unroll
                        for (int x = 0; x < 32; x += 4)
                            red_add_v4(dst + x, __uint_as_float(v[x]), __uint_as_float(v[x + 1]),
                                       __uint_as_float(v[x + 2]), __uint_as_float(v[x + 3]));
                    }
                }
                tc_fence_before();
                mbar_arrive(dq_free);
            }
        }
        if (ok) {
            ok = mbar_wait(acc_done, 0, wd, 9);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                // warpgroup 0 writes dV, warpgroup 1 writes dK
                const uint32_t tsrc = wg == 0 ? tDV : tDK;
                __nv_bfloat16* dst_base = wg == 0 ? dv : dk;
#pragma unroll 1
                for (int c = 0; c < D / 32; c++) {
                    uint32_t v[32];
                    tmem_ld32(tsrc + lrow + 32 * c, v);
                    tmem_wait_ld();
                    if (key < T) {
                        uint4* pv = (uint4*)(dst_base + ((size_t)bh * T + key) * D + 32 * c);
#pragma unroll
                        for (int x = 0; x < 4; x++)
                            pv[x] = make_uint4(pack_bf16(__uint_as_float(v[8 * x]), __uint_as_float(v[8 * x + 1])),
                                               pack_bf16(__uint_as_float(v[8 * x + 2]), __uint_as_float(v[8 * x + 3])),
                                               pack_bf16(__uint_as_float(v[8 * x + 4]), __uint_as_float(v[8 * x + 5])),
                                               pack_bf16(__uint_as_float(v[8 * x + 6]), __uint_as_float(v[8 * x + 7])));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------ B3, d = 64: 64-query sub-chunks
// The same mathematics as tc_bwd_b3 with 64-query sub-chunks: the score
// product [S|G|Y]^T = K [Q|U|dmu]^T is one N = 192 MMA per 16 of d, and E^T one
// N = 64 MMA.  One TMEM score region serves every sub-chunk.  The two
// elementwise warpgroups (queries [0,32) and [32,64) of each sub-chunk) load
// their scores into registers and arrive on sx_free; the MMA thread then
// issues the next sub-chunk's scores while they form the weights.  The weights
// have storage of their own: a | pe in TMEM, ds and p in shared memory (ds in
// the 128-query tile the dQ product reads as well), so the accumulation of
// sub-chunk j reads them while the scores of j + 1 occupy the score region.
// dQ of each 128-query tile is read after the elementwise step of the next
// tile's first sub-chunk, by when its product has completed; it is staged in
// the ds tile that product has read (one 32-column box per warpgroup) and
// added into the fp32 accumulator by one tensor reduce-add per box.  The next
// writer of that ds tile, a sub-chunk later, waits until both reduces have
// read their boxes.
// TMEM columns: S^T [0,64) G^T [64,128) Y^T [128,192) E^T [192,256),
// a|dg [256,320), dV [320,384), dK [384,448), dQ [448,512).
struct B3Q {
    static constexpr int D = 64, BK = 128, BQ = 64, QT = 128, NT = 320;
    static constexpr int NS = 3;                            // operand stages
    static constexpr int KB = BK * D * 2;                   // K or V tile
    static constexpr int SUB = BQ * 128;                    // one 64-row operand tile
    static constexpr int DO_OFF = 3 * SUB;                  // after the stacked [Q|U|dmu]
    static constexpr int ROWS_OFF = 4 * SUB;
    static constexpr int STAGE = ROWS_OFF + (BQ / 2) * 32;  // + the row scalars of 32 query pairs
    static constexpr int DSB = BK * QT * 2;                 // one ds tile, f16 [keys][128 queries]
    static constexpr int PB = BK * BQ * 2;                  // the p tile, f16 [keys][64 queries]
    static constexpr int NBAR = 1 + 2 * NS + 12;
    static constexpr int SMEM = 1024 + 2 * KB + 2 * DSB + PB + NS * STAGE + NBAR * 8 + 16;
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};

__global__ void __launch_bounds__(B3Q::NT, 1)
    tc_bwd_b3_q64(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_u,
                  const __grid_constant__ CUtensorMap tm_dmu, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_dq,
                  __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int T, int BH, int nkt,
                  float scale, float scale_log2, unsigned* status) {
    using C = B3Q;
    constexpr int NS = C::NS, D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sK = sm;
    uint8_t* sV = sK + C::KB;
    uint8_t* sDS = sV + C::KB;       // two ds tiles (128-query tiles m and m + 1)
    uint8_t* sP = sDS + 2 * C::DSB;  // p of one sub-chunk
    uint8_t* sSt = sP + C::PB;       // stage s: Q, U, dmu, dO (64 rows each), row scalars
    uint64_t* bars = (uint64_t*)(sSt + NS * C::STAGE);
    uint64_t* kv_full = bars;
    uint64_t* st_full = bars + 1;
    uint64_t* st_empty = st_full + NS;
    uint64_t* sc_full = st_empty + NS;  // the sub-chunk's scores are in TMEM
    uint64_t* sx_free = sc_full + 1;    // both warpgroups have loaded them (256 arrivals)
    uint64_t* w_full = sc_full + 2;     // the sub-chunk's weights are written (256 arrivals)
    uint64_t* w_free = sc_full + 3;     // the accumulation has read a|dg and p
    uint64_t* stg_read = sc_full + 4;   // [2], per ds tile: both dQ reduces staged there have read it (2 arrivals)
    uint64_t* stg_ready = sc_full + 6;  // [2], per warpgroup: its dQ box is staged (128 arrivals)
    uint64_t* dq_full = sc_full + 8;
    uint64_t* dq_free = sc_full + 9;    // both warpgroups have read the dQ tile (256 arrivals)
    uint64_t* drain = sc_full + 10;
    uint64_t* fin = sc_full + 11;       // the last accumulation has completed (one phase)
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int kt, bh;
    work_item(blockIdx.x, BH, nkt, &kt, &bh);  // key tiles with the most queries first
    const int k0 = kt * C::BK;
    const int nsub = (T - k0 + C::BQ - 1) / C::BQ;  // sub-chunk j: queries [k0 + 64 j, k0 + 64 j + 64)
    const Watchdog wd{status, abortf, KID_TC_BWD_B3, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(kv_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&st_full[s], 1);
            mbar_init(&st_empty[s], 1);
        }
        mbar_init(sc_full, 1);
        mbar_init(sx_free, 256);
        mbar_init(w_full, 256);
        mbar_init(w_free, 1);
        for (int x = 0; x < 2; x++) {
            mbar_init(&stg_read[x], 2);
            mbar_init(&stg_ready[x], 128);
        }
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 256);
        mbar_init(drain, 1);
        mbar_init(fin, 1);
        fence_barrier_init();
    }
    // ds tiles start at zero: the last tile of a key tile may have one
    // sub-chunk only, and the dQ product reads all 128 query rows (the rows
    // past T are discarded).
    for (int i = threadIdx.x; i < 2 * C::DSB / 16; i += C::NT) ((uint4*)sDS)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc(holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t tSc = tmem, tW = tmem + 256, tDV = tmem + 320, tDK = tmem + 384, tDQ = tmem + 448;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(kv_full, 2 * C::KB);
            tma_load_3d(sK, &tm_k, 0, k0, bh, kv_full);
            tma_load_3d(sV, &tm_v, 0, k0, bh, kv_full);
            int issued = 0;
            for (int j = 0; j < nsub; j++) {
                const int s = j % NS, t0 = k0 + j * C::BQ;
                if (j >= NS && !mbar_wait(&st_empty[s], ((j / NS) - 1) & 1, wd, 1)) break;
                mbar_expect_tx(&st_full[s], C::STAGE);
                uint8_t* st = sSt + s * C::STAGE;
                tma_load_3d(st, &tm_q, 0, t0, bh, &st_full[s]);
                tma_load_3d(st + C::SUB, &tm_u, 0, t0, bh, &st_full[s]);
                tma_load_3d(st + 2 * C::SUB, &tm_dmu, 0, t0, bh, &st_full[s]);
                tma_load_3d(st + C::DO_OFF, &tm_do, 0, t0, bh, &st_full[s]);
                tma_load_3d(st + C::ROWS_OFF, &tm_rows, 0, t0 / 2, bh, &st_full[s]);
                issued = j + 1;
            }
            mbar_wait_drain(kv_full, 0);
            for (int j = issued > NS ? issued - NS : 0; j < issued; j++) mbar_wait_drain(&st_full[j % NS], (j / NS) & 1);
        }
    } else if (warp == 1) {
        // The whole warp runs the loop, so the descriptors stay warp-uniform;
        // the elected lane (lane 0 of the converged warp) issues every tcgen05
        // instruction, so one thread issues all MMAs, in order.
        const uint32_t idS3 = idesc_mma(128, 3 * C::BQ, false, false);  // [S|G|Y]^T
        const uint32_t idS = idesc_mma(128, C::BQ, false, false);       // E^T
        const uint32_t idA = idesc_mma(128, D, false, true);            // dV, dK
        const uint32_t idQ = idesc_mma(128, D, true, true);             // dQ
        const uint32_t kaddr = smem_u32(sK), vaddr = smem_u32(sV), dsaddr = smem_u32(sDS), paddr = smem_u32(sP);
        auto scores = [&](int j) {
            const uint32_t st = smem_u32(sSt + (j % NS) * C::STAGE);
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    mma_ss(tSc, desc_kmajor(kaddr, C::BK, kk), desc_kmajor(st, 3 * C::BQ, kk), idS3, kk > 0);
                    mma_ss(tSc + 192, desc_kmajor(vaddr, C::BK, kk), desc_kmajor(st + C::DO_OFF, C::BQ, kk), idS,
                           kk > 0);
                }
                mma_commit(sc_full);
            }
            __syncwarp();
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(kv_full, 0, wd, 2)) &&
                  __all_sync(0xffffffffu, mbar_wait(&st_full[0], 0, wd, 3));
        if (ok) scores(0);
        for (int j = 0; ok && j < nsub; j++) {
            const int s = j % NS;
            if (j + 1 < nsub) {
                if (!__all_sync(0xffffffffu, mbar_wait(&st_full[(j + 1) % NS], ((j + 1) / NS) & 1, wd, 3))) break;
                // sub-chunk j's scores are in registers: the region takes j + 1's
                if (!__all_sync(0xffffffffu, mbar_wait(sx_free, j & 1, wd, 4))) break;
                scores(j + 1);
            }
            if (!__all_sync(0xffffffffu, mbar_wait(w_full, j & 1, wd, 5))) break;
            tc_fence_after();
            const uint32_t st = smem_u32(sSt + s * C::STAGE);
            const uint32_t dsb = dsaddr + ((j >> 1) & 1) * C::DSB + (j & 1) * (C::BK * 128);  // ds of sub-chunk j
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < C::BQ / 16; kk++) {
                    const uint32_t first = (j == 0 && kk == 0) ? 0u : 1u;
                    mma_ts(tDV, tW + 16 * kk, desc_mnmajor(st + C::DO_OFF, C::BQ, kk), idA, first);
                    mma_ts(tDK, tW + 16 * kk + 8, desc_mnmajor(st + C::SUB, C::BQ, kk), idA, first);
                    mma_ss(tDK, desc_kmajor(dsb, C::BK, kk), desc_mnmajor(st, C::BQ, kk), idA, 1u);
                    mma_ss(tDK, desc_kmajor(paddr, C::BK, kk), desc_mnmajor(st + 2 * C::SUB, C::BQ, kk), idA, 1u);
                }
                mma_commit(w_free);
                mma_commit(&st_empty[s]);
                if (j == nsub - 1) mma_commit(fin);
            }
            __syncwarp();
            if ((j & 1) == 1 || j == nsub - 1) {  // the 128-query tile m is complete: dQ = ds^T K
                const int m = j >> 1, x = m & 1;
                if (m >= 1 && !__all_sync(0xffffffffu, mbar_wait(dq_free, (m - 1) & 1, wd, 6))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; kk++)
                        mma_ss(tDQ, desc_mnmajor(dsaddr + x * C::DSB, C::BK, kk), desc_mnmajor(kaddr, C::BK, kk), idQ,
                               kk > 0);
                    mma_commit(dq_full);
                }
                __syncwarp();
            }
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int wg = (warp - 2) >> 2;  // queries [32 wg, 32 wg + 32) of every sub-chunk
        const int qd = warp & 3;
        const int i = qd * 32 + lane;  // key row (and, for dQ, query row)
        const int key = k0 + i;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        const bool leader = qd == 0 && lane == 0;  // issues this warpgroup's dQ reduces
        // dQ tile m: this warpgroup adds columns [32 wg, 32 wg + 32) of query
        // row i, staged as one 32-column box in block wg of ds tile m & 1
        int ndq = 0;  // dQ tiles this warpgroup has read
        auto read_dq = [&](int m) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(dq_full, m & 1, wd, 9))) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tDQ + lrow + 32 * wg, v);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(dq_free);
            uint8_t* box = sDS + (m & 1) * C::DSB + wg * (C::BK * 128);
#pragma unroll
            for (int y = 0; y < 8; y++)
                *(uint4*)(box + i * 128 + ((y ^ (i & 7)) << 4)) = make_uint4(v[4 * y], v[4 * y + 1], v[4 * y + 2], v[4 * y + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&stg_ready[wg]);
            bool done = true;
            if (leader) {  // every thread's staging writes are visible to the reduce
                done = mbar_wait(&stg_ready[wg], ndq & 1, wd, 12);
                if (done) {
                    tma_reduce_add_3d(&tm_dq, 32 * wg, k0 + m * C::QT, bh, box);
                    bulk_commit();
                }
            }
            ndq++;
            return __shfl_sync(0xffffffffu, done ? 1 : 0, 0) != 0;
        };
        bool ok = true;
        int nread = 0;  // dQ tiles read so far
        for (int j = 0; j < nsub && ok; j++) {
            const int s = j % NS, m = j >> 1, x = m & 1;
            const int t0 = k0 + j * C::BQ;
            ok = mbar_wait(sc_full, j & 1, wd, 7);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* rows = (const float*)(sSt + s * C::STAGE + C::ROWS_OFF);  // 8 floats per query pair
            const bool need_mask = t0 < k0 + C::BK || t0 + C::BQ > T;
            uint8_t* dsrow = sDS + x * C::DSB + (j & 1) * (C::BK * 128) + i * 128;
            uint8_t* prow = sP + i * 128;
            // chunk h's scores, loaded into registers; the second load comes right
            // after the first chunk's arithmetic, so the region can take the next
            // sub-chunk's scores before this one's weights are stored
            uint32_t vs[16], vg[16], vy[16], ve[16];
            auto load = [&](int c) {
                tmem_ld16(tSc + lrow + 16 * c, vs);
                tmem_ld16(tSc + lrow + 64 + 16 * c, vg);
                tmem_ld16(tSc + lrow + 128 + 16 * c, vy);
                tmem_ld16(tSc + lrow + 192 + 16 * c, ve);
                tmem_wait_ld();
            };
            auto weights = [&](int c, uint32_t(&o1)[16], uint32_t(&o2)[16]) {  // o1: a | pe, o2: ds | p
                if (need_mask) {
                    // query t = t0 + 16 c + qq is valid iff key <= t and t < T
                    const int qlo = max(key - (t0 + 16 * c), 0);
                    const int qhi = T - (t0 + 16 * c);
                    b3_chunk<true>(vs, vg, vy, ve, rows + 64 * c, qhi <= 0 ? 16 : qlo, scale, scale_log2, o1, o2);
                    if (qhi < 16) {
#pragma unroll
                        for (int y = 0; y < 8; y++) {
                            const uint32_t keep = (2 * y + 1 < qhi) ? 0xFFFFFFFFu : (2 * y < qhi ? 0xFFFFu : 0u);
                            o1[y] &= keep;
                            o1[8 + y] &= keep;
                            o2[y] &= keep;
                            o2[8 + y] &= keep;
                        }
                    }
                } else {
                    b3_chunk<false>(vs, vg, vy, ve, rows + 64 * c, 0, scale, scale_log2, o1, o2);
                }
            };
            // ds and p rows into the swizzled [keys][queries] tiles: the 16-query
            // chunk c is the 16-byte chunks 2c and 2c + 1 of the 128-byte row
            auto store = [&](int c, const uint32_t(&o1)[16], const uint32_t(&o2)[16]) {
                const int ch = 2 * c;
                tmem_st16(tW + lrow + 16 * c, o1);
                *(uint4*)(dsrow + ((ch ^ (i & 7)) << 4)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                *(uint4*)(dsrow + (((ch + 1) ^ (i & 7)) << 4)) = make_uint4(o2[4], o2[5], o2[6], o2[7]);
                *(uint4*)(prow + ((ch ^ (i & 7)) << 4)) = make_uint4(o2[8], o2[9], o2[10], o2[11]);
                *(uint4*)(prow + (((ch + 1) ^ (i & 7)) << 4)) = make_uint4(o2[12], o2[13], o2[14], o2[15]);
            };
            uint32_t o1[16], o2[16];
            load(2 * wg);
            weights(2 * wg, o1, o2);
            load(2 * wg + 1);
            tc_fence_before();
            mbar_arrive(sx_free);  // every score of the sub-chunk this thread needs is in registers
            // the accumulation of j - 1 has read a|dg and p
            if (j > 0) ok = mbar_wait(w_free, (j - 1) & 1, wd, 10);
            if ((j & 1) == 0 && m >= 2) {
                // ds tile x held the staged dQ of tile m - 2: both reduces have read it
                if (leader) {
                    bulk_wait_read_all();
                    mbar_arrive(&stg_read[x]);
                }
                if (ok) ok = mbar_wait(&stg_read[x], ((m >> 1) - 1) & 1, wd, 8);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            store(2 * wg, o1, o2);
            weights(2 * wg + 1, o1, o2);
            store(2 * wg + 1, o1, o2);
            if (!ok) break;
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(w_full);
            // the dQ product of tile m - 1 was issued before this sub-chunk's accumulation
            if ((j & 1) == 0 && m >= 1) {
                ok = read_dq(m - 1);
                nread = m;
            }
        }
        // the remaining dQ tiles; the last one may hold one sub-chunk only
        for (int mm = nread; ok && mm < (nsub + 1) / 2; mm++) ok = read_dq(mm);
        if (leader) bulk_wait_all();  // the staging outlives its reduces
        if (ok) {
            ok = mbar_wait(fin, 0, wd, 11);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const uint32_t tsrc = wg == 0 ? tDV : tDK;  // warpgroup 0 writes dV, 1 writes dK
                __nv_bfloat16* dst_base = wg == 0 ? dv : dk;
#pragma unroll 1
                for (int c = 0; c < D / 32; c++) {
                    uint32_t v[32];
                    tmem_ld32(tsrc + lrow + 32 * c, v);
                    tmem_wait_ld();
                    if (key < T) {
                        uint4* pv = (uint4*)(dst_base + ((size_t)bh * T + key) * D + 32 * c);
#pragma unroll
                        for (int y = 0; y < 4; y++)
                            pv[y] = make_uint4(pack_bf16(__uint_as_float(v[8 * y]), __uint_as_float(v[8 * y + 1])),
                                               pack_bf16(__uint_as_float(v[8 * y + 2]), __uint_as_float(v[8 * y + 3])),
                                               pack_bf16(__uint_as_float(v[8 * y + 4]), __uint_as_float(v[8 * y + 5])),
                                               pack_bf16(__uint_as_float(v[8 * y + 6]), __uint_as_float(v[8 * y + 7])));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

__global__ void __launch_bounds__(256) tc_cast_dq(const float4* __restrict__ src, uint2* __restrict__ dst, size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 x = src[i];
        dst[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    }
}

// ============================================ pass 2 at d = 128, 128-key tiles
// Forward pass 2 with key tiles of 128, so S = c Q K^T and G = U K^T are
// N = 128 MMAs (the full tensor rate) and Acc += W V is one N = 128 chain of
// eight.  TMEM holds S [0,128), X [128,256), the f16 weights W [256,320) and
// Acc [320,448) in columns of their own, so the MMA thread issues the next key
// tile's S as soon as the elementwise warps hold this tile's S in registers,
// its X once they hold X, and the accumulation after them: the scores of tile
// j + 1 run while tile j's weights are formed.  Two elementwise warpgroups
// split each tile's keys (64 each).
// The CTAs are persistent, one per SM, and take (128-row query tile, head)
// items in work_item's order (longest tiles first within a head group) from a
// counter, so that one item's start overlaps the previous item's end:
//   - four 32 KB slots hold item l's Q and U tiles in one pair (2 (l & 1) and
//     the next) and its two-stage K ring in the other pair; the pairs swap
//     roles from item to item, so once every S and X product of item l has
//     run, item l + 1's Q, U and first K tiles load while item l's last
//     weights, accumulation and output store run;
//   - V has a ring of its own, and the output tile a staging slot of its own,
//     so Acc is read out while the next item's scores run;
//   - the MMA warp that issues S and X writes a record {item, key tile | last} per
//     tile, released with the tile's s_full; the elementwise warps and the
//     accumulation warp read it there (a ring of NINFO records), and an item
//     number of -1 ends every role's loop;
//   - the elementwise warps read an item's output out of Acc after they have
//     formed the next item's first weights (so the last accumulation's
//     latency is hidden), and load each item's per-row lse and gbar one item
//     ahead (the loader claims items two ahead and publishes the next one).
struct DualW {
    static constexpr int D = 128, BM = 128, BN = 128, NT = 352;  // TMA, S|X MMA, 8 elementwise, Acc MMA
    static constexpr int AB = BM * D * 2;  // one 32 KB slot: a Q, U, K, V or output tile
    static constexpr int KB = BN * D * 2;
    static constexpr int NS = 2;           // K stages per item, V stages
    static constexpr int NINFO = 4;        // tile records in flight
    // a_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full, s_free, x_free, w_full, w_free,
    // acc_done, acc_free, sx_done, item_full, drain
    static constexpr int NBAR = 1 + 4 * NS + 10;
    static constexpr int SMEM = 1024 + 4 * AB + NS * KB + AB + NBAR * 8 + 24 + 8 * NINFO;
    static constexpr unsigned TMEM_COLS = 512;  // S [0,128), X [128,256), W [256,320), Acc [320,448)
    static_assert(SMEM <= 232448, "one CTA per SM must fit");
};

// The item (query tile qt = ntq - 1 - rank, head bh) of work-list position
// `item`, its first row and its number of 128-key tiles.
__device__ __forceinline__ void dualw_item(int item, int BH, int ntq, int T, int* bh, int* q0, int* nkt) {
    int rank;
    work_item(item, BH, ntq, &rank, bh);
    *q0 = (ntq - 1 - rank) * DualW::BM;
    *nkt = min(*q0 + DualW::BM - 1, T - 1) / DualW::BN + 1;
}

__global__ void __launch_bounds__(DualW::NT, 1)
    tc_dual_w(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_out, const float* lse, const float* gbar, int T, int BH,
              int ntq, int* next_item, float scale_log2, unsigned* status) {
    // (next_item: a device counter, zero at launch; items gridDim.x onwards
    // are handed out from it.  lse, gbar and the counter are written by pass
    // 1 and read only past the griddepcontrol.wait below: lse and gbar are not
    // __restrict__, so the compiler may not move their loads above it.)
    using C = DualW;
    constexpr int NS = C::NS, D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* sSlot = sm;              // four 32 KB slots: Q, U and the K ring, by item parity
    uint8_t* sV = sSlot + 4 * C::AB;  // V stage s at s KB
    uint8_t* sOut = sV + NS * C::KB;  // the output tile, staged for its tensor store
    uint64_t* bars = (uint64_t*)(sOut + C::AB);
    uint64_t* a_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + NS;
    uint64_t* v_full = k_empty + NS;
    uint64_t* v_empty = v_full + NS;
    uint64_t* s_full = v_empty + NS;    // S and X of the tile are in TMEM and its record is written
    uint64_t* s_free = s_full + 1;      // the elementwise warps hold S in registers (256 arrivals)
    uint64_t* x_free = s_full + 2;      // ... and X (256 arrivals)
    uint64_t* w_full = s_full + 3;      // W of the tile is written (256 arrivals)
    uint64_t* w_free = s_full + 4;      // the accumulation has read W
    uint64_t* acc_done = s_full + 5;    // an item's last accumulation has run
    uint64_t* acc_free = s_full + 6;    // the elementwise warps hold an item's Acc in registers (256)
    uint64_t* sx_done = s_full + 7;     // every S and X product of an item has run
    uint64_t* item_full = s_full + 8;   // the next item number is in item_slot
    uint64_t* drain = s_full + 9;
    uint32_t* holder = (uint32_t*)(bars + C::NBAR);
    volatile int* abortf = (volatile int*)(holder + 1);
    volatile int* item_slot = (volatile int*)(holder + 2);  // [2][2] by item parity: {item, next item}
    volatile int* info = (volatile int*)(holder + 6);       // [NINFO][2] {item, key tile | last << 16} by tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = ntq * BH;
    const Watchdog wd{status, abortf, (unsigned)KID_TC_PASS2, wait_limit(status)};

    if (threadIdx.x == 0) {
        *abortf = 0;
        mbar_init(a_full, 1);
        for (int s = 0; s < NS; s++) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(s_full, 2);  // the products' commit and the record's arrival
        mbar_init(s_free, 256);
        mbar_init(x_free, 256);
        mbar_init(w_full, 256);
        mbar_init(w_free, 1);
        mbar_init(acc_done, 1);
        mbar_init(acc_free, 256);
        mbar_init(sx_done, 1);
        mbar_init(item_full, 1);
        mbar_init(drain, 2);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t tS = tmem, tX = tmem + 128, tW = tmem + 256, tAcc = tmem + 320;
    // launched as a programmatic dependent of pass 1: its outputs (the f16
    // copies, U, lse, gbar and the zeroed counter) are complete past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_a1);
            prefetch_tmap(&tm_a2);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int kiss = 0, viss = 0, aiss = 0;  // K tiles, V tiles and Q|U pairs issued
            int g0 = 0;                        // the item's first key tile, counted over this CTA's items
            // items l and l + 1: this CTA's first item, then the counter's, each
            // claimed an item ahead of its use so that the atomic's latency is hidden
            int cur = blockIdx.x;
            int nxt = (int)gridDim.x + atomicAdd(next_item, 1);
            bool ok = true;
            for (int l = 0;; l++) {
                // item l decoded before the wait, so that only the loads follow it
                int bh = 0, q0 = 0, nkt = 0;
                if (cur < n_items) dualw_item(cur, BH, ntq, T, &bh, &q0, &nkt);
                // every S and X product of item l - 1 has run: all four slots are free
                if (l > 0 && ok) ok = mbar_wait(sx_done, (l - 1) & 1, wd, 12);
                if (!ok || cur >= n_items) {
                    item_slot[2 * (l & 1)] = -1;
                    mbar_arrive(item_full);
                    break;
                }
                uint8_t* sA = sSlot + (l & 1) * 2 * C::AB;
                uint8_t* sK = sSlot + ((l & 1) ^ 1) * 2 * C::AB;
                mbar_expect_tx(a_full, 2 * C::AB);
#pragma unroll
                for (int r = 0; r < D / 64; r++) {
                    tma_load_3d(sA + r * C::BM * 128, &tm_a1, r * 64, q0, bh, a_full);
                    tma_load_3d(sA + C::AB + r * C::BM * 128, &tm_a2, r * 64, q0, bh, a_full);
                }
                aiss++;
                item_slot[2 * (l & 1)] = cur;
                item_slot[2 * (l & 1) + 1] = nxt < n_items ? nxt : -1;
                mbar_arrive(item_full);
                const int nn = nxt < n_items ? (int)gridDim.x + atomicAdd(next_item, 1) : n_items;
                cur = nxt;
                nxt = nn;
                // K(j), then V(j - 1): V lags K by one tile, so that K(j), which needs
                // only X(j - 2) to have run, is not held behind V(j - 1)'s wait for the
                // accumulation of tile j - 3 (which completes later)
                for (int j = 0; j <= nkt; j++) {
                    if (j < nkt) {
                        const int g = g0 + j, s = g % NS;
                        // the K stage's earlier reader in this item is tile g - NS
                        // (sx_done covered the earlier items)
                        if (j >= NS && !(ok = mbar_wait(&k_empty[s], ((g / NS) - 1) & 1, wd, 1))) break;
                        mbar_expect_tx(&k_full[s], C::KB);
#pragma unroll
                        for (int r = 0; r < D / 64; r++)
                            tma_load_3d(sK + s * C::KB + r * C::BN * 128, &tm_k, r * 64, j * C::BN, bh, &k_full[s]);
                        kiss = g + 1;
                    }
                    if (j >= 1) {  // V(j - 1); V's ring runs across items
                        const int g = g0 + j - 1, s = g % NS;
                        if (g >= NS && !(ok = mbar_wait(&v_empty[s], ((g / NS) - 1) & 1, wd, 1))) break;
                        mbar_expect_tx(&v_full[s], C::KB);
#pragma unroll
                        for (int r = 0; r < D / 64; r++)
                            tma_load_3d(sV + s * C::KB + r * C::BN * 128, &tm_v, r * 64, (j - 1) * C::BN, bh,
                                        &v_full[s]);
                        viss = g + 1;
                    }
                }
                g0 += nkt;
            }
            // every load issued lands before the CTA exits
            if (aiss > 0) mbar_wait_drain(a_full, (aiss - 1) & 1);
            for (int g = kiss > NS ? kiss - NS : 0; g < kiss; g++) mbar_wait_drain(&k_full[g % NS], (g / NS) & 1);
            for (int g = viss > NS ? viss - NS : 0; g < viss; g++) mbar_wait_drain(&v_full[g % NS], (g / NS) & 1);
        }
    } else if (warp == 1) {
        // S and X: the whole warp runs the loop, the elected lane issues
        const uint32_t idS = idesc_mma(128, C::BN, false, false);
        int g0 = 0;
        for (int l = 0;; l++) {
            if (!__all_sync(0xffffffffu, mbar_wait(item_full, l & 1, wd, 13))) break;
            const int item = item_slot[2 * (l & 1)];
            if (item < 0) {
                // the end, passed on in the next record once both elementwise
                // warpgroups have taken the last tile's S (s_free): they have
                // then waited on its s_full phase, which the end's arrivals
                // must not complete in their place
                if (g0 > 0 && !__all_sync(0xffffffffu, mbar_wait(s_free, (g0 - 1) & 1, wd, 15))) break;
                if (elect_one()) {
                    info[2 * (g0 % C::NINFO)] = -1;
                    mbar_arrive(s_full);
                    mbar_arrive(s_full);
                }
                __syncwarp();
                break;
            }
            int bh, q0, nkt;
            dualw_item(item, BH, ntq, T, &bh, &q0, &nkt);
            const uint32_t a1 = smem_u32(sSlot + (l & 1) * 2 * C::AB), a2 = a1 + C::AB;
            uint8_t* sK = sSlot + ((l & 1) ^ 1) * 2 * C::AB;
            bool ok = __all_sync(0xffffffffu, mbar_wait(a_full, l & 1, wd, 2));
            for (int j = 0; ok && j < nkt; j++) {
                const int g = g0 + j, s = g % NS;
                const uint32_t kaddr = smem_u32(sK + s * C::KB);
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&k_full[s], (g / NS) & 1, wd, 3)))) break;
                // tile g - 1's S is in registers: tile g's may overwrite it; then X likewise
                if (g > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(s_free, (g - 1) & 1, wd, 9)))) break;
                tc_fence_after();
                if (elect_one()) {
                    info[2 * (g % C::NINFO)] = item;
                    info[2 * (g % C::NINFO) + 1] = j | (j == nkt - 1 ? 1 << 16 : 0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tS, desc_kmajor(a1, C::BM, kk), desc_kmajor(kaddr, C::BN, kk), idS, kk > 0);
                }
                __syncwarp();
                if (g > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(x_free, (g - 1) & 1, wd, 11)))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; kk++)
                        mma_ss(tX, desc_kmajor(a2, C::BM, kk), desc_kmajor(kaddr, C::BN, kk), idS, kk > 0);
                    mma_commit(s_full);
                    mma_commit(&k_empty[s]);             // K(g) has no other reader
                    if (j == nkt - 1) mma_commit(sx_done);  // the item's slots may be reloaded
                    mbar_arrive(s_full);                 // the record above is written
                }
                __syncwarp();
            }
            if (!ok) break;
            g0 += nkt;
        }
        if (elect_one()) mma_commit(drain);  // one arrival per issuing warp
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else if (warp == C::NT / 32 - 1) {
        // the accumulation Acc += W V, item after item
        const uint32_t idA = idesc_mma(128, D, false, true);
        int l = 0;  // items whose last accumulation is issued
        for (int g = 0;; g++) {
            if (!__all_sync(0xffffffffu, mbar_wait(w_full, g & 1, wd, 5))) break;
            const int item = info[2 * (g % C::NINFO)];
            if (item < 0) break;
            const int jl = info[2 * (g % C::NINFO) + 1], j = jl & 0xFFFF, s = g % NS;
            const bool last = (jl >> 16) != 0;  // the item's last key tile
            // the elementwise warps have read the previous item's Acc
            if (j == 0 && l > 0 && !__all_sync(0xffffffffu, mbar_wait(acc_free, (l - 1) & 1, wd, 14))) break;
            if (!__all_sync(0xffffffffu, mbar_wait(&v_full[s], (g / NS) & 1, wd, 4))) break;
            tc_fence_after();
            const uint32_t vaddr = smem_u32(sV + s * C::KB);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; kk++)
                    mma_ts(tAcc, tW + kk * 8, desc_mnmajor(vaddr, C::BN, kk), idA, (j > 0 || kk > 0) ? 1u : 0u);
                if (last) mma_commit(acc_done);  // one phase per item: the epilogue's wait
                mma_commit(w_free);
                mma_commit(&v_empty[s]);
            }
            __syncwarp();
            if (last) l++;
        }
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0);
    } else {
        const int wg = (warp - 2) >> 2;  // keys [64 wg, 64 wg + 64) of every tile
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const uint32_t lrow = (uint32_t)(qd * 32) << 16;
        const bool leader = qd == 0 && lane == 0;  // issues the warpgroup's output stores
        const uint64_t SL2 = f2(scale_log2, scale_log2);
        uint8_t* slot = sOut + wg * (C::BM * 128);  // this warpgroup's 64 output columns
        // Every named-barrier step below is reached by all four warps of the
        // warpgroup (a wait that fails skips work, not the step), and the
        // warps leave the item loop together, right after a warpgroup-wide
        // AND, so that none of them waits at a named barrier the others never
        // reach.
        bool ok = true;
        int g = 0;
        int pbh = 0, pq0 = 0;                          // the item whose output is still in Acc
        int pf_item = -1;                              // the next item, and its row's lse and gbar
        float pf_lse = 0.f, pf_gbar = 0.f;
        // item lp's output: Acc to registers (then the next item's
        // accumulation may overwrite it), bf16 into this warpgroup's half of
        // the staging slot once its previous store has read it, one tensor
        // store per warpgroup
        auto epilogue = [&](int lp) {
            if (ok) ok = mbar_wait(acc_done, lp & 1, wd, 8);
            ok = named_bar_and(1 + wg, 128, ok);
            if (!ok) return;
            tc_fence_after();
            uint32_t va[32], vb[32];
            tmem_ld32(tAcc + lrow + 64 * wg, va);
            tmem_ld32(tAcc + lrow + 64 * wg + 32, vb);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(acc_free);
            if (leader) bulk_wait_read_all();
            named_bar_sync(1 + wg, 128);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                *(uint4*)(slot + sw_off(row, 8 * i, C::BM)) =
                    make_uint4(pack_bf16(__uint_as_float(va[8 * i]), __uint_as_float(va[8 * i + 1])),
                               pack_bf16(__uint_as_float(va[8 * i + 2]), __uint_as_float(va[8 * i + 3])),
                               pack_bf16(__uint_as_float(va[8 * i + 4]), __uint_as_float(va[8 * i + 5])),
                               pack_bf16(__uint_as_float(va[8 * i + 6]), __uint_as_float(va[8 * i + 7])));
                *(uint4*)(slot + sw_off(row, 32 + 8 * i, C::BM)) =
                    make_uint4(pack_bf16(__uint_as_float(vb[8 * i]), __uint_as_float(vb[8 * i + 1])),
                               pack_bf16(__uint_as_float(vb[8 * i + 2]), __uint_as_float(vb[8 * i + 3])),
                               pack_bf16(__uint_as_float(vb[8 * i + 4]), __uint_as_float(vb[8 * i + 5])),
                               pack_bf16(__uint_as_float(vb[8 * i + 6]), __uint_as_float(vb[8 * i + 7])));
            }
            fence_proxy_async_smem();
            named_bar_sync(1 + wg, 128);
            if (leader) {
                tma_store_3d(&tm_out, 64 * wg, pq0, pbh, slot);
                bulk_commit();
            }
        };
        for (int l = 0;; l++) {
            // the next item's first record
            int item = -1;
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, wd, 6));
                if (ok) item = info[2 * (g % C::NINFO)];
            }
            if (!named_bar_and(1 + wg, 128, ok && item >= 0)) {
                if (l > 0) epilogue(l - 1);
                // the end, for the accumulation warp: after the last output is
                // read (its acc_done wait follows every arrival on the last
                // tile's w_full phase, which this arrival must not join)
                if (ok && item < 0) mbar_arrive(w_full);
                break;
            }
            int bh, q0, nkt;
            dualw_item(item, BH, ntq, T, &bh, &q0, &nkt);
            const int t = q0 + row;
            const bool valid = t < T;
            if (item != pf_item) {
                const int tc = min(t, T - 1);
                pf_lse = lse[(size_t)bh * T + tc];
                pf_gbar = gbar[(size_t)bh * T + tc];
            }
            const float L2 = valid ? pf_lse * LOG2E : 0.f;
            const float g1 = valid ? 1.f - pf_gbar : 0.f;
            const uint64_t NL2 = f2(-L2, -L2), G1 = f2(g1, g1);
            // the next item's, one item ahead (used only at its start)
            pf_item = item_slot[2 * (l & 1) + 1];
            if (pf_item >= 0) {
                int nbh, nq0, nnkt;
                dualw_item(pf_item, BH, ntq, T, &nbh, &nq0, &nnkt);
                const int tc = min(nq0 + row, T - 1);
                pf_lse = lse[(size_t)nbh * T + tc];
                pf_gbar = gbar[(size_t)nbh * T + tc];
            }
            for (int j = 0; j < nkt; j++, g++) {
                if (ok && j > 0) ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, wd, 6));
                if (ok) {
                    tc_fence_after();
                    const int k0 = j * C::BN;
                    const int lim = (k0 + C::BN - 1 > q0) ? t - k0 : C::BN;
                    const bool need_mask = lim < C::BN;
                    // W of one 32-key chunk c: w = p (x + 1 - gbar), p = exp2(c s - L)
                    auto weights = [&](int c, const uint32_t(&vs)[32], const uint32_t(&vx)[32],
                                       uint32_t(&pk)[16]) {
#pragma unroll
                        for (int i = 0; i < 16; i++) {  // keys 2i, 2i + 1 of the chunk, one f32x2 op each
                            const int cc = c * 32 + 2 * i;
                            const float2 xs = uf2(
                                ffma2(f2(__uint_as_float(vs[2 * i]), __uint_as_float(vs[2 * i + 1])), SL2, NL2));
                            float p0 = fast_exp2(xs.x), p1 = fast_exp2(xs.y);
                            if (need_mask) {
                                if (cc > lim) p0 = 0.f;
                                if (cc + 1 > lim) p1 = 0.f;
                            }
                            const uint64_t xv = f2(__uint_as_float(vx[2 * i]), __uint_as_float(vx[2 * i + 1]));
                            const float2 w = uf2(fmul2(f2(p0, p1), fadd2(xv, G1)));
                            pk[i] = pack_f16(w.x, w.y);
                        }
                    };
                    const int c0 = 2 * wg, c1 = 2 * wg + 1;
                    uint32_t pk0[16], pk1[16];
                    uint32_t vs0[32], vs1[32];
                    tmem_ld32(tS + lrow + c0 * 32, vs0);
                    tmem_ld32(tS + lrow + c1 * 32, vs1);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(s_free);  // S of the tile this thread needs is in registers
                    {
                        uint32_t vx[32];
                        tmem_ld32(tX + lrow + c0 * 32, vx);
                        tmem_wait_ld();
                        weights(c0, vs0, vx, pk0);
                    }
                    {
                        uint32_t vx[32];
                        tmem_ld32(tX + lrow + c1 * 32, vx);
                        tmem_wait_ld();
                        tc_fence_before();
                        mbar_arrive(x_free);  // ... and X
                        weights(c1, vs1, vx, pk1);
                    }
                    if (g > 0) ok = mbar_wait(w_free, (g - 1) & 1, wd, 10);  // the previous accumulation read W
                    ok = __all_sync(0xffffffffu, ok);
                    if (ok) {
                        tc_fence_after();
                        tmem_st16(tW + lrow + c0 * 16, pk0);
                        tmem_st16(tW + lrow + c1 * 16, pk1);
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(w_full);
                    }
                }
                // the previous item's output, once this item's first weights are out
                if (j == 0 && l > 0) epilogue(l - 1);
            }
            pbh = bh;
            pq0 = q0;
        }
        if (leader) bulk_wait_all();  // the slot stays valid until the last store has read it
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ================================================================= host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

// A 16-bit [BH][T][D] tensor viewed as 3-D (D, T, BH) with a box of 64 x rows
// x 1 and the 128-byte swizzle; rows past T (within a head) read as zero.
bool make_map(CUtensorMap* m, const void* base, int D, int T, int BH, int rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define PLX_TRY(x)                         \
    do {                                   \
        cudaError_t e_ = (x);              \
        if (e_ != cudaSuccess) return e_;  \
    } while (0)


// Workspace of the tensor-core forward: f16 copies of q, k, v, then U (f16),
// gbar (fp32) and the work counter of the persistent pass 2.
struct TcFwdWs {
    __half *q16, *k16, *v16, *U;
    float* gbar;
    int* item_ctr;
};
TcFwdWs tc_fwd_ws(void* ws, int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T, nd2 = align256(n * d * 2);
    char* p = (char*)ws;
    TcFwdWs w;
    w.q16 = (__half*)p;
    w.k16 = (__half*)(p + nd2);
    w.v16 = (__half*)(p + 2 * nd2);
    w.U = (__half*)(p + 3 * nd2);
    w.gbar = (float*)(p + 4 * nd2);
    w.item_ctr = (int*)(p + 4 * nd2 + align256(n * 4));
    return w;
}

// Workspace of the tensor-core backward.
struct TcBwdWs {
    float *R, *dq_acc, *ebar, *partial;
    float* rows;  // per head ceil(T/2) query pairs x 8 floats
    __half *U, *dmu, *q16, *k16, *v16, *do16;
};
TcBwdWs tc_bwd_ws(void* ws, int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T, nd4 = align256(n * d * 4), nd2 = align256(n * d * 2);
    char* p = (char*)ws;
    TcBwdWs w;
    w.R = (float*)p; p += nd4;
    w.dq_acc = (float*)p; p += nd4;
    w.U = (__half*)p; p += nd2;
    w.dmu = (__half*)p; p += nd2;
    w.q16 = (__half*)p; p += nd2;
    w.k16 = (__half*)p; p += nd2;
    w.v16 = (__half*)p; p += nd2;
    w.do16 = (__half*)p; p += nd2;
    w.ebar = (float*)p; p += align256(n * 4);
    w.rows = (float*)p; p += align256((size_t)B * H * ((T + 1) / 2) * 32);
    w.partial = (float*)p;
    return w;
}
size_t tc_bwd_bytes(int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T;
    const size_t nchunks = ((size_t)B * T + 511) / 512;  // RowCfg<d>::ROWS_PER_CTA
    return 2 * align256(n * d * 4) + 6 * align256(n * d * 2) + align256(n * 4) +
           align256((size_t)B * H * ((T + 1) / 2) * 32) +
           align256((size_t)H * nchunks * d * d * 4);
}

// Row scalars: per head ceil(T/2) query pairs of 8 floats, viewed as 3-D
// (8, pairs, BH) with a box of 8 x pairs_box x 1 (no swizzle).
// fp32 [BH][T][D] in 32-column boxes of `rows` rows, 128-byte swizzle.
bool make_map_f32(CUtensorMap* m, const void* base, int D, int T, int BH, int rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)T * D * 4};
    cuuint32_t box[3] = {32, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_rows_map(CUtensorMap* m, const void* base, int T, int BH, int pairs_box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t np = (cuuint64_t)(T + 1) / 2;
    cuuint64_t dims[3] = {8, np, (cuuint64_t)BH};
    cuuint64_t strides[2] = {32, np * 32};
    cuuint32_t box[3] = {8, (cuuint32_t)pairs_box, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t to_f16(const void* const* src, __half* const* dst, int count, size_t n, cudaStream_t s) {
    CvtJob job{};
    for (int i = 0; i < count; i++) {
        job.src[i] = (const uint4*)src[i];
        job.dst[i] = (uint4*)dst[i];
    }
    const size_t n8 = n / 8;  // n = B H T d, a multiple of 64
    const unsigned gx = (unsigned)std::min<size_t>((n8 + 255) / 256, 148 * 8);
    timing_begin(s, "tc_to_f16");
    tc_to_f16<<<dim3(gx, count), 256, 0, s>>>(job, n8);
    timing_end(s);
    return cudaGetLastError();
}

template <int D>
cudaError_t fwd_impl(const FwdArgs& a, const TcFwdWs& w, const std::function<cudaError_t()>& after_pass1 = {}) {
    const int BH = a.B * a.H;
    const float scale_log2 = LOG2E / sqrtf((float)D);
    const size_t n = (size_t)BH * a.T * D;
    // pass 1 reads the bf16 inputs (a 16-bit map copies the bytes as they
    // are) and writes the f16 copies of q, k, v that pass 2 reads
    CUtensorMap mq_in, mk_in, mv_in, mk16_128, mv16_128, mq128, mu128, mk64, mv64, mmu, mout;
    if (!make_map(&mq_in, a.q, D, a.T, BH, 128) || !make_map(&mk_in, a.k, D, a.T, BH, 128) ||
        !make_map(&mout, a.out, D, a.T, BH, 128) ||
        !make_map(&mv_in, a.v, D, a.T, BH, 128) || !make_map(&mv16_128, w.v16, D, a.T, BH, 128) ||
        !make_map_f32(&mmu, a.mu_k, D, a.T, BH, 128) ||
        !make_map(&mk16_128, w.k16, D, a.T, BH, 128) || !make_map(&mq128, w.q16, D, a.T, BH, 128) ||
        !make_map(&mu128, w.U, D, a.T, BH, 128) || !make_map(&mk64, w.k16, D, a.T, BH, 64) ||
        !make_map(&mv64, w.v16, D, a.T, BH, 64))
        return cudaErrorInvalidValue;
    (void)n;
    {  // pass 1: two query tiles per CTA, projection after the key loop
        using C = P1PP<D>;
        const int npairs = ((a.T + C::BM - 1) / C::BM + 1) / 2;
        PLX_TRY(cudaFuncSetAttribute(tc_pass1_pp<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_pass1");
        tc_pass1_pp<D><<<npairs * BH, C::NT, C::SMEM, a.stream>>>(
            mq_in, mk_in, mk16_128, mmu, mu128, mq128, mv_in, mv16_128, a.P, a.lse, w.gbar, a.T,
            a.H, BH, npairs, scale_log2, D == 128 ? w.item_ctr : nullptr, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    }
    if (after_pass1) PLX_TRY(after_pass1());
    if constexpr (D == 128) {  // pass 2: 128-key tiles, persistent CTAs, one per SM
        using C = DualW;
        const int ntq = (a.T + C::BM - 1) / C::BM;
        int dev = 0, sms = 0;
        PLX_TRY(cudaGetDevice(&dev));
        PLX_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        const int cap = persistent_cta_cap();
        const int grid = std::min(cap > 0 ? std::min(cap, sms) : sms, ntq * BH);
        PLX_TRY(cudaFuncSetAttribute(tc_dual_w, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_pass2");
        {  // a programmatic dependent of pass 1: its CTAs set up on the SMs pass 1's last CTAs free
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(grid);
            cfg.blockDim = dim3(C::NT);
            cfg.dynamicSmemBytes = C::SMEM;
            cfg.stream = a.stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            PLX_TRY(cudaLaunchKernelEx(&cfg, tc_dual_w, mq128, mu128, mk16_128, mv16_128, mout, (const float*)a.lse,
                                       (const float*)w.gbar, a.T, BH, ntq, w.item_ctr, scale_log2, a.status));
        }
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    } else {  // pass 2
        using C = DualCfg<D>;
        const int ntq = (a.T + C::BM - 1) / C::BM;
        PLX_TRY(cudaFuncSetAttribute(tc_dual<D, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_pass2");
        tc_dual<D, 0><<<ntq * BH, C::NT, C::SMEM, a.stream>>>(mq128, mu128, mk64, mv64, mout, a.lse, w.gbar,
                                                                  nullptr, a.T, BH, ntq, scale_log2, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    }
    return cudaSuccess;
}

template <int D>
// parts: 1 = the dO (or all) operand copies and B1, 2 = B2 onwards, 3 = all.
cudaError_t bwd_impl(const BwdArgs& a, bool copies_ready, int parts = 3) {
    const int BH = a.B * a.H;
    const float scale = 1.f / sqrtf((float)D);
    const float scale_log2 = LOG2E * scale;
    const size_t n = (size_t)BH * a.T * D;
    TcBwdWs w = tc_bwd_ws(a.ws, a.B, a.H, a.T, D);
    CUtensorMap mq128, mdo128, mk64, mv64, mk128, mv128, mq64, mu64, mdmu64, mdo64, mrows, mR;
    if (!make_map(&mq128, w.q16, D, a.T, BH, 128) || !make_map(&mdo128, w.do16, D, a.T, BH, 128) ||
        !make_map_f32(&mR, w.R, D, a.T, BH, 128) ||
        !make_map(&mk64, w.k16, D, a.T, BH, 64) || !make_map(&mv64, w.v16, D, a.T, BH, 64) ||
        !make_map(&mk128, w.k16, D, a.T, BH, 128) || !make_map(&mv128, w.v16, D, a.T, BH, 128) ||
        !make_map(&mq64, w.q16, D, a.T, BH, 64) || !make_map(&mu64, w.U, D, a.T, BH, 64) ||
        !make_map(&mdmu64, w.dmu, D, a.T, BH, 64) || !make_map(&mdo64, w.do16, D, a.T, BH, 64) ||
        !make_rows_map(&mrows, w.rows, a.T, BH, 32))
        return cudaErrorInvalidValue;
    if (!(parts & 1)) {
    } else if (copies_ready) {  // the forward of the same step made the copies of q, k, v
        const void* src[1] = {a.dout};
        __half* dst[1] = {w.do16};
        PLX_TRY(to_f16(src, dst, 1, n, a.stream));
    } else {
        const void* src[4] = {a.q, a.k, a.v, a.dout};
        __half* dst[4] = {w.q16, w.k16, w.v16, w.do16};
        PLX_TRY(to_f16(src, dst, 4, n, a.stream));
    }
    if (!(parts & 1)) {
    } else if constexpr (D == 128) {  // B1: R = sum p e k, ebar = sum p e (two query tiles per CTA)
        using C = DualPP<D>;
        const int npairs = ((a.T + C::BM - 1) / C::BM + 1) / 2;
        PLX_TRY(cudaFuncSetAttribute(tc_dual_pp<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_bwd_b1");
        tc_dual_pp<D, 1><<<npairs * BH, C::NT, C::SMEM, a.stream>>>(mq128, mdo128, mk64, mv64, mR, a.lse, nullptr,
                                                                     w.ebar, a.T, BH, npairs, scale_log2, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    } else {  // B1: R = sum p e k, ebar = sum p e
        using C = DualCfg<D>;
        const int ntq = (a.T + C::BM - 1) / C::BM;
        PLX_TRY(cudaFuncSetAttribute(tc_dual<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_bwd_b1");
        tc_dual<D, 1><<<ntq * BH, C::NT, C::SMEM, a.stream>>>(mq128, mdo128, mk64, mv64, mR, a.lse, nullptr,
                                                                  w.ebar, a.T, BH, ntq, scale_log2, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    }
    if (!(parts & 2)) return cudaSuccess;
    {  // B2: row math and the dP_h partials
        using R = RowCfg<D>;
        const int nchunks = (a.B * a.T + R::ROWS_PER_CTA - 1) / R::ROWS_PER_CTA;
        if (D == 64) {
            PLX_TRY(cudaFuncSetAttribute(tc_b2, cudaFuncAttributeMaxDynamicSharedMemorySize, B2T::SMEM));
            int dev = 0, sms = 0;
            PLX_TRY(cudaGetDevice(&dev));
            PLX_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
            const int cap = persistent_cta_cap();  // persistent: two CTAs per SM
            const int grid = std::min(cap > 0 ? std::min(cap, 2 * sms) : 2 * sms, nchunks * a.H);
            timing_begin(a.stream, "tc_bwd_b2");
            tc_b2<<<grid, B2T::NT, B2T::SMEM, a.stream>>>(w.q16, a.mu_k, a.P, a.lse, w.R, w.ebar, w.U, w.dmu,
                                                          w.dq_acc, w.rows, w.partial, a.B, a.H, a.T, nchunks,
                                                          a.status);
        } else {
            const size_t sm = R::smem(1);
            PLX_TRY(cudaFuncSetAttribute(tc_rows<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
            timing_begin(a.stream, "tc_bwd_b2");
            tc_rows<D, 1><<<dim3(nchunks, a.H), R::NT, sm, a.stream>>>((const __nv_bfloat16*)a.q, a.mu_k, a.P,
                                                                       a.lse, w.R, w.ebar, w.U, nullptr, w.dmu,
                                                                       w.dq_acc, w.rows, w.partial, a.B, a.H, a.T);
        }
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
        const int dd4 = D * D / 4;
        timing_begin(a.stream, "tc_dp_reduce");
        tc_dp_reduce<<<dim3((dd4 + 255) / 256, a.H), 256, 0, a.stream>>>((const float4*)w.partial, (float4*)a.dP,
                                                                           nchunks, dd4);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    }
    if constexpr (D == 64) {  // B3: dK, dV, dQ (64-query sub-chunks)
        using C = B3Q;
        CUtensorMap mdq;
        if (!make_map_f32(&mdq, w.dq_acc, D, a.T, BH, C::QT)) return cudaErrorInvalidValue;
        const int nkt = (a.T + C::BK - 1) / C::BK;
        PLX_TRY(cudaFuncSetAttribute(tc_bwd_b3_q64, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_bwd_b3");
        tc_bwd_b3_q64<<<nkt * BH, C::NT, C::SMEM, a.stream>>>(mk128, mv128, mq64, mu64, mdmu64, mdo64, mrows,
                                                               mdq, (__nv_bfloat16*)a.dk, (__nv_bfloat16*)a.dv,
                                                               a.T, BH, nkt, scale, scale_log2, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    } else {  // B3: dK, dV, dQ
        using C = B3Cfg<D>;
        const int nkt = (a.T + C::BK - 1) / C::BK;
        PLX_TRY(cudaFuncSetAttribute(tc_bwd_b3<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        timing_begin(a.stream, "tc_bwd_b3");
        tc_bwd_b3<D><<<nkt * BH, C::NT, C::SMEM, a.stream>>>(
            mk128, mv128, mq64, mu64, mdmu64, mdo64, mrows, w.dq_acc, (__nv_bfloat16*)a.dk, (__nv_bfloat16*)a.dv,
            a.T, BH, nkt, scale, scale_log2, a.status);
        timing_end(a.stream);
        PLX_TRY(cudaGetLastError());
    }
    {
        const size_t n4 = n / 4;
        const unsigned gx = (unsigned)std::min<size_t>((n4 + 255) / 256, 148 * 8);
        timing_begin(a.stream, "tc_cast_dq");
        tc_cast_dq<<<gx, 256, 0, a.stream>>>((const float4*)w.dq_acc, (uint2*)a.dq, n4);
        timing_end(a.stream);
    }
    return cudaGetLastError();
}

template <int D>
cudaError_t probe_impl(const ProbeArgs& a) {
    using C = ProbeCfg<D>;
    const int BH = a.B * a.H;
    const float scale_log2 = LOG2E / sqrtf((float)D);
    const size_t n = (size_t)BH * a.T * D, nd2 = align256(n * 2);
    __half* q16 = (__half*)a.ws;
    __half* r16 = (__half*)((char*)a.ws + nd2);
    __half* k16 = (__half*)((char*)a.ws + 2 * nd2);
    __half* v16 = (__half*)((char*)a.ws + 3 * nd2);
    CUtensorMap mq, mr, mk, mv;
    if (!make_map(&mq, q16, D, a.T, BH, 128) || !make_map(&mr, r16, D, a.T, BH, 128) ||
        !make_map(&mk, k16, D, a.T, BH, 64) || !make_map(&mv, v16, D, a.T, BH, 64))
        return cudaErrorInvalidValue;
    {
        const void* src[4] = {a.q, a.rho, a.k, a.v};
        __half* dst[4] = {q16, r16, k16, v16};
        PLX_TRY(to_f16(src, dst, 4, n, a.stream));
    }
    const int ntq = (a.T + C::BM - 1) / C::BM;
    PLX_TRY(cudaFuncSetAttribute(tc_probe_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    timing_begin(a.stream, "tc_probe");
    tc_probe_kernel<D><<<ntq * BH, C::NT, C::SMEM, a.stream>>>(mq, mr, mk, mv, (__nv_bfloat16*)a.out, a.lse, a.T,
                                                                BH, ntq, scale_log2, a.status);
    timing_end(a.stream);
    return cudaGetLastError();
}

}  // namespace

bool tc_available() { return encode_fn() != nullptr; }

bool tc_make_map(void* map, const void* base, int D, int T, int BH, int rows) {
    return make_map(reinterpret_cast<CUtensorMap*>(map), base, D, T, BH, rows);
}

size_t tc_fwd_ws_bytes(int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T;
    return 4 * align256(n * d * 2) + align256(n * 4) + 256;
}

size_t tc_bwd_ws_bytes(int B, int H, int T, int d) { return tc_bwd_bytes(B, H, T, d); }

cudaError_t tc_fwd(const FwdArgs& a) {
    if (a.dtype != 1) return cudaErrorNotSupported;
    if (a.d == 64) return fwd_impl<64>(a, tc_fwd_ws(a.ws, a.B, a.H, a.T, 64));
    return fwd_impl<128>(a, tc_fwd_ws(a.ws, a.B, a.H, a.T, 128));
}

// Forward and backward of one step in one workspace (the backward's): the
// forward's f16 copies of q, k and v are written where the backward reads
// them, its U in the backward's U region (B2 rewrites it after pass 2 has read
// it) and its gbar in the dq accumulator's (written from B2 on), so the
// backward converts dO alone.  B1 needs only pass 1's results, so it runs on a
// second stream beside pass 2 (the two kernels each leave the tensor pipe
// partly idle); B2 waits for both.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
cudaError_t side_stream(SideStream** out, std::unique_lock<std::mutex>* lock) {
    static SideStream cache[64];
    static std::mutex mu[64];
    int dev = 0;
    PLX_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    *lock = std::unique_lock<std::mutex>(mu[dev]);  // the events are reused: one caller enqueues at a time
    SideStream& x = cache[dev];
    if (!x.s) {
        PLX_TRY(cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking));
        PLX_TRY(cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming));
        PLX_TRY(cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming));
    }
    *out = &x;
    return cudaSuccess;
}

template <int D>
cudaError_t fwd_bwd_impl(const FwdArgs& f, const BwdArgs& b) {
    const TcBwdWs w = tc_bwd_ws(b.ws, b.B, b.H, b.T, D);
    TcFwdWs fw;
    fw.q16 = w.q16;
    fw.k16 = w.k16;
    fw.v16 = w.v16;
    fw.U = w.U;
    fw.gbar = w.dq_acc;
    fw.item_ctr = (int*)w.rows;  // B2 writes the rows only after pass 2
    SideStream* ss = nullptr;
    std::unique_lock<std::mutex> lock;
    PLX_TRY(side_stream(&ss, &lock));
    auto b1_beside = [&]() -> cudaError_t {
        PLX_TRY(cudaEventRecord(ss->fork, f.stream));
        PLX_TRY(cudaStreamWaitEvent(ss->s, ss->fork, 0));
        BwdArgs b1 = b;
        b1.stream = ss->s;
        PLX_TRY(bwd_impl<D>(b1, true, 1));
        return cudaEventRecord(ss->join, ss->s);
    };
    PLX_TRY(fwd_impl<D>(f, fw, b1_beside));
    PLX_TRY(cudaStreamWaitEvent(b.stream, ss->join, 0));
    return bwd_impl<D>(b, true, 2);
}

cudaError_t tc_fwd_bwd(const FwdArgs& f, const BwdArgs& b) {
    if (f.dtype != 1) return cudaErrorNotSupported;
    return f.d == 64 ? fwd_bwd_impl<64>(f, b) : fwd_bwd_impl<128>(f, b);
}

size_t tc_probe_ws_bytes(int B, int H, int T, int d) {
    const size_t n = (size_t)B * H * T;
    return 4 * align256(n * d * 2);
}

cudaError_t tc_probe(const ProbeArgs& a) {
    if (a.dtype != 1) return cudaErrorNotSupported;
    return a.d == 64 ? probe_impl<64>(a) : probe_impl<128>(a);
}

cudaError_t tc_bwd(const BwdArgs& a) {
    if (a.dtype != 1) return cudaErrorNotSupported;
    return a.d == 64 ? bwd_impl<64>(a, false) : bwd_impl<128>(a, false);
}

}  // namespace plx
