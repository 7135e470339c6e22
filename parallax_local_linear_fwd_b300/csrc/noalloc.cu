// parallax_fwd_noalloc: the forward for callers that must not allocate device
// memory.
//
// Some callers cannot call cudaMalloc.  Examples: a host whose device memory
// belongs to another allocator (a framework's caching allocator, or an arena
// with a fixed budget) that must not have memory taken behind its back; a
// latency-critical loop where cudaMalloc/cudaFree would synchronise the
// device; or a plugin that may not allocate once it is initialised.
// parallax_fwd allocates its workspace (the probe u and gbar) stream-ordered
// on every call.  This entry point instead uses one fixed scratch array that
// is compiled into the library.  It runs the same SIMT forward kernels as
// parallax_fwd does on the SIMT path.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads this library holds it until the process exits.  Host code cannot
// use the array's name as a device address.  The first call on each device
// therefore looks up the address with cudaGetSymbolAddress, with that device
// current, and caches it together with the identity of the device's CUDA
// context.  A later call in another context of that device (after
// cudaDeviceReset destroyed the one the address belonged to) looks the
// address up again instead of using a stale one.  Make the first call, and
// the first call after a reset, outside any stream capture.
// All calls share the one array, which keeps the last call's contents.  The
// forward writes every scratch element it reads, so nothing needs clearing.
// Calls that overlap on the GPU (different streams, or threads that share a
// device) race on the array, and the caller must serialise them.
// The SIMT forward kernels have no bounded device waits, so no watchdog word
// is needed either: this path touches no memory but the caller's buffers and
// the static array.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "parallax.h"
#include "plx_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_noalloc_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identity of the calling thread's current CUDA context (unique for the
// process's lifetime, so a context created after a reset never repeats it).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (CtxGetCurrentFn)p;
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (CtxGetIdFn)p;
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Once per device and context, with that device current: look up the device
// address of the static array.  No allocation happens here.
int noalloc_setup(void** scratch) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PLX_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PLX_ERR_UNSUPPORTED;
    // cudaGetDevice alone does not create the context; cudaSetDevice does
    // (it initialises the device's primary context) and allocates nothing
    if (cudaSetDevice(dev) != cudaSuccess) return PLX_ERR_CUDA;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return PLX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return PLX_ERR_CUDA;
        if (major != 10 || minor != 3) return PLX_ERR_UNSUPPORTED;
        void* s = nullptr;
        if (cudaGetSymbolAddress(&s, g_noalloc_scratch) != cudaSuccess || s == nullptr) return PLX_ERR_CUDA;
        g_scratch_ptr[dev] = s;
        g_scratch_ctx[dev] = ctx;
    }
    *scratch = g_scratch_ptr[dev];
    return PLX_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int parallax_fwd_noalloc(const void* q, const void* k, const void* v, const float* P, void* out,
                                    float* lse, float* mu_k, int B, int H, int T, int d, int dtype,
                                    void* stream) {
    if (B < 1 || H < 1 || T < 1 || d < 1) return PLX_ERR_INVALID_ARG;
    if (dtype != PLX_FP32 && dtype != PLX_BF16) return PLX_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
    if ((unsigned long long)B * H * T * d >= (1ull << 31)) return PLX_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return PLX_ERR_UNSUPPORTED;
    if (!q || !k || !v || !P || !out || !lse || !mu_k) return PLX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(P) || !aligned16(out) ||
        !aligned16(lse) || !aligned16(mu_k))
        return PLX_ERR_INVALID_ARG;
    if (plx::simt_fwd_ws_bytes(B, H, T, d) > kScratchBytes) return PLX_ERR_TOO_LARGE;
    void* scratch = nullptr;
    int rc = noalloc_setup(&scratch);
    if (rc) return rc;
    plx::FwdArgs a{q, k, v, P, out, lse, mu_k, scratch, B, H, T, d, dtype, (cudaStream_t)stream, nullptr};
    return plx::simt_fwd(a) == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}
