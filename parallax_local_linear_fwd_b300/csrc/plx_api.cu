// C ABI of libparallax.so: argument checks, workspace handling, kernel-family
// dispatch and the device watchdog word.  Declarations and contracts are in
// include/parallax.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "parallax.h"
#include "plx_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status[kMaxDevices] = {};  // per-device watchdog word (4 x u32)
int g_arch_ok[kMaxDevices] = {};        // 0 unknown, 1 sm_103, -1 other
std::atomic<int> g_path{PLX_PATH_AUTO};
std::atomic<int> g_persist_cap{0};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Returns PLX_OK and the current device's status word, creating it once.
int device_state(unsigned** status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PLX_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PLX_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return PLX_ERR_CUDA;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1) return PLX_ERR_UNSUPPORTED;
    if (!g_status[dev]) {
        unsigned* p = nullptr;
        if (cudaMalloc(&p, 4 * sizeof(unsigned)) != cudaSuccess) return PLX_ERR_CUDA;
        if (cudaMemset(p, 0, 4 * sizeof(unsigned)) != cudaSuccess) {
            cudaFree(p);
            return PLX_ERR_CUDA;
        }
        g_status[dev] = p;
    }
    *status = g_status[dev];
    return PLX_OK;
}

int check_sizes(int B, int H, int T, int d, int dtype) {
    if (B < 1 || H < 1 || T < 1 || d < 1) return PLX_ERR_INVALID_ARG;
    if (dtype != PLX_FP32 && dtype != PLX_BF16) return PLX_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return PLX_ERR_UNSUPPORTED;
    const unsigned long long n = (unsigned long long)B * H * T * d;
    if (n >= (1ull << 31)) return PLX_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return PLX_ERR_UNSUPPORTED;
    return PLX_OK;
}

// Which family serves this call: 1 = SIMT, 2 = tensor core, <0 = error code.
int pick_family(int dtype) {
    const int path = g_path.load();
    if (path == PLX_PATH_SIMT) return 1;
    if (path == PLX_PATH_TC) return dtype == PLX_BF16 && plx::tc_available() ? 2 : -PLX_ERR_UNSUPPORTED;
    return (dtype == PLX_BF16 && plx::tc_available()) ? 2 : 1;
}

size_t fwd_ws_for(int fam, int B, int H, int T, int d) {
    return fam == 2 ? plx::tc_fwd_ws_bytes(B, H, T, d) : plx::simt_fwd_ws_bytes(B, H, T, d);
}
size_t bwd_ws_for(int fam, int B, int H, int T, int d) {
    return fam == 2 ? plx::tc_bwd_ws_bytes(B, H, T, d) : plx::simt_bwd_ws_bytes(B, H, T, d);
}

int fwd_common(const void* q, const void* k, const void* v, const float* P, void* out, float* lse,
               float* mu_k, void* ws, bool own_ws, int B, int H, int T, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, T, d, dtype);
    if (rc) return rc;
    if (!q || !k || !v || !P || !out || !lse || !mu_k) return PLX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(P) || !aligned16(out) ||
        !aligned16(lse) || !aligned16(mu_k))
        return PLX_ERR_INVALID_ARG;
    if (!own_ws && (!ws || ((uintptr_t)ws & 255u))) return PLX_ERR_INVALID_ARG;
    const int fam = pick_family(dtype);
    if (fam < 0) return -fam;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t bytes = fwd_ws_for(fam, B, H, T, d);
    if (own_ws && cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return PLX_ERR_CUDA;
    plx::FwdArgs a{q, k, v, P, out, lse, mu_k, ws, B, H, T, d, dtype, s, status};
    cudaError_t e = fam == 2 ? plx::tc_fwd(a) : plx::simt_fwd(a);
    if (own_ws) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}


// ------------------------------------------------------------- host step
// Heads [h0, h0 + nh) of a [B][H][rows] host tensor (row_bytes per head)
// against the chunk's own [B][nh][rows] device region.
cudaError_t copy_heads(void* host, void* dev, bool to_device, size_t row_bytes, int B, int H, int h0, int nh,
                       cudaStream_t s) {
    const size_t part = (size_t)nh * row_bytes, full = (size_t)H * row_bytes;
    char* h = (char*)host + (size_t)h0 * row_bytes;
    if (to_device) return cudaMemcpy2DAsync(dev, part, h, full, part, (size_t)B, cudaMemcpyHostToDevice, s);
    return cudaMemcpy2DAsync(h, full, dev, part, part, (size_t)B, cudaMemcpyDeviceToHost, s);
}

// True for host memory (pinned, registered or pageable), false for device or
// managed memory.
bool is_host(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}


// ------------------------------------------------------------- timing
struct Pending {
    int kid;
    cudaEvent_t a, b;
};
std::mutex g_tmu;
std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_timing{0};
std::vector<const char*> g_names;
std::vector<double> g_total_ms;
std::vector<long long> g_count;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_event_pool;
thread_local int t_kid = -1;
thread_local cudaEvent_t t_ev = nullptr;

int kernel_id(const char* name) {
    for (size_t i = 0; i < g_names.size(); i++)
        if (g_names[i] == name || std::strcmp(g_names[i], name) == 0) return (int)i;
    g_names.push_back(name);
    g_total_ms.push_back(0.0);
    g_count.push_back(0);
    return (int)g_names.size() - 1;
}

cudaEvent_t get_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

namespace plx {
void timing_begin(cudaStream_t s, const char* name) {
    g_launches.fetch_add(1);
    t_kid = -1;
    if (!g_timing.load()) return;
    std::lock_guard<std::mutex> lock(g_tmu);
    cudaEvent_t e = get_event();
    if (!e || cudaEventRecord(e, s) != cudaSuccess) {
        if (e) g_event_pool.push_back(e);
        return;
    }
    t_kid = kernel_id(name);
    t_ev = e;
}
void timing_end(cudaStream_t s) {
    if (t_kid < 0) return;
    std::lock_guard<std::mutex> lock(g_tmu);
    cudaEvent_t e = get_event();
    if (!e || cudaEventRecord(e, s) != cudaSuccess) {
        if (e) g_event_pool.push_back(e);
        g_event_pool.push_back(t_ev);
    } else {
        g_pending.push_back({t_kid, t_ev, e});
    }
    t_kid = -1;
}
int persistent_cta_cap() { return g_persist_cap.load(); }
}  // namespace plx

extern "C" {

unsigned long long parallax_launch_count(void) { return g_launches.load(); }

int parallax_timing_enable(int on) { return g_timing.exchange(on ? 1 : 0); }

int parallax_timing_collect(void) {
    std::lock_guard<std::mutex> lock(g_tmu);
    int rc = 0;
    for (const Pending& p : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess)
            rc = -PLX_ERR_CUDA;
        else {
            g_total_ms[p.kid] += ms;
            g_count[p.kid] += 1;
        }
        g_event_pool.push_back(p.a);
        g_event_pool.push_back(p.b);
    }
    g_pending.clear();
    return rc ? rc : (int)g_names.size();
}

int parallax_timing_get(int i, const char** name, double* total_ms, long long* launches) {
    std::lock_guard<std::mutex> lock(g_tmu);
    if (i < 0 || (size_t)i >= g_names.size()) return PLX_ERR_INVALID_ARG;
    if (name) *name = g_names[i];
    if (total_ms) *total_ms = g_total_ms[i];
    if (launches) *launches = g_count[i];
    return PLX_OK;
}

void parallax_timing_reset(void) {
    std::lock_guard<std::mutex> lock(g_tmu);
    for (size_t i = 0; i < g_names.size(); i++) {
        g_total_ms[i] = 0.0;
        g_count[i] = 0;
    }
}


int parallax_fwd(const void* q, const void* k, const void* v, const float* P, void* out, float* lse,
                 float* mu_k, int B, int H, int T, int d, int dtype, void* stream) {
    return fwd_common(q, k, v, P, out, lse, mu_k, nullptr, true, B, H, T, d, dtype, stream);
}

int parallax_fwd_ws(const void* q, const void* k, const void* v, const float* P, void* out, float* lse,
                    float* mu_k, void* workspace, int B, int H, int T, int d, int dtype, void* stream) {
    return fwd_common(q, k, v, P, out, lse, mu_k, workspace, false, B, H, T, d, dtype, stream);
}

size_t parallax_fwd_workspace_bytes(int B, int H, int T, int d, int dtype) {
    if (check_sizes(B, H, T, d, dtype)) return 0;
    const int fam = pick_family(dtype);
    if (fam < 0) return 0;
    return fwd_ws_for(fam, B, H, T, d);
}

size_t parallax_bwd_workspace_bytes(int B, int H, int T, int d, int dtype) {
    if (check_sizes(B, H, T, d, dtype)) return 0;
    const int fam = pick_family(dtype);
    if (fam < 0) return 0;
    return bwd_ws_for(fam, B, H, T, d);
}

int parallax_bwd(const void* q, const void* k, const void* v, const float* P, const float* lse,
                 const float* mu_k, const void* dout, void* dq, void* dk, void* dv, float* dP, void* workspace,
                 int B, int H, int T, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, T, d, dtype);
    if (rc) return rc;
    if (!q || !k || !v || !P || !lse || !mu_k || !dout || !dq || !dk || !dv || !dP)
        return PLX_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, P, lse, mu_k, dout, dq, dk, dv, dP};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PLX_ERR_INVALID_ARG;
    if (workspace && ((uintptr_t)workspace & 255u)) return PLX_ERR_INVALID_ARG;
    const int fam = pick_family(dtype);
    if (fam < 0) return -fam;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool own = workspace == nullptr;
    void* ws = workspace;
    if (own && cudaMallocAsync(&ws, bwd_ws_for(fam, B, H, T, d), s) != cudaSuccess) return PLX_ERR_CUDA;
    plx::BwdArgs a{q, k, v, P, lse, mu_k, dout, dq, dk, dv, dP, ws, B, H, T, d, dtype, s, status};
    cudaError_t e = fam == 2 ? plx::tc_bwd(a) : plx::simt_bwd(a);
    if (own) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

size_t parallax_fwd_bwd_workspace_bytes(int B, int H, int T, int d, int dtype) {
    if (check_sizes(B, H, T, d, dtype)) return 0;
    const int fam = pick_family(dtype);
    if (fam < 0) return 0;
    const size_t f = fwd_ws_for(fam, B, H, T, d), b = bwd_ws_for(fam, B, H, T, d);
    return f > b ? f : b;
}

int parallax_fwd_bwd(const void* q, const void* k, const void* v, const float* P, const void* dout, void* out,
                     float* lse, float* mu_k, void* dq, void* dk, void* dv, float* dP, void* workspace, int B, int H,
                     int T, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, T, d, dtype);
    if (rc) return rc;
    if (!q || !k || !v || !P || !dout || !out || !lse || !mu_k || !dq || !dk || !dv || !dP)
        return PLX_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, P, dout, out, lse, mu_k, dq, dk, dv, dP};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PLX_ERR_INVALID_ARG;
    if (workspace && ((uintptr_t)workspace & 255u)) return PLX_ERR_INVALID_ARG;
    const int fam = pick_family(dtype);
    if (fam < 0) return -fam;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool own = workspace == nullptr;
    void* ws = workspace;
    if (own && cudaMallocAsync(&ws, parallax_fwd_bwd_workspace_bytes(B, H, T, d, dtype), s) != cudaSuccess)
        return PLX_ERR_CUDA;
    plx::FwdArgs fa{q, k, v, P, out, lse, mu_k, ws, B, H, T, d, dtype, s, status};
    plx::BwdArgs ba{q, k, v, P, lse, mu_k, dout, dq, dk, dv, dP, ws, B, H, T, d, dtype, s, status};
    cudaError_t e;
    if (fam == 2) {
        e = plx::tc_fwd_bwd(fa, ba);
    } else {
        e = plx::simt_fwd(fa);
        if (e == cudaSuccess) e = plx::simt_bwd(ba);
    }
    if (own) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

size_t parallax_fwd_probe_workspace_bytes(int B, int H, int T, int d, int dtype) {
    if (check_sizes(B, H, T, d, dtype) || dtype != PLX_BF16 || !plx::tc_available()) return 0;
    return plx::tc_probe_ws_bytes(B, H, T, d);
}

int parallax_fwd_probe(const void* q, const void* k, const void* v, const void* rho, void* out, float* lse,
                       void* workspace, int B, int H, int T, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, T, d, dtype);
    if (rc) return rc;
    if (dtype != PLX_BF16 || !plx::tc_available()) return PLX_ERR_UNSUPPORTED;
    if (!q || !k || !v || !rho || !out || !lse) return PLX_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, rho, out, lse};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PLX_ERR_INVALID_ARG;
    if (workspace && ((uintptr_t)workspace & 255u)) return PLX_ERR_INVALID_ARG;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool own = workspace == nullptr;
    void* ws = workspace;
    if (own && cudaMallocAsync(&ws, plx::tc_probe_ws_bytes(B, H, T, d), s) != cudaSuccess) return PLX_ERR_CUDA;
    plx::ProbeArgs a{q, k, v, rho, out, lse, ws, B, H, T, d, dtype, s, status};
    cudaError_t e = plx::tc_probe(a);
    if (own) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

size_t parallax_decode_workspace_bytes(int B, int H, int Lmax, int d, int dtype) {
    if (check_sizes(B, H, Lmax, d, dtype)) return 0;
    return plx::decode_ws_bytes(B, H, Lmax, d);
}

int parallax_decode(const void* q, const void* k_cache, const void* v_cache, const int* lens, const float* P,
                    void* out, float* lse, void* workspace, int B, int H, int Lmax, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, Lmax, d, dtype);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !P || !out || !lse) return PLX_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k_cache, v_cache, P, out, lse};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PLX_ERR_INVALID_ARG;
    if (lens && ((uintptr_t)lens & 3u)) return PLX_ERR_INVALID_ARG;
    if (workspace && ((uintptr_t)workspace & 255u)) return PLX_ERR_INVALID_ARG;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool own = workspace == nullptr;
    void* ws = workspace;
    if (own && cudaMallocAsync(&ws, plx::decode_ws_bytes(B, H, Lmax, d), s) != cudaSuccess) return PLX_ERR_CUDA;
    plx::DecodeArgs a{q, k_cache, v_cache, lens, P, out, lse, ws, B, H, Lmax, d, dtype, s, status};
    cudaError_t e = plx::decode(a);
    if (own) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

size_t parallax_decode_probe_workspace_bytes(int B, int H, int Lmax, int d, int dtype) {
    if (check_sizes(B, H, Lmax, d, dtype) || dtype != PLX_BF16) return 0;
    return plx::decode_probe_ws_bytes(B, H, Lmax, d);
}

int parallax_decode_probe(const void* q, const void* k_cache, const void* v_cache, const int* lens, const void* rho,
                          void* out, float* lse, void* workspace, int B, int H, int Lmax, int d, int dtype,
                          void* stream) {
    int rc = check_sizes(B, H, Lmax, d, dtype);
    if (rc) return rc;
    if (dtype != PLX_BF16) return PLX_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !rho || !out || !lse) return PLX_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k_cache, v_cache, rho, out, lse};
    for (const void* p : ptrs)
        if (!aligned16(p)) return PLX_ERR_INVALID_ARG;
    if (lens && ((uintptr_t)lens & 3u)) return PLX_ERR_INVALID_ARG;
    if (workspace && ((uintptr_t)workspace & 255u)) return PLX_ERR_INVALID_ARG;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const bool own = workspace == nullptr;
    void* ws = workspace;
    if (own && cudaMallocAsync(&ws, plx::decode_probe_ws_bytes(B, H, Lmax, d), s) != cudaSuccess) return PLX_ERR_CUDA;
    plx::DecodeArgs a{q, k_cache, v_cache, lens, nullptr, out, lse, ws, B, H, Lmax, d, dtype, s, status, rho};
    cudaError_t e = plx::decode_probe(a);
    if (own) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    if (e == cudaErrorNotSupported) return PLX_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

int parallax_step_host(const void* q, const void* k, const void* v, const float* P, const void* dout, void* out,
                       float* lse, float* mu_k, void* dq, void* dk, void* dv, float* dP, int chunks, int B, int H,
                       int T, int d, int dtype, void* stream) {
    int rc = check_sizes(B, H, T, d, dtype);
    if (rc) return rc;
    if (!q || !k || !v || !P || !dout || !out || !dq || !dk || !dv || !dP) return PLX_ERR_INVALID_ARG;
    if (chunks < 0 || chunks > H) return PLX_ERR_INVALID_ARG;
    {
        const void* host_ptrs[] = {q, k, v, P, dout, out, dq, dk, dv, dP, lse, mu_k};
        for (const void* p : host_ptrs)
            if (p && !is_host(p)) return PLX_ERR_INVALID_ARG;
    }
    const int fam = pick_family(dtype);
    if (fam < 0) return -fam;
    unsigned* status = nullptr;
    rc = device_state(&status);
    if (rc) return rc;
    if (chunks == 0) chunks = H < 8 ? H : 8;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t es = dtype == PLX_BF16 ? 2 : 4;
    const size_t act_row = (size_t)T * d * es, f32_row = (size_t)T * d * 4, lse_row = (size_t)T * 4;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };

    // chunk c holds heads [h0[c], h0[c] + nh[c]); every tensor of a chunk starts 256-byte aligned
    enum { Q, K, V, DO, OUT, DQ, DK, DV, MU, LSE, NT_ };
    std::vector<int> h0(chunks), nh(chunks);
    std::vector<size_t> off((size_t)chunks * NT_);
    size_t total = 0;
    for (int c = 0, h = 0; c < chunks; c++) {
        nh[c] = H / chunks + (c < H % chunks ? 1 : 0);
        h0[c] = h;
        h += nh[c];
        for (int t = 0; t < NT_; t++) {
            const size_t row = t == MU ? f32_row : (t == LSE ? lse_row : act_row);
            off[(size_t)c * NT_ + t] = total;
            total += up((size_t)B * nh[c] * row);
        }
    }
    const size_t hmax = (size_t)(H + chunks - 1) / chunks;
    const size_t pd_bytes = (size_t)H * d * d * 4;
    const size_t o_P = total, o_dP = o_P + up(pd_bytes), o_ws = o_dP + up(pd_bytes);
    size_t ws_bytes = fwd_ws_for(fam, B, (int)hmax, T, d);
    const size_t bw = bwd_ws_for(fam, B, (int)hmax, T, d);
    if (bw > ws_bytes) ws_bytes = bw;
    total = o_ws + up(ws_bytes);

    char* base = nullptr;
    if (cudaMallocAsync((void**)&base, total, s) != cudaSuccess) return PLX_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess && x != cudaSuccess) e = x;
        return e == cudaSuccess;
    };
    cudaStream_t s_in = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> ev((size_t)2 * chunks + 2, nullptr);
    chk(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking));
    chk(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking));
    for (auto& x : ev) chk(cudaEventCreateWithFlags(&x, cudaEventDisableTiming));
    cudaEvent_t e_alloc = ev[0], e_end = ev[1];
    cudaEvent_t* e_in = ev.data() + 2;
    cudaEvent_t* e_comp = ev.data() + 2 + chunks;
    auto dev = [&](int c, int t) { return (void*)(base + off[(size_t)c * NT_ + t]); };
    float* Pd = (float*)(base + o_P);
    float* dPd = (float*)(base + o_dP);
    void* ws = base + o_ws;

    // copy engine in: P, then every chunk's inputs back to back
    if (chk(cudaEventRecord(e_alloc, s)) && chk(cudaStreamWaitEvent(s_in, e_alloc, 0)) &&
        chk(cudaMemcpyAsync(Pd, P, pd_bytes, cudaMemcpyHostToDevice, s_in))) {
        const void* src[4] = {q, k, v, dout};
        for (int c = 0; c < chunks && e == cudaSuccess; c++) {
            for (int t = Q; t <= DO; t++)
                if (!chk(copy_heads((void*)src[t], dev(c, t), true, act_row, B, H, h0[c], nh[c], s_in))) break;
            chk(cudaEventRecord(e_in[c], s_in));
        }
    }
    // compute on the caller's stream, chunk by chunk; copy engine out behind it
    for (int c = 0; c < chunks && e == cudaSuccess; c++) {
        if (!chk(cudaStreamWaitEvent(s, e_in[c], 0))) break;
        const float* Pc = Pd + (size_t)h0[c] * d * d;
        plx::FwdArgs fa{dev(c, Q), dev(c, K), dev(c, V), Pc, dev(c, OUT), (float*)dev(c, LSE), (float*)dev(c, MU),
                        ws, B, nh[c], T, d, dtype, s, status};
        plx::BwdArgs ba{dev(c, Q), dev(c, K), dev(c, V), Pc, (const float*)dev(c, LSE), (const float*)dev(c, MU),
                        dev(c, DO), dev(c, DQ), dev(c, DK), dev(c, DV), dPd + (size_t)h0[c] * d * d, ws,
                        B, nh[c], T, d, dtype, s, status};
        if (fam == 2) {  // one workspace: the backward reuses the forward's f16 copies
            if (!chk(plx::tc_fwd_bwd(fa, ba))) break;
        } else {
            if (!chk(plx::simt_fwd(fa)) || !chk(plx::simt_bwd(ba))) break;
        }
        if (!chk(cudaEventRecord(e_comp[c], s)) || !chk(cudaStreamWaitEvent(s_out, e_comp[c], 0))) break;
        void* dst[4] = {out, dq, dk, dv};
        for (int t = OUT; t <= DV; t++)
            if (!chk(copy_heads(dst[t - OUT], dev(c, t), false, act_row, B, H, h0[c], nh[c], s_out))) break;
        if (mu_k) chk(copy_heads(mu_k, dev(c, MU), false, f32_row, B, H, h0[c], nh[c], s_out));
        if (lse) chk(copy_heads(lse, dev(c, LSE), false, lse_row, B, H, h0[c], nh[c], s_out));
        chk(cudaMemcpyAsync(dP + (size_t)h0[c] * d * d, dPd + (size_t)h0[c] * d * d, (size_t)nh[c] * d * d * 4,
                            cudaMemcpyDeviceToHost, s_out));
    }
    // the caller's stream orders after both copy streams, then frees the memory
    cudaError_t e2 = cudaSuccess;
    if (s_in && s_out && ev[0] && ev[1]) {
        cudaError_t a = cudaEventRecord(e_alloc, s_in);
        cudaError_t b = a == cudaSuccess ? cudaStreamWaitEvent(s, e_alloc, 0) : a;
        cudaError_t c2 = cudaEventRecord(e_end, s_out);
        cudaError_t d2 = c2 == cudaSuccess ? cudaStreamWaitEvent(s, e_end, 0) : c2;
        e2 = b != cudaSuccess ? b : d2;
    }
    if (e == cudaSuccess) e = e2;
    if (e2 == cudaSuccess) {
        cudaError_t f = cudaFreeAsync(base, s);
        if (e == cudaSuccess) e = f;
    } else {
        // the copy streams could not be joined: wait for them before freeing
        if (s_in) cudaStreamSynchronize(s_in);
        if (s_out) cudaStreamSynchronize(s_out);
        cudaStreamSynchronize(s);
        cudaFree(base);
    }
    for (auto& x : ev)
        if (x) cudaEventDestroy(x);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
    return e == cudaSuccess ? PLX_OK : PLX_ERR_CUDA;
}

int parallax_last_device_error(void* stream, unsigned* detail) {
    if (detail) *detail = 0;
    unsigned* status = nullptr;
    int rc = device_state(&status);
    if (rc) return rc;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return PLX_ERR_CUDA;
    unsigned word[4] = {0, 0, 0, 0};
    if (cudaMemcpy(word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return PLX_ERR_CUDA;
    if (word[0] == 0) return PLX_OK;
    if (detail) *detail = word[1];
    // clear the flag and the detail; word [2] (the wait limit) stays
    if (cudaMemset(status, 0, 2 * sizeof(unsigned)) != cudaSuccess) return PLX_ERR_CUDA;
    return PLX_ERR_TIMEOUT;
}

int parallax_set_wait_limit(long long cycles) {
    unsigned* status = nullptr;
    int rc = device_state(&status);
    if (rc) return rc;
    // word [2] of the status word, in units of 64 cycles (0 = the default)
    unsigned units = 0;
    if (cycles > 0) {
        const long long u = (cycles + 63) / 64;
        units = u > 0xFFFFFFFFll ? 0xFFFFFFFFu : (unsigned)u;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return PLX_ERR_CUDA;
    if (cudaMemcpy(status + 2, &units, sizeof(units), cudaMemcpyHostToDevice) != cudaSuccess) return PLX_ERR_CUDA;
    return PLX_OK;
}

int parallax_set_path(int path) {
    if (path != PLX_PATH_AUTO && path != PLX_PATH_SIMT && path != PLX_PATH_TC) return -1;
    return g_path.exchange(path);
}

int parallax_set_persistent_ctas(int ctas) {
    if (ctas < 0) return -1;
    return g_persist_cap.exchange(ctas);
}

const char* parallax_strerror(int code) {
    switch (code) {
        case PLX_OK: return "success";
        case PLX_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size)";
        case PLX_ERR_UNSUPPORTED: return "unsupported configuration (head dim, dtype, path or device)";
        case PLX_ERR_CUDA: return "CUDA runtime error";
        case PLX_ERR_TIMEOUT: return "device-side wait timed out";
        case PLX_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of parallax_fwd_noalloc (32 MiB)";
        default: return "unknown status code";
    }
}

}  // extern "C"
