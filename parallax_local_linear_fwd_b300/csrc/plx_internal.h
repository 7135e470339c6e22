// Internal interface between the C ABI layer (plx_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace plx {

// Kernel identifiers used in the watchdog word (id << 16 | wait site).
enum KernelId : unsigned {
    KID_TC_PASS1 = 1,
    KID_TC_PASS2 = 2,
    KID_TC_BWD_B1 = 3,
    KID_TC_BWD_B3 = 4,
    KID_TC_PROJ = 5,
    KID_TC_PROBE = 6,
    KID_TC_BWD_B2 = 7,
    KID_DECODE = 8,
};

struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* P;
    void* out;
    float* lse;
    float* mu_k;
    void* ws;  // workspace, 256-byte aligned, fwd_ws_bytes() long
    int B, H, T, d, dtype;
    cudaStream_t stream;
    unsigned* status;  // device watchdog word
};

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* P;
    const float* lse;
    const float* mu_k;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    float* dP;
    void* ws;
    int B, H, T, d, dtype;
    cudaStream_t stream;
    unsigned* status;
};

struct DecodeArgs {
    const void* q;     // [B,H,d] one new query per (sequence, head)
    const void* k;     // [B,H,Lmax,d] key cache
    const void* v;     // [B,H,Lmax,d] value cache
    const int* lens;   // [B] valid keys per sequence (device), or nullptr = Lmax
    const float* P;    // [H,d,d] (the committed probe form)
    void* out;         // [B,H,d]
    float* lse;        // [B,H]
    void* ws;          // decode_ws_bytes() or decode_probe_ws_bytes()
    int B, H, Lmax, d, dtype;
    cudaStream_t stream;
    unsigned* status;  // device watchdog word
    const void* rho = nullptr;  // [B,H,d] the given probe (decode_probe), same dtype as q
};

struct ProbeArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* rho;  // [B,H,T,d] the given probe
    void* out;
    float* lse;
    void* ws;
    int B, H, T, d, dtype;
    cudaStream_t stream;
    unsigned* status;
};

// Launch accounting / timing hooks (plx_api.cu).  Bracket every launch:
//   timing_begin(stream, "name"); kernel<<<...>>>(...); timing_end(stream);
void timing_begin(cudaStream_t s, const char* name);
void timing_end(cudaStream_t s);

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// SIMT (FFMA) family: any dtype, d in {64,128}.
size_t simt_fwd_ws_bytes(int B, int H, int T, int d);
size_t simt_bwd_ws_bytes(int B, int H, int T, int d);
cudaError_t simt_fwd(const FwdArgs& a);
cudaError_t simt_bwd(const BwdArgs& a);
// The SIMT backward after its first kernel (B2, dP, B3, dq cast), reading
// R and ebar from the SIMT workspace; lets another family supply B1.
cudaError_t simt_bwd_after_b1(const BwdArgs& a);
void simt_bwd_ws_b1_outputs(void* ws, int B, int H, int T, int d, float** R, float** ebar);
// dP_h = sum_{b,t} du delta^T (delta = q - mu_k) by the SIMT two-stage
// fixed-order reduction; `partial` holds simt_dp_partial_bytes() bytes.
size_t simt_dp_partial_bytes(int B, int H, int T, int d);
cudaError_t simt_dP(const void* q, const float* mu_k, const float* du, float* partial, float* dP, int B, int H,
                    int T, int d, int dtype, cudaStream_t stream);

// Decode (SIMT, HBM-bound split-KV), any dtype, d in {64,128}.
size_t decode_ws_bytes(int B, int H, int Lmax, int d);
cudaError_t decode(const DecodeArgs& a);

// Tensor-core (tcgen05) family: bf16, d in {64,128}.
bool tc_available();
// A 16-bit [BH][T][D] tensor viewed as 3-D (D, T, BH) with a box of 64 x rows
// x 1 and the 128-byte swizzle (rows past T read as zero); false on failure.
bool tc_make_map(void* map, const void* base, int D, int T, int BH, int rows);
// One-pass decode for bf16 caches (tensor-core M = V^T diag(p) K per chunk).
size_t decode_tc_ws_bytes(int B, int H, int Lmax, int d);
cudaError_t decode_tc(const DecodeArgs& a);
size_t decode_probe_ws_bytes(int B, int H, int Lmax, int d);
cudaError_t decode_probe(const DecodeArgs& a);
size_t tc_fwd_ws_bytes(int B, int H, int T, int d);
size_t tc_bwd_ws_bytes(int B, int H, int T, int d);
// CTAs the persistent kernels (pass 2 at d = 128, B2 at d = 64) launch at
// most: their own count per SM when 0 (parallax_set_persistent_ctas).
int persistent_cta_cap();

cudaError_t tc_fwd(const FwdArgs& a);
cudaError_t tc_bwd(const BwdArgs& a);
cudaError_t tc_fwd_bwd(const FwdArgs& f, const BwdArgs& b);
// One-pass forward with a given probe (o = o^SA - Sigma_KV rho), bf16.
size_t tc_probe_ws_bytes(int B, int H, int T, int d);
cudaError_t tc_probe(const ProbeArgs& a);

}  // namespace plx
