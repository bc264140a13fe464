// attn_noalloc.cu - backward pass for callers that cannot allocate device memory.
//
// attn_bwd needs two workspaces besides its inputs and outputs: the row terms
// D [B,H,N] and the fp32 dQ accumulator [B,H,N,d].  Some callers cannot
// provide them: plug-ins whose host framework owns every allocation and offers
// none to them, and real-time programs that must not allocate after start-up.  attn_bwd_noalloc keeps both workspaces in one
// file-scope device array of fixed size instead, so the caller passes only
// its inputs and outputs.
//
// The array occupies kNoallocScratchFloats * 4 bytes (16 MiB) on every GPU
// that loads this library, for as long as the library stays loaded.
#include <mutex>

#include "../../include/attn.h"
#include "attn_common.cuh"

namespace attn {
namespace {

constexpr long long kNoallocScratchFloats = 4ll * 1024 * 1024;  // 16 MiB of fp32

// D occupies the first round_up(B*H*N, 64) floats (keeping dq_accum 256-byte
// aligned), dq_accum the next B*H*N*d floats.
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array for the current device.  In host code the
// array's name only stands in for the symbol; the address the kernels need
// comes from cudaGetSymbolAddress, called once per device with that device
// current.
int scratch_for_current_device(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ready[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return ATTN_ERR_UNSUPPORTED_DEVICE;
        }
        g_scratch_ptr[dev] = static_cast<float*>(p);
        g_scratch_ready[dev] = true;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

int noalloc_impl(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                 float scale, void* stream) {
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    const long long rows = static_cast<long long>(B) * H * N;
    const long long d_floats = (rows + 63) / 64 * 64;
    if (d_floats + rows * d > kNoallocScratchFloats) return ATTN_ERR_SCRATCH_TOO_SMALL;
    float* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    float* D = scratch;
    float* dq_accum = scratch + d_floats;
    // The preprocess overwrites D and zeroes dq_accum, so what an earlier call
    // left in the array does not matter.
    rc = attn_bwd_preprocess(q, k, v, dO, lse, D, dq_accum, B, H, N, d, causal, scale, stream);
    if (rc) return rc;
    return attn_bwd(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, N, d, causal, scale, stream);
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                     void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                     float scale, void* stream) {
    return attn::noalloc_impl(q, k, v, dO, lse, dq, dk, dv, B, H, N, d, causal, scale, stream);
}

}  // extern "C"
