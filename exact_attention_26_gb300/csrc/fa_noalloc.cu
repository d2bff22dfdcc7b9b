// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a caller-provided workspace (the per-row D_i and base-2 L vectors).
// Some callers cannot obtain one: a host that reserves all device memory up front
// in its own pool and forbids side allocations, or a latency-critical loop where a
// cudaMalloc (which may synchronise the device) is not acceptable.  This entry
// point takes the same inputs and outputs as fa_bwd but uses a fixed scratch array
// compiled into the library instead, so it allocates nothing.
//
// The scratch is a file-scope device array of FA_NOALLOC_SCRATCH_BYTES (8 MiB); every GPU
// that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is fetched
// with cudaGetSymbolAddress once per device, on the first call made while that
// device is current, and cached.
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;  // 8 MiB + 256 bytes

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxScratchDevices] = {};

int scratch_of_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices)
        return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
            return FA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dout, float *dq, float *dk, float *dv,
                              int B, int H, int N, int d, int causal, float scale, void *stream) {
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    if (need == 0)  // invalid sizes or head dimension: let fa_bwd report which
        return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, nullptr, 0,
                      stream);
    if (need > fa::kScratchBytes) return FA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int rc = fa::scratch_of_current_device(&scratch);
    if (rc != FA_OK) return rc;
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, scratch,
                  fa::kScratchBytes, stream);
}
