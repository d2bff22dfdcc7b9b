// Unit-rate probes: the per-SM issue rate of the two units the attention kernels
// lean on, measured on the running GPU with clock64 stamps, one CTA per SM.
//
//   * dense bf16 tcgen05.mma (kind::f16, M = 128, fp32 accumulate) at N = 256 (the
//     widest shape, the tensor core's peak) and N = 64 (the shape of the backward's
//     S^T, dP^T and dQ^T products at d = 128);
//   * MUFU ex2.approx.f32, the exponential of the online softmax.
//
// Multiplied by the SM count and the SM clock, the first gives the clock-derived
// tensor peak beside the measured GEMM peak, the last the exponential ceiling of
// the softmax (one ex2 per score element).  Operands are zero: the tensor core's
// rate does not depend on the data.
#include <algorithm>
#include <vector>

#include "fa_internal.h"
#include "fa_probe.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// A (128 rows x 128 B) at 0, B (256 rows x 128 B) at 16 KB, mbarrier at 48 KB.
// The launch asks for kProbeSmem so that no second CTA fits on an SM.
constexpr uint32_t kProbeSmem = 120 * 1024;
constexpr int kMmaPerTile = 4;  // K = 64 bf16 per 128-byte row, 16 per instruction

template <int N>
__global__ void __launch_bounds__(128, 1)
    fa_probe_mma_kernel(int iters, unsigned long long *cycles, int *status,
                        unsigned long long limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms: 1024-B aligned
    uint8_t *g = smem_raw + (base - raw);
    for (int i = threadIdx.x; i < (48 * 1024) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(g)[i] = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t bar = base + 48 * 1024;
    uint32_t *slot = reinterpret_cast<uint32_t *>(g + 48 * 1024 + 64);
    int *abort_flag = reinterpret_cast<int *>(g + 48 * 1024 + 128);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();  // the zeroed tiles are read by the tensor core
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x < 32) {
        const Guard gd{status, abort_flag, limit_ns};
        constexpr uint32_t idesc = idesc_bf16_f32(128, N, false, false);
        const uint64_t da = sdesc_sw128(base, 16, 1024);
        const uint64_t db = sdesc_sw128(base + 16 * 1024, 16, 1024);
        // one tile to warm the pipe, then the timed run
#pragma unroll
        for (int k = 0; k < kMmaPerTile; ++k)
            mma_ss_elect(tmem, desc_add(da, 32 * k), desc_add(db, 32 * k), idesc, k > 0);
        tc_commit_elect(bar);
        bool ok = mbar_wait_warp(bar, 0, gd, SITE_PROBE);
        const long long t0 = clock64();
        if (ok) {
            for (int i = 0; i < iters; ++i) {
#pragma unroll
                for (int k = 0; k < kMmaPerTile; ++k)
                    mma_ss_elect(tmem, desc_add(da, 32 * k), desc_add(db, 32 * k), idesc, 1u);
            }
            tc_commit_elect(bar);
            ok = mbar_wait_warp(bar, 1, gd, SITE_PROBE);
        }
        const long long t1 = clock64();
        if (threadIdx.x == 0) cycles[blockIdx.x] = ok ? (unsigned long long)(t1 - t0) : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

constexpr int kEx2Chains = 8;  // independent dependency chains per thread

__global__ void __launch_bounds__(1024, 1)
    fa_probe_ex2_kernel(int iters, float *sink, unsigned long long *cycles) {
    float x[kEx2Chains];
#pragma unroll
    for (int k = 0; k < kEx2Chains; ++k) x[k] = -1e-3f * (float)(threadIdx.x + k);
    __syncthreads();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kEx2Chains; ++k) x[k] = -ex2(x[k]);  // stays in (-1, 0)
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kEx2Chains; ++k) s += x[k];
    if (s == 1.0f) sink[0] = s;  // never true; keeps the chains live
    if (threadIdx.x == 0) cycles[blockIdx.x] = (unsigned long long)(t1 - t0);
}

// Streaming read: each thread XORs 16-byte words of the buffer into a register,
// L1 not allocated; nothing is written unless the XOR equals a value it never
// takes in practice (that keeps the loads live).
__global__ void __launch_bounds__(512)
    fa_probe_read_kernel(const uint4 *__restrict__ p, size_t n16, unsigned *sink) {
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
        uint4 w;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "l"(p + i));
        acc.x ^= w.x;
        acc.y ^= w.y;
        acc.z ^= w.z;
        acc.w ^= w.w;
    }
    if ((acc.x ^ acc.y ^ acc.z ^ acc.w) == 0x9e3779b9u) sink[0] = acc.x;
}

}  // namespace

// Per-CTA clock64 intervals of the three probes, module globals (the library
// allocates no device memory per call).
constexpr int kProbeMaxSms = 1024;
__device__ unsigned long long g_probe_cycles[3 * kProbeMaxSms];
__device__ float g_probe_sink[1];

__device__ unsigned g_probe_read_sink[1];

int run_read_probe(int num_sms, const void *buf, size_t bytes, int iters, cudaStream_t stream,
                   double *gbs) {
    void *sink = nullptr;
    if (cudaGetSymbolAddress(&sink, g_probe_read_sink) != cudaSuccess) return FA_ERR_CUDA;
    const uint4 *p = static_cast<const uint4 *>(buf);
    const size_t n16 = bytes / 16;
    const unsigned grid = (unsigned)num_sms * 4;
    fa_probe_read_kernel<<<grid, 512, 0, stream>>>(p, n16, static_cast<unsigned *>(sink));
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
        if (a) cudaEventDestroy(a);
        return FA_ERR_CUDA;
    }
    int rc = FA_OK;
    float ms = 0.f;
    if (cudaEventRecord(a, stream) != cudaSuccess) rc = FA_ERR_CUDA;
    for (int i = 0; rc == FA_OK && i < iters; ++i)
        fa_probe_read_kernel<<<grid, 512, 0, stream>>>(p, n16, static_cast<unsigned *>(sink));
    if (rc == FA_OK && (cudaGetLastError() != cudaSuccess || cudaEventRecord(b, stream) != cudaSuccess ||
                        cudaEventSynchronize(b) != cudaSuccess ||
                        cudaEventElapsedTime(&ms, a, b) != cudaSuccess || ms <= 0.f))
        rc = FA_ERR_CUDA;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (rc == FA_OK) *gbs = (double)n16 * 16.0 * iters / (ms * 1e-3) / 1e9;
    return rc;
}

int run_unit_probes(int num_sms, int iters, int *status, cudaStream_t stream, double *rates) {
    if (num_sms < 1 || num_sms > kProbeMaxSms) return FA_ERR_UNSUPPORTED;
    void *cyc = nullptr, *sink = nullptr;
    if (cudaGetSymbolAddress(&cyc, g_probe_cycles) != cudaSuccess ||
        cudaGetSymbolAddress(&sink, g_probe_sink) != cudaSuccess)
        return FA_ERR_CUDA;
    unsigned long long *cycles = static_cast<unsigned long long *>(cyc);
    auto k256 = fa_probe_mma_kernel<256>;
    auto k64 = fa_probe_mma_kernel<64>;
    for (auto kern : {k256, k64})
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kProbeSmem) != cudaSuccess)
            return FA_ERR_CUDA;
    if (cudaFuncSetAttribute(fa_probe_ex2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kProbeSmem) != cudaSuccess)
        return FA_ERR_CUDA;
    k256<<<num_sms, 128, kProbeSmem, stream>>>(iters, cycles, status, kWaitLimitNs);
    k64<<<num_sms, 128, kProbeSmem, stream>>>(iters, cycles + num_sms, status, kWaitLimitNs);
    fa_probe_ex2_kernel<<<num_sms, 1024, kProbeSmem, stream>>>(
        4 * iters, static_cast<float *>(sink), cycles + 2 * num_sms);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    std::vector<unsigned long long> host(3 * (size_t)num_sms);
    if (cudaMemcpy(host.data(), cycles, host.size() * sizeof(unsigned long long),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    for (int which = 0; which < 3; ++which) {
        std::vector<unsigned long long> c(host.begin() + which * num_sms,
                                          host.begin() + (which + 1) * num_sms);
        for (unsigned long long x : c)
            if (x == 0) return FA_ERR_TIMEOUT;  // an MMA completion wait gave up
        std::nth_element(c.begin(), c.begin() + num_sms / 2, c.end());
        const double n = which == 0 ? 256.0 : 64.0;
        const double work = which < 2 ? 2.0 * 128.0 * n * 16.0 * kMmaPerTile * iters
                                      : 1024.0 * kEx2Chains * 4.0 * iters;
        rates[which] = work / (double)c[num_sms / 2];
    }
    return FA_OK;
}

}  // namespace fa
