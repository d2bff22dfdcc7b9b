// Host side of the C ABI declared in include/fa.h: argument validation, the
// per-device cache, TMA tensor-map encoding, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_internal.h"
#include "fa_probe.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// Device status record written by the kernels' bounded waits: [0] error code,
// [1] wait site of the first error.  One copy per device (module global).
__device__ int g_status[2];

constexpr int kMaxDevices = 64;

struct DeviceCache {
    bool ready = false;
    int num_sms = 0;
    int *status = nullptr;
};

std::mutex g_mutex;
DeviceCache g_devices[kMaxDevices];

int current_device(DeviceCache **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceCache &dc = g_devices[dev];
    if (!dc.ready) {
        int sms = 0;
        void *status = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        if (cudaGetSymbolAddress(&status, g_status) != cudaSuccess) return FA_ERR_CUDA;
        dc.num_sms = sms;
        dc.status = static_cast<int *>(status);
        dc.ready = true;
    }
    *out = &dc;
    return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 3-D tiled map (unit element strides, no interleave, 256-byte L2 promotion, zero
// fill past the bounds).  A map is a pure function of its arguments, so the last
// few encodings are kept and reused: calls that repeat a tensor and shape (every
// step of a training loop, every decode step) skip the driver call.  Keys hold the
// address, so a freed and reallocated tensor at the same address with the same
// shape gets the identical map.
int encode_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr, const cuuint64_t (&dims)[3],
              const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
    struct Entry {
        const void *ptr;
        int dtype, swizzle;
        cuuint64_t dims[3], strides[2];
        cuuint32_t box[3];
        CUtensorMap map;
    };
    constexpr int kEntries = 32;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    static std::mutex m;
    auto same = [&](const Entry &e) {
        return e.ptr == ptr && e.dtype == (int)dtype && e.swizzle == (int)swizzle &&
               e.dims[0] == dims[0] && e.dims[1] == dims[1] && e.dims[2] == dims[2] &&
               e.strides[0] == strides[0] && e.strides[1] == strides[1] && e.box[0] == box[0] &&
               e.box[1] == box[1] && e.box[2] == box[2];
    };
    {
        std::lock_guard<std::mutex> lock(m);
        for (int i = 0; i < used; ++i)
            if (same(cache[i])) {
                *map = cache[i].map;
                return FA_OK;
            }
    }
    auto enc = encode_tiled();
    if (!enc) return FA_ERR_CUDA;
    cuuint64_t d3[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t s2[2] = {strides[0], strides[1]};
    cuuint32_t b3[3] = {box[0], box[1], box[2]};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(ptr), d3, s2, b3, elem_strides,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(m);
    Entry &e = cache[next];
    e.ptr = ptr;
    e.dtype = (int)dtype;
    e.swizzle = (int)swizzle;
    for (int i = 0; i < 3; ++i) e.dims[i] = dims[i], e.box[i] = box[i];
    for (int i = 0; i < 2; ++i) e.strides[i] = strides[i];
    e.map = *map;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return FA_OK;
}

// 3-D map over a contiguous bf16 [BH][N][d] tensor: x = column within the head
// dimension, y = row, z = (batch, head).  Boxes are 64 columns (128 bytes, one
// swizzle span) by `box_rows` rows; rows past N read as zeros.
int make_bhnd_map(CUtensorMap *map, const void *ptr, int BH, int N, int d, int box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a packed token-major bf16 [T][heads][d] tensor: x = column, y = head,
// z = token.  A box of 64 columns x 1 head x `box_rows` tokens lands in shared
// memory as [box_rows][64], like a box of make_bhnd_map; tokens past T read as zeros.
int make_thd_map(CUtensorMap *map, const void *ptr, int T, int heads, int d, int box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * (cuuint64_t)d * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a contiguous fp32 tensor (the dQ output) for tiled bulk adds,
// unswizzled: dims (d, n1, n2) with row pitch d and plane pitch n1 * d elements,
// boxes of 32 columns x box1 x box2, which are row-major 128-byte rows in shared
// memory.  Fixed layout [BH][N][d]: (d, N, BH), box (32, 32, 1); packed
// token-major [T][heads][d]: (d, heads, T), box (32, 1, 32).
int make_f32_map(CUtensorMap *map, const void *ptr, int d, int n1, int n2, int box1, int box2) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n1, (cuuint64_t)n2};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)n1 * (cuuint64_t)d * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)box1, (cuuint32_t)box2};
    return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 3-D map over bytes (e4m3 codes): dims x (innermost), y, z with the given row and
// plane pitches (multiples of 16 bytes); boxes of box_x (128: one swizzle span) by
// box_y by 1; elements past the dims read as zeros.
int make_u8_map(CUtensorMap *map, const void *ptr, uint64_t nx, uint64_t ny, uint64_t nz,
                uint64_t pitch_y, uint64_t pitch_z, uint32_t box_x, uint32_t box_y) {
    const cuuint64_t dims[3] = {(cuuint64_t)nx, (cuuint64_t)ny, (cuuint64_t)nz};
    const cuuint64_t strides[2] = {(cuuint64_t)pitch_y, (cuuint64_t)pitch_z};
    const cuuint32_t box[3] = {box_x, box_y, 1};
    return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_sizes(int B, int H, int N, int d, bool fwd) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if ((long long)B * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
    if (fwd) {
        if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    } else {
        if (d != 64 && d != 96 && d != 128) return FA_ERR_UNSUPPORTED;
    }
    return FA_OK;
}

int check_scale(float scale) {
    return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

constexpr float kLog2e = 1.4426950408889634074f;

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// One warp waits, through the same bounded wait the attention kernels use, on an
// mbarrier that nothing ever arrives on; the wait gives up after `limit_ns`,
// records FA_ERR_TIMEOUT in the status word and the kernel returns.
__global__ void __launch_bounds__(32) fa_wait_selftest_kernel(int *status,
                                                             unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const Guard g{status, &abort_flag, limit_ns};
    mbar_wait_warp(smem_u32(&bar), 0, g, SITE_SELFTEST);
}

}  // namespace

namespace {
// Kernels whose dynamic shared memory limit has been raised, per device.
struct SmemAttr {
    const void *kernel;
    int device, bytes;
};
std::mutex g_attr_mutex;
SmemAttr g_attr[256];
int g_attr_count = 0;
}  // namespace

int ensure_smem_attr(const void *kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    for (int i = 0; i < g_attr_count; ++i)
        if (g_attr[i].kernel == kernel && g_attr[i].device == dev && g_attr[i].bytes >= bytes)
            return FA_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    if (g_attr_count < 256) g_attr[g_attr_count++] = {kernel, dev, bytes};
    return FA_OK;
}

int kernel_num_regs(const void *kernel) {
    static std::mutex m;
    static const void *keys[64];
    static int vals[64];
    static int n = 0;
    std::lock_guard<std::mutex> lock(m);
    for (int i = 0; i < n; ++i)
        if (keys[i] == kernel) return vals[i];
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess) return -1;
    if (n < 64) {
        keys[n] = kernel;
        vals[n++] = a.numRegs;
    }
    return a.numRegs;
}

// Keys per K/V tile of the one-tile forward kernel (the one that cuts key ranges).
int fwd_block_n(int d) { return d == 256 ? 64 : 128; }

}  // namespace fa

using namespace fa;

namespace fa {
namespace {
// Query heads per key/value head, or 0 if Hkv does not divide H.
int gqa_group(int H, int Hkv) {
    if (Hkv < 1 || Hkv > H || H % Hkv != 0) return 0;
    return H / Hkv;
}
}  // namespace
}  // namespace fa

namespace fa {
namespace {
// Chunk (K/V tiles; 0: no cut), chunks of the longest key range and workspace bytes
// of a forward with cut key ranges, for the current device.
struct FwdSplit {
    int chunk, s_max;
    const FwdSegPlan *seg;  // the balanced plan, when the library chose one
    size_t bytes, l_offset;
};
int fwd_split_plan(int B, int H, int N, int d, int causal, int kv_chunk_keys, FwdSplit *out) {
    DeviceCache *dc = nullptr;
    const int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    const int bn = fwd_block_n(d);
    const int forced = kv_chunk_keys > 0 ? (kv_chunk_keys + bn - 1) / bn : 0;
    FwdSplit s{};
    // automatic: a balanced plan first, else even chunks or no cut
    s.seg = forced > 0 ? nullptr : fwd_seg_plan(d, B * H, N, causal, dc->num_sms);
    s.chunk = s.seg ? 0 : fwd_split_chunk(d, B * H, N, causal, dc->num_sms, forced);
    if (s.chunk > 0 || s.seg) {
        const int n_kv = (N + bn - 1) / bn;
        s.s_max = s.seg ? s.seg->s_max : (n_kv + s.chunk - 1) / s.chunk;
        const size_t rows = (size_t)B * H * N * s.s_max;
        s.l_offset = round_up(rows * d * sizeof(float), 256);
        s.bytes = s.l_offset + round_up(rows * sizeof(float), 256);
    }
    *out = s;
    return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" int fa_fwd_split_segments(int B, int H, int N, int d, int causal, int num_sms,
                                     int *out, int cap) {
    if (check_sizes(B, H, N, d, true) != FA_OK || num_sms < 1 || cap < 0 || (cap > 0 && !out))
        return FA_ERR_INVALID_ARG;
    const FwdSegPlan *plan = fwd_seg_plan(d, B * H, N, causal ? 1 : 0, num_sms);
    if (!plan) return 0;
    for (int c = 0; c < plan->tab.n_cta; ++c)
        for (int i = plan->tab.start[c]; i < plan->tab.start[c + 1] && i < cap; ++i) {
            const uint32_t w0 = plan->tab.seg[i][0], w1 = plan->tab.seg[i][1];
            int *e = out + 7 * i;
            e[0] = (int)(w0 & 0xffffu);
            e[1] = (int)(w0 >> 16);
            e[2] = (int)(w1 & 0xfffu);
            e[3] = (int)((w1 >> 12) & 0xfffu);
            e[4] = (int)((w1 >> 24) & 0xfu);
            e[5] = (int)(w1 >> 28);
            e[6] = c;
        }
    return plan->n_seg;
}

extern "C" size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal, int kv_chunk) {
    if (check_sizes(B, H, N, d, true) != FA_OK || kv_chunk < 0) return 0;
    FwdSplit s{};
    if (fwd_split_plan(B, H, N, d, causal, kv_chunk, &s) != FA_OK) return 0;
    return s.bytes;
}

extern "C" int fa_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int H, int Hkv, int N, int d, int causal, float scale, int kv_chunk,
                         void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !o || !lse || kv_chunk < 0) return FA_ERR_INVALID_ARG;
    int rc = check_sizes(B, H, N, d, true);
    if (rc != FA_OK) return rc;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    if ((rc = check_scale(scale)) != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;
    FwdSplit sp{};
    if ((rc = fwd_split_plan(B, H, N, d, causal, kv_chunk, &sp)) != FA_OK) return rc;
    if (sp.chunk > 0 || sp.seg) {
        if (!workspace || workspace_bytes < sp.bytes) return FA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_MISALIGNED;
    }
    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    FwdParams p{};
    const int BH = B * H;
    if ((rc = make_bhnd_map(&p.tm_q, q, BH, N, d, 128)) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_k, k, B * Hkv, N, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_v, v, B * Hkv, N, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    p.o = o;
    p.lse = lse;
    p.N = N;
    p.BH = BH;
    p.H = H;
    p.group = group;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.kv_chunk = sp.chunk;
    p.seg = sp.seg;
    if (sp.chunk > 0 || sp.seg) {
        p.ws_o = static_cast<float *>(workspace);
        p.ws_l = reinterpret_cast<float *>(static_cast<char *>(workspace) + sp.l_offset);
        p.s_max = sp.s_max;
    }
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_fwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int H, int Hkv, int N, int d, int causal, float scale, void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int rc = check_sizes(B, H, N, d, true);
    if (rc != FA_OK) return rc;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    if ((rc = check_scale(scale)) != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;

    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    FwdParams p{};
    const int BH = B * H;
    if ((rc = make_bhnd_map(&p.tm_q, q, BH, N, d, 128)) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_k, k, B * Hkv, N, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_v, v, B * Hkv, N, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    p.o = o;
    p.lse = lse;
    p.N = N;
    p.BH = BH;
    p.H = H;
    p.group = group;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_fwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *q_descale,
                          const float *k_descale, const float *v_descale, void *o, float *lse,
                          int B, int H, int Hkv, int N, int d, int causal, float scale,
                          void *stream) {
    if (!q8 || !k8 || !vt8 || !q_descale || !k_descale || !v_descale || !o || !lse)
        return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if ((long long)B * H * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    int rc = check_scale(scale);
    if (rc != FA_OK) return rc;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse) ||
        !aligned4(q_descale) || !aligned4(k_descale) || !aligned4(v_descale))
        return FA_ERR_MISALIGNED;
    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    FwdParams p{};
    const int BH = B * H, BHkv = B * Hkv;
    const uint64_t np = ((uint64_t)N + 15) / 16 * 16;
    const uint64_t row = (uint64_t)d;  // bytes per row of q8 / k8
    if ((rc = make_u8_map(&p.tm_q, q8, d, N, BH, row, row * N, 128, 128)) != FA_OK) return rc;
    if ((rc = make_u8_map(&p.tm_k, k8, d, N, BHkv, row, row * N, 128, 128)) != FA_OK) return rc;
    if ((rc = make_u8_map(&p.tm_v, vt8, np, d, BHkv, np, np * d, 128, (uint32_t)d)) != FA_OK)
        return rc;
    p.o = o;
    p.lse = lse;
    p.N = N;
    p.BH = BH;
    p.H = H;
    p.group = group;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.fp8 = 1;
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_fwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" size_t fa_quantize_fp8_workspace_bytes(int BH, int N, int d) {
    if (BH < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return 0;
    const size_t chunks = ((size_t)N + 127) / 128;
    return ((size_t)BH * chunks * sizeof(float) + 15) / 16 * 16;
}

extern "C" int fa_quantize_fp8(const void *x, void *codes, float *descale, int BH, int N, int d,
                               int block_rows, const float *signs, int transpose, void *workspace,
                               size_t workspace_bytes, void *stream) {
    if (!x || !codes || !descale) return FA_ERR_INVALID_ARG;
    if (BH < 1 || N < 1 || (long long)BH * N >= (1LL << 31)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (block_rows < 0 || block_rows % 128 != 0) return FA_ERR_INVALID_ARG;
    const size_t need = fa_quantize_fp8_workspace_bytes(BH, N, d);
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(codes) || !aligned4(descale) || !aligned16(workspace) ||
        (signs && !aligned16(signs)))
        return FA_ERR_MISALIGNED;
    DeviceCache *dc = nullptr;
    int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    QuantParams p{};
    p.x = x;
    p.codes = codes;
    p.descale = descale;
    p.partial = static_cast<float *>(workspace);
    p.signs = signs;
    p.BH = BH;
    p.N = N;
    p.d = d;
    p.block_rows = block_rows;
    p.transpose = transpose ? 1 : 0;
    p.Np = (N + 15) / 16 * 16;
    return launch_quant(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                      int H, int N, int d, int causal, float scale, void *stream) {
    return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, stream);
}

extern "C" int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                             const int *cu_seqlens, int B, int H, int Hkv, int total_tokens,
                             int max_seqlen, int d, int causal, float scale, void *stream) {
    if (!q || !k || !v || !o || !lse || !cu_seqlens) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || total_tokens < 1 || max_seqlen < 1) return FA_ERR_INVALID_ARG;
    if ((long long)total_tokens * H >= (1LL << 31) || (long long)B * H >= (1LL << 31))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    int rc = check_scale(scale);
    if (rc != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return FA_ERR_MISALIGNED;
    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    FwdParams p{};
    if ((rc = make_thd_map(&p.tm_q, q, total_tokens, H, d, 128)) != FA_OK) return rc;
    if ((rc = make_thd_map(&p.tm_k, k, total_tokens, Hkv, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    if ((rc = make_thd_map(&p.tm_v, v, total_tokens, Hkv, d, fwd_kv_box_rows(d))) != FA_OK) return rc;
    p.o = o;
    p.lse = lse;
    p.N = max_seqlen;
    p.BH = B * H;
    p.H = H;
    p.group = group;
    p.cu_seqlens = cu_seqlens;
    p.total_tokens = total_tokens;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_fwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (check_sizes(B, H, N, d, false) != FA_OK) return 0;
    const size_t npad = round_up((size_t)N, kBwdPad);
    // delta[BH][Npad] and lse2[BH][Npad], fp32 each, and the work-item counter
    return 2 * (size_t)B * (size_t)H * npad * sizeof(float) + kBwdCounterBytes;
}

extern "C" int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, float *dq, float *dk, float *dv,
                          int B, int H, int Hkv, int N, int d, int causal, float scale,
                          void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    int rc = check_sizes(B, H, N, d, false);
    if (rc != FA_OK) return rc;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    if ((rc = check_scale(scale)) != FA_OK) return rc;
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace))
        return FA_ERR_MISALIGNED;

    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    BwdParams p{};
    const int BH = B * H;
    const int npad = (int)round_up((size_t)N, kBwdPad);
    const int q_rows = bwd_block_q(d);  // query rows per backward q-block
    if ((rc = make_bhnd_map(&p.tm_q, q, BH, N, d, q_rows)) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_do, dout, BH, N, d, q_rows)) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_k, k, B * Hkv, N, d, 128)) != FA_OK) return rc;
    if ((rc = make_bhnd_map(&p.tm_v, v, B * Hkv, N, d, 128)) != FA_OK) return rc;
    if ((rc = make_f32_map(&p.tm_dq, dq, d, N, BH, 32, 1)) != FA_OK) return rc;
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.ws_delta = static_cast<float *>(workspace);
    p.ws_lse2 = p.ws_delta + (size_t)BH * (size_t)npad;
    p.ws_counter = reinterpret_cast<int *>(p.ws_lse2 + (size_t)BH * (size_t)npad);
    p.N = N;
    p.Npad = npad;
    p.BH = BH;
    p.H = H;
    p.group = group;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_bwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, float *dq, float *dk, float *dv,
                             const int *cu_seqlens, int B, int H, int Hkv, int total_tokens,
                             int max_seqlen, int d, int causal, float scale, void *workspace,
                             size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens)
        return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || total_tokens < 1 || max_seqlen < 1) return FA_ERR_INVALID_ARG;
    if ((long long)total_tokens * H >= (1LL << 31) ||
        (long long)B * H * (long long)round_up((size_t)max_seqlen, kBwdPad) >= (1LL << 31))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 96 && d != 128) return FA_ERR_UNSUPPORTED;
    const int group = gqa_group(H, Hkv);
    if (group == 0) return FA_ERR_INVALID_ARG;
    int rc = check_scale(scale);
    if (rc != FA_OK) return rc;
    const size_t need = fa_bwd_workspace_bytes(B, H, max_seqlen, d);
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return FA_ERR_MISALIGNED;
    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return rc;
    BwdParams p{};
    const int BH = B * H;
    const int npad = (int)round_up((size_t)max_seqlen, kBwdPad);
    const int q_rows = bwd_block_q(d);
    if ((rc = make_thd_map(&p.tm_q, q, total_tokens, H, d, q_rows)) != FA_OK) return rc;
    if ((rc = make_thd_map(&p.tm_do, dout, total_tokens, H, d, q_rows)) != FA_OK) return rc;
    if ((rc = make_thd_map(&p.tm_k, k, total_tokens, Hkv, d, 128)) != FA_OK) return rc;
    if ((rc = make_thd_map(&p.tm_v, v, total_tokens, Hkv, d, 128)) != FA_OK) return rc;
    if ((rc = make_f32_map(&p.tm_dq, dq, d, H, total_tokens, 1, 32)) != FA_OK) return rc;
    p.o = o;
    p.dout = dout;
    p.lse = lse;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.ws_delta = static_cast<float *>(workspace);
    p.ws_lse2 = p.ws_delta + (size_t)BH * (size_t)npad;
    p.ws_counter = reinterpret_cast<int *>(p.ws_lse2 + (size_t)BH * (size_t)npad);
    p.N = max_seqlen;
    p.Npad = npad;
    p.BH = BH;
    p.H = H;
    p.group = group;
    p.cu_seqlens = cu_seqlens;
    p.total_tokens = total_tokens;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    p.num_sms = dc->num_sms;
    return launch_bwd(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fa_bwd(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, float *dq, float *dk, float *dv, int B,
                      int H, int N, int d, int causal, float scale, void *workspace,
                      size_t workspace_bytes, void *stream) {
    return fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, H, N, d, causal, scale, workspace,
                      workspace_bytes, stream);
}

namespace fa {
namespace {

// Decode sizes.  R = (H / Hkv) * Nq query rows share each key/value head.
int check_decode_sizes(int B, int H, int Hkv, int Nq, int Nk, int d) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || Nq > 65535) return FA_ERR_INVALID_ARG;
    if (gqa_group(H, Hkv) == 0) return FA_ERR_INVALID_ARG;
    if ((long long)(H / Hkv) * Nq > 65535) return FA_ERR_INVALID_ARG;
    if ((long long)B * H * Nq >= (1LL << 31) || (long long)B * Hkv * Nk >= (1LL << 31))
        return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// Key ranges of the decode split: the requested count (0 = automatic) clamped so
// that every range holds whole pipeline stages and none is empty.  The automatic
// count minimises a wave model of the launch: with `slots` CTAs resident at once,
// a launch of C CTAs of T stages each takes about ceil(C / slots) * (T + 4) stage
// times (four stages of fill and merge per CTA), and each range keeps at least
// eight stages so the ring has something to overlap.  BHkv key/value heads, R
// query rows per key/value head.
void decode_split_uncached(long long BHkv, int R, int Nk, int d, bool paged, int requested,
                           int num_sms, int *S, int *keys_per_split) {
    const long long bk = decode_block_keys(d, R, paged);
    const long long tiles = (Nk + bk - 1) / bk;
    const long long qb = decode_query_block(d, R, paged);
    const long long base = BHkv * ((R + qb - 1) / qb);
    long long s = 1;
    if (requested > 0) {
        s = requested;
    } else {
        // Wave model: C CTAs of T stages each cost about ceil(C / slots) * (T + 4)
        // stage times (the 4 stands for a CTA's ring fill, merge write and launch),
        // minimised over every split down to one stage per CTA.  Short caches are
        // latency-bound, so they split finely (B1 H8 Nk1024 d128: 16 ranges, 7.6 us,
        // against 14.0 us with at least 8 stages per range).
        const long long slots =
            (long long)(num_sms > 0 ? num_sms : 1) * decode_ctas_per_sm(d, R, paged);
        long long cap = tiles;
        if (cap < 1) cap = 1;
        if (cap > 1024) cap = 1024;
        long long best = -1;
        for (long long c = 1; c <= cap; ++c) {
            const long long waves = (base * c + slots - 1) / slots;
            const long long cost = waves * ((tiles + c - 1) / c + 4);
            if (best < 0 || cost < best) {
                best = cost;
                s = c;
            }
        }
    }
    if (s > tiles) s = tiles;
    if (s > 65535) s = 65535;
    if (s < 1) s = 1;
    const long long per = ((tiles + s - 1) / s) * bk;
    *keys_per_split = (int)per;
    *S = (int)((Nk + per - 1) / per);
}

// The same, remembered for the last shapes asked (a decode loop repeats one shape).
void decode_split(long long BHkv, int R, int Nk, int d, bool paged, int requested, int num_sms,
                  int *S, int *keys_per_split) {
    struct Entry {
        long long BHkv;
        int R, Nk, d, paged, requested, num_sms, S, per;
    };
    constexpr int kEntries = 16;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    static std::mutex m;
    {
        std::lock_guard<std::mutex> lock(m);
        for (int i = 0; i < used; ++i) {
            const Entry &e = cache[i];
            if (e.BHkv == BHkv && e.R == R && e.Nk == Nk && e.d == d && e.paged == (int)paged &&
                e.requested == requested && e.num_sms == num_sms) {
                *S = e.S;
                *keys_per_split = e.per;
                return;
            }
        }
    }
    decode_split_uncached(BHkv, R, Nk, d, paged, requested, num_sms, S, keys_per_split);
    std::lock_guard<std::mutex> lock(m);
    cache[next] = Entry{BHkv, R, Nk, d, (int)paged, requested, num_sms, *S, *keys_per_split};
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
}

size_t decode_ws_bytes(long long rows, int S, int d) {  // rows = B * H * Nq
    if (S <= 1) return 0;
    const size_t po = (size_t)rows * S * d * sizeof(float);
    return round_up(po, 256) + (size_t)rows * S * sizeof(float);
}

// Shared tail of fa_decode and fa_decode_paged: split, workspace, launch.
int decode_launch(DecodeParams &p, int B, int num_splits, void *workspace, size_t workspace_bytes,
                  void *stream) {
    DeviceCache *dc = nullptr;
    int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    const int R = p.group * p.Nq;
    decode_split((long long)B * p.Hkv, R, p.Nk, p.d, p.paged != 0, num_splits, dc->num_sms, &p.S,
                 &p.keys_per_split);
    const long long rows = (long long)B * p.H * p.Nq;
    const size_t need = decode_ws_bytes(rows, p.S, p.d);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return FA_ERR_MISALIGNED;
        p.part_o = static_cast<float *>(workspace);
        p.part_l = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             round_up((size_t)rows * p.S * p.d * sizeof(float), 256));
    }
    p.BH = B * p.H;
    if (decode_uses_mma(p.d, R, p.paged != 0)) {
        // tensor-core kernel: q as one [B*H*Nq][d] matrix in boxes of 128 rows, the
        // cache in boxes of one pipeline stage of keys
        if ((rc = make_bhnd_map(&p.tm_q, p.q, 1, (int)rows, p.d, 128)) != FA_OK) return rc;
        const int bk = decode_block_keys(p.d, R, false);
        if ((rc = make_bhnd_map(&p.tm_k, p.k, B * p.Hkv, p.Nk, p.d, bk)) != FA_OK) return rc;
        if ((rc = make_bhnd_map(&p.tm_v, p.v, B * p.Hkv, p.Nk, p.d, bk)) != FA_OK) return rc;
    }
    p.status = dc->status;
    p.limit_ns = kWaitLimitNs;
    return launch_decode(p, static_cast<cudaStream_t>(stream));
}

// Key ranges a decode launch uses, or -(error code).
int decode_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits, bool paged) {
    int rc = check_decode_sizes(B, H, Hkv, Nq, Nk, d);
    if (rc != FA_OK) return -rc;
    if (num_splits < 0) return -FA_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    if ((rc = current_device(&dc)) != FA_OK) return -rc;
    int S = 1, per = 0;
    decode_split((long long)B * Hkv, (H / Hkv) * Nq, Nk, d, paged, num_splits, dc->num_sms, &S,
                 &per);
    return S;
}

}  // namespace
}  // namespace fa

extern "C" int fa_decode_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits) {
    return decode_num_splits(B, H, Hkv, Nq, Nk, d, num_splits, false);
}

extern "C" int fa_decode_uses_tensor_cores(int H, int Hkv, int Nq, int d, int paged) {
    const int rc = check_decode_sizes(1, H, Hkv, Nq, 1, d);
    if (rc != FA_OK) return -rc;
    return decode_uses_mma(d, (H / Hkv) * Nq, paged != 0) ? 1 : 0;
}

extern "C" size_t fa_decode_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d,
                                            int num_splits) {
    const int S = fa_decode_num_splits(B, H, Hkv, Nq, Nk, d, num_splits);
    if (S < 1) return 0;
    return decode_ws_bytes((long long)B * H * Nq, S, d);
}

extern "C" int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int H, int Hkv, int Nq, int Nk, int d, float scale, int num_splits,
                         void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int rc = check_decode_sizes(B, H, Hkv, Nq, Nk, d);
    if (rc != FA_OK) return rc;
    if (num_splits < 0) return FA_ERR_INVALID_ARG;
    if ((rc = check_scale(scale)) != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;
    DecodeParams p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.scale_log2 = scale * kLog2e;
    return decode_launch(p, B, num_splits, workspace, workspace_bytes, stream);
}

namespace fa {
namespace {

// Sizes of a paged decode; the longest possible sequence page_size * max_pages
// plays the role of Nk for the split.
int check_paged_sizes(int B, int H, int Hkv, int Nq, int d, int page_size, int max_pages,
                      int num_pages) {
    if (page_size < 1 || max_pages < 1 || num_pages < 1) return FA_ERR_INVALID_ARG;
    const long long nk = (long long)page_size * max_pages;
    if (nk >= (1LL << 31) || (long long)B * max_pages >= (1LL << 31)) return FA_ERR_INVALID_ARG;
    return check_decode_sizes(B, H, Hkv, Nq, 1, d);
}

}  // namespace
}  // namespace fa

extern "C" int fa_decode_paged_num_splits(int B, int H, int Hkv, int Nq, int d, int page_size,
                                          int max_pages_per_seq, int num_splits) {
    int rc = check_paged_sizes(B, H, Hkv, Nq, d, page_size, max_pages_per_seq, 1);
    if (rc != FA_OK) return -rc;
    return decode_num_splits(B, H, Hkv, Nq, page_size * max_pages_per_seq, d, num_splits, true);
}

extern "C" size_t fa_decode_paged_workspace_bytes(int B, int H, int Hkv, int Nq, int d,
                                                  int page_size, int max_pages_per_seq,
                                                  int num_splits) {
    const int S =
        fa_decode_paged_num_splits(B, H, Hkv, Nq, d, page_size, max_pages_per_seq, num_splits);
    if (S < 1) return 0;
    return decode_ws_bytes((long long)B * H * Nq, S, d);
}

extern "C" int fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                               const int *block_table, const int *seq_lens, void *o, float *lse,
                               int B, int H, int Hkv, int Nq, int d, int page_size,
                               int max_pages_per_seq, int num_pages, float scale, int num_splits,
                               void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse)
        return FA_ERR_INVALID_ARG;
    int rc = check_paged_sizes(B, H, Hkv, Nq, d, page_size, max_pages_per_seq, num_pages);
    if (rc != FA_OK) return rc;
    if (num_splits < 0) return FA_ERR_INVALID_ARG;
    if ((rc = check_scale(scale)) != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        !aligned16(lse) || !aligned4(block_table) || !aligned4(seq_lens))
        return FA_ERR_MISALIGNED;
    DecodeParams p{};
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.o = o;
    p.lse = lse;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.Nq = Nq;
    p.Nk = page_size * max_pages_per_seq;
    p.d = d;
    p.paged = 1;
    p.page_size = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.scale_log2 = scale * kLog2e;
    return decode_launch(p, B, num_splits, workspace, workspace_bytes, stream);
}

extern "C" const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension not supported";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: pointer not aligned (16 bytes for tensors)";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime or driver call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
        case FA_ERR_BAD_INDEX:
            return "FA_ERR_BAD_INDEX: a block-table entry, sequence length or sequence offset "
                   "was out of range";
        default: return "unknown fa_status";
    }
}

extern "C" int fa_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    DeviceCache *dc = nullptr;
    if (current_device(&dc) != FA_OK) return FA_ERR_CUDA;
    int rec[2] = {0, 0};
    if (cudaMemcpy(rec, dc->status, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (rec[0] != 0) {
        const int zero[2] = {0, 0};
        if (cudaMemcpy(dc->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return rec[0];
}

extern "C" int fa_probe_read_bandwidth(const void *buf, size_t bytes, int iters, void *stream,
                                       double *gbs) {
    if (!buf || !gbs || !aligned16(buf) || bytes < ((size_t)1 << 20) || (bytes & 15) ||
        iters < 1 || iters > 1000)
        return FA_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    return run_read_probe(dc->num_sms, buf, bytes, iters, static_cast<cudaStream_t>(stream), gbs);
}

extern "C" int fa_probe_unit_rates(double *rates, int iters, void *stream) {
    if (rates == nullptr || iters < 16 || iters > (1 << 20)) return FA_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    rc = run_unit_probes(dc->num_sms, iters, dc->status, static_cast<cudaStream_t>(stream), rates);
    if (rc == FA_ERR_TIMEOUT) {  // the record is this call's; clear it
        const int zero[2] = {0, 0};
        if (cudaMemcpy(dc->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return rc;
}

extern "C" int fa_selftest_wait_timeout(unsigned long long limit_ns, void *stream) {
    if (limit_ns < 1000ull || limit_ns > 5000000000ull) return FA_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    int rc = current_device(&dc);
    if (rc != FA_OK) return rc;
    fa_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dc->status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
