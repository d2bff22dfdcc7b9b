// e4m3 block quantisation of Q, K and V for the low-precision forward
// ("FlashAttention: Move Less, Not Compute Less", section "FA1 to FA3: Optimization
// Moves Closer to the Hardware": FP8 with block quantisation and incoherent
// processing; course page "10 FlashAttention", section "FlashAttention-1 -> 2 -> 3").
//
// Readings (the pages give neither the format nor the block shape): e4m3 with
// round-to-nearest-even and saturation at +-448; one scale per block of
// `block_rows` rows of a head (0: one per head), chosen so that the block's
// largest magnitude maps to 448, in fixed fp32 steps (amax, inv = 448 / amax,
// t = x * inv, code = e4m3(t), descale = amax / 448; an all-zero block takes
// inv = descale = 1); incoherent processing multiplies every row by
// diag(signs) H / sqrt(d) (H the Sylvester-Hadamard matrix), which leaves Q K^T
// unchanged and spreads an outlier column over all columns.
//
// One CTA per 128-row chunk.  With one scale per 128 rows a single pass suffices:
// the chunk's rows stay in registers between its maximum and its conversion.
// Larger blocks (a whole head for V) take two passes, both bound by HBM: the first
// writes the largest magnitude of every chunk, the second reduces the maxima of
// its scale block and converts.  Codes go out plain, or transposed per head to
// [d][Np] (Np = N rounded up to 16) through shared memory.  Warp w of a CTA takes
// rows 16w .. 16w + 15 of the chunk; lane l holds columns [E l, E l + E), E = d / 32,
// so the Hadamard transform is E-wide butterflies in registers, then shuffles.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kChunk = 128;  // rows per CTA
constexpr int kThreads = 256;
constexpr float kE4m3Max = 448.f;

template <int D, bool HAD>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *__restrict__ row,
                                         const float *__restrict__ signs, int lane,
                                         float (&v)[D / 32]) {
    constexpr int E = D / 32;
    const __nv_bfloat16 *src = row + lane * E;
    if constexpr (E == 2) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(src));
        v[0] = f.x;
        v[1] = f.y;
    } else {
        uint32_t w[E / 2];
        if constexpr (E == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(src);
            w[0] = u.x; w[1] = u.y;
        } else {
            const uint4 u = *reinterpret_cast<const uint4 *>(src);
            w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        }
#pragma unroll
        for (int i = 0; i < E / 2; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    if constexpr (HAD) {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] *= signs[lane * E + e];
        // y = H x: for every stage h, the pair (i, i + h) with bit h of i clear
        // becomes (x_i + x_{i+h}, x_i - x_{i+h})
#pragma unroll
        for (int h = 1; h < E; h <<= 1)
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (!(e & h)) {
                    const float a = v[e], b = v[e + h];
                    v[e] = a + b;
                    v[e + h] = a - b;
                }
#pragma unroll
        for (int h = E; h < D; h <<= 1) {
            const int lm = h / E;
            const bool upper = lane & lm;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, v[e], lm);
                v[e] = upper ? o - v[e] : v[e] + o;
            }
        }
        constexpr float kNorm = (D == 64) ? 0.125f : (D == 128) ? 0.08838834764831845f : 0.0625f;
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] *= kNorm;
    }
}

constexpr int kRowsPerWarp = kChunk / (kThreads / 32);

// Element e of a lane's bf16 pairs, widened exactly to fp32.
template <int W>
__device__ __forceinline__ float bf16_at(const uint32_t (&w)[W], int e) {
    const uint32_t u = w[e >> 1];
    return __uint_as_float((e & 1) ? (u & 0xffff0000u) : (u << 16));
}

// Rows rr of this warp's share of the chunk, all loads issued before any use (the
// rows are independent; a warp keeps kRowsPerWarp of them in flight).  Rows past N
// read as zeros.
template <int D, bool HAD>
__device__ __forceinline__ void load_chunk(const QuantParams &p, int bh, int chunk, int warp,
                                           int lane, float (&v)[kRowsPerWarp][D / 32]) {
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x) + (size_t)bh * p.N * D;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int row = chunk * kChunk + warp * kRowsPerWarp + rr;
        if (row < p.N) {
            load_row<D, HAD>(x + (size_t)row * D, p.signs, lane, v[rr]);
        } else {
#pragma unroll
            for (int e = 0; e < D / 32; ++e) v[rr][e] = 0.f;
        }
    }
}

// Without the transform the rows are kept as the raw bf16 pairs (half the
// registers of fp32 values, so more CTAs fit on an SM); value(e) widens exactly.
template <int D>
__device__ __forceinline__ void load_chunk_raw(const QuantParams &p, int bh, int chunk, int warp,
                                               int lane, uint32_t (&w)[kRowsPerWarp][D / 64]) {
    constexpr int W = D / 64;  // 32-bit words (bf16 pairs) per lane per row
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(p.x) + (size_t)bh * p.N * D;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int row = chunk * kChunk + warp * kRowsPerWarp + rr;
        const __nv_bfloat16 *src = x + (size_t)row * D + lane * 2 * W;
        if (row < p.N) {
            if constexpr (W == 1) {
                w[rr][0] = *reinterpret_cast<const uint32_t *>(src);
            } else if constexpr (W == 2) {
                const uint2 u = *reinterpret_cast<const uint2 *>(src);
                w[rr][0] = u.x; w[rr][1] = u.y;
            } else {
                const uint4 u = *reinterpret_cast<const uint4 *>(src);
                w[rr][0] = u.x; w[rr][1] = u.y; w[rr][2] = u.z; w[rr][3] = u.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i) w[rr][i] = 0u;
        }
    }
}

// Largest |value| of a lane's raw rows: bf16 magnitudes (sign bit cleared) order
// like unsigned integers, so the maximum is taken on the bits (which also keeps the
// compiler from holding every widened value live until the conversion).
template <int R, int W>
__device__ __forceinline__ float raw_absmax(const uint32_t (&w)[R][W]) {
    uint32_t mi = 0;
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
        for (int i = 0; i < W; ++i) {
            mi = max(mi, w[rr][i] & 0x7fffu);
            mi = max(mi, (w[rr][i] >> 16) & 0x7fffu);
        }
    return __uint_as_float(mi << 16);
}

// Largest magnitude over the CTA (all threads get it).
__device__ __forceinline__ float block_max(float m, float *red, int warp, int lane) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
    return r;
}

template <int D, bool HAD>
__global__ void __launch_bounds__(kThreads)
    fa_quant_amax_kernel(const __grid_constant__ QuantParams p) {
    constexpr int E = D / 32;
    const int n_chunks = (p.N + kChunk - 1) / kChunk;
    const int bh = blockIdx.x / n_chunks, chunk = blockIdx.x % n_chunks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float v[HAD ? kRowsPerWarp : 1][E];
    uint32_t raw[HAD ? 1 : kRowsPerWarp][D / 64];
    if constexpr (HAD)
        load_chunk<D, true>(p, bh, chunk, warp, lane, v);
    else
        load_chunk_raw<D>(p, bh, chunk, warp, lane, raw);
    float m = 0.f;
    if constexpr (HAD) {
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
            for (int e = 0; e < E; ++e) m = fmaxf(m, fabsf(v[rr][e]));
    } else {
        m = raw_absmax(raw);
    }
    __shared__ float red[kThreads / 32];
    m = block_max(m, red, warp, lane);
    if (threadIdx.x == 0) p.partial[blockIdx.x] = m;  // = [bh][chunk]
}

// FUSED (block_rows = 128, one scale block per chunk): the chunk's own maximum, no
// first pass.  Otherwise the maxima of the scale block's chunks from the first pass.
template <int D, bool HAD, bool TRANSPOSE, bool FUSED>
__global__ void __launch_bounds__(kThreads, (D <= 128 && !HAD) ? 3 : 1)
    fa_quant_convert_kernel(const __grid_constant__ QuantParams p) {
    constexpr int E = D / 32;
    const int n_chunks = (p.N + kChunk - 1) / kChunk;
    const int bh = blockIdx.x / n_chunks, chunk = blockIdx.x % n_chunks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cpg = FUSED ? 1 : (p.block_rows > 0 ? p.block_rows / kChunk : n_chunks);
    const int grp = chunk / cpg;
    const int g0 = grp * cpg, g1 = min(g0 + cpg, n_chunks);
    __shared__ float red[kThreads / 32];
    float v[HAD ? kRowsPerWarp : 1][E];
    uint32_t raw[HAD ? 1 : kRowsPerWarp][D / 64];
    if constexpr (HAD)
        load_chunk<D, true>(p, bh, chunk, warp, lane, v);
    else
        load_chunk_raw<D>(p, bh, chunk, warp, lane, raw);
    auto val = [&](int rr, int e) -> float {
        if constexpr (HAD)
            return v[rr][e];
        else
            return bf16_at(raw[rr], e);
    };
    float m = 0.f;
    if constexpr (FUSED && HAD) {
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
            for (int e = 0; e < E; ++e) m = fmaxf(m, fabsf(v[rr][e]));
    } else if constexpr (FUSED) {
        m = raw_absmax(raw);
    } else {
        for (int c = g0 + (int)threadIdx.x; c < g1; c += kThreads)
            m = fmaxf(m, p.partial[(size_t)bh * n_chunks + c]);
    }
    const float amax = block_max(m, red, warp, lane);
    const bool zero = !(amax > 0.f);
    const float inv = zero ? 1.f : __fdiv_rn(kE4m3Max, amax);
    if (chunk == g0 && threadIdx.x == 0) {
        const int n_groups = (n_chunks + cpg - 1) / cpg;
        p.descale[(size_t)bh * n_groups + grp] = zero ? 1.f : __fdiv_rn(amax, kE4m3Max);
    }

    uint8_t *codes = reinterpret_cast<uint8_t *>(p.codes);
    // TRANSPOSE: the chunk's codes in row order first, [kChunk][D] bytes
    __shared__ __align__(16) uint8_t tile[TRANSPOSE ? kChunk * D : 16];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int lr = warp * kRowsPerWarp + rr;
        const int row = chunk * kChunk + lr;
        if (!TRANSPOSE && row >= p.N) break;
        uint32_t w[(E + 3) / 4];
        float t[E];
#pragma unroll
        for (int e = 0; e < E; ++e) t[e] = __fmul_rn(val(rr, e), inv);
        if constexpr (E == 2) {
            w[0] = pack_e4m3x4(t[0], t[1], 0.f, 0.f) & 0xffffu;
        } else {
#pragma unroll
            for (int i = 0; i < E / 4; ++i)
                w[i] = pack_e4m3x4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
        }
        // rows past N hold zeros: the zero padding of V^T
        uint8_t *dst = TRANSPOSE ? tile + lr * D + lane * E
                                 : codes + ((size_t)bh * p.N + row) * D + lane * E;
        if constexpr (E == 2)
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w[0];
        else if constexpr (E == 4)
            *reinterpret_cast<uint32_t *>(dst) = w[0];
        else
            *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    }
    if constexpr (TRANSPOSE) {
        __syncthreads();
        // output row c of this head, bytes [n0 + 32 s, n0 + 32 s + 32): thread task
        // (c, s); a warp takes 32 consecutive c, so its byte reads of one tile row
        // fall in 8 words (no bank conflicts)
        const int n0 = chunk * kChunk;
        for (int task = threadIdx.x; task < D * (kChunk / 32); task += kThreads) {
            const int c = task % D, sgm = task / D;
            const int nb = n0 + 32 * sgm;
            if (nb >= p.Np) continue;
            uint32_t u[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint8_t *t = tile + (32 * sgm + 4 * i) * D + c;
                u[i] = (uint32_t)t[0] | ((uint32_t)t[D] << 8) | ((uint32_t)t[2 * D] << 16) |
                       ((uint32_t)t[3 * D] << 24);
            }
            uint4 *out = reinterpret_cast<uint4 *>(codes + ((size_t)bh * D + c) * p.Np + nb);
            out[0] = make_uint4(u[0], u[1], u[2], u[3]);
            if (nb + 16 < p.Np) out[1] = make_uint4(u[4], u[5], u[6], u[7]);
        }
    }
}

template <int D, bool HAD>
int launch_quant_t(const QuantParams &p, cudaStream_t stream) {
    const long long n_chunks = (p.N + kChunk - 1) / kChunk;
    const long long grid = n_chunks * p.BH;
    if (grid > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if (p.block_rows == kChunk) {  // one scale block per chunk: a single pass
        if (p.transpose)
            fa_quant_convert_kernel<D, HAD, true, true><<<(unsigned)grid, kThreads, 0, stream>>>(p);
        else
            fa_quant_convert_kernel<D, HAD, false, true><<<(unsigned)grid, kThreads, 0, stream>>>(p);
        return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    fa_quant_amax_kernel<D, HAD><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    if (p.transpose)
        fa_quant_convert_kernel<D, HAD, true, false><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    else
        fa_quant_convert_kernel<D, HAD, false, false><<<(unsigned)grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_quant_d(const QuantParams &p, cudaStream_t stream) {
    return p.signs ? launch_quant_t<D, true>(p, stream) : launch_quant_t<D, false>(p, stream);
}

}  // namespace

int launch_quant(const QuantParams &p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_quant_d<64>(p, stream);
        case 128: return launch_quant_d<128>(p, stream);
        case 256: return launch_quant_d<256>(p, stream);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
