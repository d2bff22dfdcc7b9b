// Decode attention with the key range split across CTAs and an LSE merge
// (course page "10 FlashAttention", section "The decode variant: FlashDecoding":
// a decode step has one or a few query rows per sequence, so parallelising over
// (batch, head) alone leaves most SMs idle; each CTA instead takes one key range,
// produces a partial result with its own running max and sum, and a second kernel
// merges the partials with the same rescaling the online softmax uses).
//
// The work is a matrix-vector product that streams the key/value cache once, so
// it is bound by HBM bandwidth, not by the tensor cores: keys and values reach
// shared memory through plain bulk copies (a key range of one head is contiguous)
// in an mbarrier ring, and CUDA cores do the arithmetic.  Per CTA: one producer
// warp and four compute warps; compute warp w takes keys [w*KW, w*KW + KW) of
// every stage, its lanes split the head dimension, and each warp keeps its own
// running (max, sum, output) per query row until the four are merged at the end.
#include <atomic>

#include "fa_internal.h"

#include "fa_ptx.cuh"

namespace fa {
namespace {

template <int D>
struct DecTile {
    static constexpr int BK = (D == 256) ? 32 : 64;   // keys per stage
    static constexpr int STAGES = (D == 64) ? 4 : 3;
    static constexpr int NWC = 4;                       // compute warps
    static constexpr int KW = BK / NWC;                 // keys per compute warp per stage
    // head-dim elements per lane, and the lanes that hold some (d = 96: 24 lanes of
    // 4, so every lane's shared-memory reads stay 8-byte vectors; lanes 24-31 hold
    // zeros and touch no memory)
    static constexpr int E = (D == 96) ? 4 : D / 32;
    static constexpr int LANES = D / E;
    static constexpr uint32_t TILE_BYTES = BK * D * 2;  // K (or V) rows of one stage, bf16
    static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 2 * STAGES * 8 + 16;
    static constexpr int THREADS = 32 * (NWC + 1);
    static_assert(KW % 8 == 0, "keys are reduced in groups of eight");
};

// Query rows per CTA: one for plain decode, a block of them otherwise.
template <int D>
constexpr int dec_qblock() { return D == 256 ? 4 : 8; }

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;
// The tensor-core kernel's reference max moves only when a tile's max passes it by
// more than 2^8 (as in the forward): a stale reference cancels exactly in O/l and L.
constexpr float kRescaleLog2Dec = 8.0f;

// Eight per-lane partial dot products (one per key of a group) -> the full
// 32-lane sum of key ((lane >> 2) & 7) in every lane, with 9 shuffles instead of
// 40: each exchange step halves the keys a lane keeps.
__device__ __forceinline__ float reduce8_transpose(const float (&v)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[i + 4];
        const float keep = b4 ? v[i + 4] : v[i];
        a[i] = keep + __shfl_xor_sync(kFull, send, 16);
    }
    float b[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? a[i] : a[i + 2];
        const float keep = b3 ? a[i + 2] : a[i];
        b[i] = keep + __shfl_xor_sync(kFull, send, 8);
    }
    float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(kFull, b2 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(kFull, c, 2);
    c += __shfl_xor_sync(kFull, c, 1);
    return c;
}

// E consecutive bf16 values (E = 2, 4 or 8; address aligned to 2E bytes) from
// shared memory in one load, exactly widened to fp32.
template <int E>
__device__ __forceinline__ void lds_bf16(const uint8_t *p, float (&x)[E]) {
    uint32_t u[E / 2];
    if constexpr (E == 2) {
        u[0] = *reinterpret_cast<const uint32_t *>(p);
    } else if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(p);
        u[0] = w.x; u[1] = w.y;
    } else {
        const uint4 w = *reinterpret_cast<const uint4 *>(p);
        u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w;
    }
#pragma unroll
    for (int w = 0; w < E / 2; ++w) {
        x[2 * w] = __uint_as_float(u[w] << 16);
        x[2 * w + 1] = __uint_as_float(u[w] & 0xffff0000u);
    }
}

// Record a device-side argument error once (code and site) and stop this CTA.
__device__ __forceinline__ void flag_bad_index(int *status, volatile int *abort_flag, int site) {
    *abort_flag = 1;
    atomicCAS(status + 1, 0, site);
    atomicExch(status, FA_ERR_BAD_INDEX);
}

template <int D, int QB, bool PAGED>
__global__ void __launch_bounds__(DecTile<D>::THREADS, 2)
    fa_decode_split_kernel(const __grid_constant__ DecodeParams p) {
    using T = DecTile<D>;
    griddep_launch_dependents();  // the merge kernel may launch while the ranges run
    constexpr int E = T::E, KW = T::KW, BK = T::BK, STAGES = T::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + T::OFF_BAR;            // [STAGES]
    const uint32_t bar_empty = bar_full + 8 * STAGES;        // [STAGES]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + T::OFF_BAR + 16 * STAGES);
    const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *k = reinterpret_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *v = reinterpret_cast<const __nv_bfloat16 *>(p.v);
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.o);
    float *lse = p.lse, *part_o = p.part_o, *part_l = p.part_l;
    const int Nq = p.Nq, S = p.S;
    const float scale_log2 = p.scale_log2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool lane_on = T::LANES == 32 || lane < T::LANES;
    // One CTA per (key/value head, key range, block of query rows).  With grouped
    // queries the rows of key/value head kvh are the Nq rows of each of the `group`
    // query heads that read it (row r: head r / Nq of the group, position r % Nq),
    // so the cache is read once for all of them.
    const int kvh = blockIdx.x, split = blockIdx.y, i0 = blockIdx.z * QB;
    const int R = p.group * Nq;
    const int nq = min(QB, R - i0);
    const int b = kvh / p.Hkv;
    auto qrow = [&](int r) -> size_t {  // flat [B][H][Nq] index of row r of this kv head
        return (size_t)(b * p.H + (kvh % p.Hkv) * p.group + r / Nq) * Nq + r % Nq;
    };
    // Keys of this head: the whole cache, or the sequence's own length when paged
    // (checked on the device: 1 <= len <= page_size * max_pages).
    int len = p.Nk;
    if constexpr (PAGED) len = p.seq_lens[b];
    const bool bad_len = PAGED && (len < 1 || len > p.Nk);
    const int k0 = split * p.keys_per_split;
    const int k1 = bad_len ? k0 : min(len, k0 + p.keys_per_split);
    const int n_tiles = k1 > k0 ? (k1 - k0 + BK - 1) / BK : 0;  // 0: this range is empty

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, T::NWC);
        }
        *abort_flag = 0;
        if (bad_len) flag_bad_index(p.status, abort_flag, SITE_DEC_BAD_LEN);
        fence_mbar_init();
    }
    __syncthreads();
    const Guard g{p.status, abort_flag, p.limit_ns};

    float m[QB], l[QB], acc[QB][E];
    if (warp == T::NWC) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop.  Contiguous cache: lane 0 issues one copy of K
        // and one of V per stage.  Paged cache: lane i looks up page i of the stage
        // (all lookups in flight at once), the warp votes on their validity, and every
        // lane issues the copies of its own page segment.
        int issued = 0;
        const int h = kvh % p.Hkv;
        const int *bt = PAGED ? p.block_table + (size_t)b * p.max_pages : nullptr;
        for (int t = 0; t < n_tiles; ++t) {
            const int slot = t % STAGES;
            if (t >= STAGES && !mbar_wait_warp(bar_empty + 8 * slot, ((t / STAGES) - 1) & 1, g,
                                               SITE_DEC_EMPTY))
                break;
            const int j0 = k0 + t * BK;
            const int rows = min(BK, k1 - j0);
            const uint32_t dst = sbase + slot * T::STAGE_BYTES;
            const uint32_t fb = bar_full + 8 * slot;
            if constexpr (PAGED) {
                // every physical page of this stage is checked before any byte is
                // promised or read: an entry outside [0, num_pages) stops the CTA
                const int ps = p.page_size;
                const int pg0 = j0 / ps, nseg = (j0 + rows - 1) / ps - pg0 + 1;
                bool ok = true;
                for (int i = lane; i < nseg; i += 32) {
                    const int phys = bt[pg0 + i];
                    ok = ok && phys >= 0 && phys < p.num_pages;
                }
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) flag_bad_index(p.status, abort_flag, SITE_DEC_BAD_PAGE);
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(2 * rows * D * 2));
                __syncwarp();
                for (int i = lane; i < nseg; i += 32) {
                    const int pg = pg0 + i;
                    const int js = max(j0, pg * ps), je = min(j0 + rows, (pg + 1) * ps);
                    const size_t src = (((size_t)bt[pg] * p.Hkv + h) * ps + (js - pg * ps)) * D;
                    const uint32_t off = (uint32_t)((js - j0) * D * 2), bytes = (uint32_t)((je - js) * D * 2);
                    bulk_load(dst + off, k + src, bytes, fb);
                    bulk_load(dst + T::TILE_BYTES + off, v + src, bytes, fb);
                }
            } else {
                if (lane == 0) {
                    const size_t src = ((size_t)kvh * p.Nk + j0) * D;
                    const uint32_t bytes = (uint32_t)(rows * D * 2);
                    mbar_arrive_expect_tx(fb, 2 * bytes);
                    bulk_load(dst, k + src, bytes, fb);
                    bulk_load(dst + T::TILE_BYTES, v + src, bytes, fb);
                }
            }
            ++issued;
        }
        if (lane == 0 && *abort_flag) {
            // let every copy still in flight land before the CTA exits
            volatile int never = 0;
            const Guard g2{p.status, &never, kWaitLimitNs};
            for (int t = (issued > STAGES ? issued - STAGES : 0); t < issued; ++t)
                mbar_wait(bar_full + 8 * (t % STAGES), (t / STAGES) & 1, g2, SITE_DEC_DRAIN);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute warps
        float qv[QB][E];
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
            m[qi] = -INFINITY;
            l[qi] = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                acc[qi][e] = 0.f;
                qv[qi][e] = (qi < nq && lane_on) ? __bfloat162float(q[qrow(i0 + qi) * D + lane * E + e])
                                                 : 0.f;
            }
        }
        const int mykey = (lane >> 2) & 7;  // key of a group of eight that this lane scores
        for (int t = 0; t < n_tiles; ++t) {
            const int slot = t % STAGES;
            if (!mbar_wait_warp(bar_full + 8 * slot, (t / STAGES) & 1, g, SITE_DEC_FULL)) break;
            const int nvalid = min(KW, k1 - (k0 + t * BK + warp * KW));  // warp-uniform
            if (nvalid > 0) {
                const uint8_t *Ks = smem + slot * T::STAGE_BYTES + (size_t)warp * KW * D * 2 + lane * E * 2;
                const uint8_t *Vs = Ks + T::TILE_BYTES;
                float sc[QB][KW / 8];
#pragma unroll
                for (int grp = 0; grp < KW / 8; ++grp) {
                    float part[QB][8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        float kx[E];
                        if (lane_on) {
                            lds_bf16<E>(Ks + (size_t)(grp * 8 + r) * D * 2, kx);
                        } else {
#pragma unroll
                            for (int e = 0; e < E; ++e) kx[e] = 0.f;
                        }
#pragma unroll
                        for (int qi = 0; qi < QB; ++qi) {
                            float a = 0.f;
#pragma unroll
                            for (int e = 0; e < E; ++e) a = fmaf(qv[qi][e], kx[e], a);
                            part[qi][r] = a;
                        }
                    }
#pragma unroll
                    for (int qi = 0; qi < QB; ++qi) {
                        const float s2 = reduce8_transpose(part[qi], lane) * scale_log2;
                        sc[qi][grp] = (grp * 8 + mykey < nvalid) ? s2 : -INFINITY;
                    }
                }
                float p[QB][KW / 8];
#pragma unroll
                for (int qi = 0; qi < QB; ++qi) {
                    float mx = sc[qi][0];
#pragma unroll
                    for (int grp = 1; grp < KW / 8; ++grp) mx = fmaxf(mx, sc[qi][grp]);
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                    const float m_new = fmaxf(m[qi], mx);  // finite: this warp has a valid key
                    const float alpha = ex2(m[qi] - m_new);
                    float rs = 0.f;
#pragma unroll
                    for (int grp = 0; grp < KW / 8; ++grp) {
                        p[qi][grp] = ex2(sc[qi][grp] - m_new);  // exp2(-inf) = 0 for masked keys
                        rs += p[qi][grp];
                    }
                    rs += __shfl_xor_sync(kFull, rs, 16);
                    rs += __shfl_xor_sync(kFull, rs, 8);
                    rs += __shfl_xor_sync(kFull, rs, 4);
                    l[qi] = l[qi] * alpha + rs;
                    m[qi] = m_new;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[qi][e] *= alpha;
                }
#pragma unroll
                for (int r = 0; r < KW; ++r) {
                    if (r < nvalid) {
                        float vx[E];
                        if (lane_on) {
                            lds_bf16<E>(Vs + (size_t)r * D * 2, vx);
                        } else {
#pragma unroll
                            for (int e = 0; e < E; ++e) vx[e] = 0.f;
                        }
#pragma unroll
                        for (int qi = 0; qi < QB; ++qi) {
                            const float pr = __shfl_sync(kFull, p[qi][r / 8], (r % 8) << 2);
#pragma unroll
                            for (int e = 0; e < E; ++e) acc[qi][e] = fmaf(pr, vx[e], acc[qi][e]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
    }

    // ---------------------------------------------------------------- merge warps
    // Every stage has been consumed (or the CTA is aborting); the ring's memory now
    // holds each compute warp's (max, sum, unnormalised output) per query row.
    __syncthreads();
    float *red = reinterpret_cast<float *>(smem);  // [NWC][QB][D + 2]
    constexpr int RS = D + 2;
    if (warp < T::NWC) {
#pragma unroll
        for (int qi = 0; qi < QB; ++qi) {
            float *rw = red + (warp * QB + qi) * RS;
            if (lane_on) {
#pragma unroll
                for (int e = 0; e < E; ++e) rw[lane * E + e] = acc[qi][e];
            }
            if (lane == 0) {
                rw[D] = m[qi];
                rw[D + 1] = l[qi];
            }
        }
    }
    __syncthreads();
    if (warp < T::NWC && !*abort_flag) {
        for (int qi = warp; qi < nq; qi += T::NWC) {
            float mw[T::NWC], M = -INFINITY;
#pragma unroll
            for (int w = 0; w < T::NWC; ++w) {
                mw[w] = red[(w * QB + qi) * RS + D];
                M = fmaxf(M, mw[w]);
            }
            float L = 0.f, out[E];
#pragma unroll
            for (int e = 0; e < E; ++e) out[e] = 0.f;
#pragma unroll
            for (int w = 0; w < T::NWC; ++w) {
                // a warp without keys has mw = -inf: f = 0 (and no keys at all: f unused)
                const float f = (mw[w] == -INFINITY) ? 0.f : ex2(mw[w] - M);
                const float *rw = red + (w * QB + qi) * RS;
                L = fmaf(rw[D + 1], f, L);
                if (lane_on) {
#pragma unroll
                    for (int e = 0; e < E; ++e) out[e] = fmaf(rw[lane * E + e], f, out[e]);
                }
            }
            // an empty key range (a short sequence's tail ranges) contributes
            // L = -inf and O = 0 to the merge
            const bool empty = (M == -INFINITY);
            const float inv = empty ? 0.f : 1.f / L;
            const float l_nat = empty ? -INFINITY : (M + lg2(L)) * kLn2;  // natural-log LSE
            const size_t row = qrow(i0 + qi);
            if (S == 1) {
                if (lane_on) {
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        const uint32_t pk = pack_bf16(out[e] * inv, out[e + 1] * inv);
                        *reinterpret_cast<uint32_t *>(o + row * D + lane * E + e) = pk;
                    }
                }
                if (lane == 0) lse[row] = l_nat;
            } else {
                const size_t prow = ((size_t)kvh * S + split) * R + i0 + qi;
                if (lane_on) {
                    float *po = part_o + prow * D + lane * E;
#pragma unroll
                    for (int e = 0; e < E; ++e) po[e] = out[e] * inv;
                }
                if (lane == 0) part_l[prow] = l_nat;
            }
        }
    }
}

// Merge of the S partial results of one query row: L = log sum_s exp(L_s),
// O = sum_s exp(L_s - L) O_s.  One warp per row; lanes split the head dimension.
// Rows are numbered like the split kernel's: key/value head, then its R rows.
template <int D>
__global__ void __launch_bounds__(128)
    fa_decode_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_l,
                             __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, long long rows,
                             int R, int S, int Nq, int H, int Hkv, int group) {
    constexpr int E = DecTile<D>::E;
    griddep_wait();  // every key range's partial result is written
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const bool lane_on = DecTile<D>::LANES == 32 || lane < DecTile<D>::LANES;
    const long long kvh = row / R;
    const int r = (int)(row % R);
    const long long b = kvh / Hkv;
    const size_t orow = (size_t)(b * H + (kvh % Hkv) * group + r / Nq) * Nq + r % Nq;
    const float *pl = part_l + (size_t)kvh * S * R + r;  // stride R over splits
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, pl[(size_t)s * R]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float W = 0.f, out[E];
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = 0.f;
    for (int s = 0; s < S; ++s) {
        const float w = __expf(pl[(size_t)s * R] - M);
        W += w;
        if (lane_on) {
            const float *po = part_o + (((size_t)kvh * S + s) * R + r) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) out[e] = fmaf(w, po[e], out[e]);
        }
    }
    const float inv = 1.f / W;
    if (lane_on) {
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const uint32_t pk = pack_bf16(out[e] * inv, out[e + 1] * inv);
            *reinterpret_cast<uint32_t *>(o + orow * D + lane * E + e) = pk;
        }
    }
    if (lane == 0) lse[orow] = M + __logf(W);
}

// The merge of the key ranges (S > 1), a programmatic dependent of the kernel that
// wrote the partial results.
template <int D>
int launch_decode_combine(const DecodeParams &p, cudaStream_t stream) {
    const int R = p.group * p.Nq;
    if (p.S > 1) {
        const long long rows = (long long)(p.BH / p.group) * R;
        // a programmatic dependent of the split kernel: launched as its last CTAs
        // start, it waits for the whole grid before reading the partial results
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
        cfg.blockDim = dim3(128);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D>, (const float *)p.part_o,
                               (const float *)p.part_l, reinterpret_cast<__nv_bfloat16 *>(p.o),
                               p.lse, rows, R, p.S, p.Nq, p.H, p.Hkv, p.group) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

template <int D, int QB, bool PAGED>
int launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
    using T = DecTile<D>;
    auto kern = fa_decode_split_kernel<D, QB, PAGED>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)T::SMEM_BYTES) != FA_OK)
        return FA_ERR_CUDA;
    const int R = p.group * p.Nq;
    const dim3 grid((unsigned)(p.BH / p.group), (unsigned)p.S, (unsigned)((R + QB - 1) / QB));
    kern<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return launch_decode_combine<D>(p, stream);
}

// ---------------------------------------------------------------------------
// Tensor-core decode, for R = (H / Hkv) Nq >= 2 query rows per
// key/value head (a few new tokens per sequence, or grouped queries).  With
// several rows the score and output products are small matrix products, and on
// CUDA cores their multiply-adds (2 R d per key), not the cache stream, bound the
// kernel.  Here they run as tcgen05 products with M = 128: the CTA's rows of one
// key/value head (up to 128; the rest of the 128 are padding whose results are
// dropped) against tiles of BK keys of K and V (64, or 128 at d = 64: a stage of
// at least 16 KB each) that TMA streams through a ring.  Per tile j:
//   S(j) = Q K_j^T    (A and B from shared memory, N = BK, K = d) into one of two
//                     S slots
//   softmax of the CTA's rows (thread r owns row r: the forward's online softmax
//   with its lazy reference max), P(j) as bf16 over S(j)
//   O += P(j) V_j     (A = P from tensor memory, N = d, K = BK)
// S(j+2) is issued right after PV(j) frees its slot, so the next S is ready while
// the softmax works.  Warps 0-3: softmax (warp w rows 32w..32w+31; warps without
// rows idle); warp 4: TMEM allocation and MMA issue (one elected lane); warp 5:
// TMA producer.  The key range split and the merge of the ranges are the CUDA-core
// kernel's (same partial-result layout).
template <int D>
struct DecMmaTile {
    static constexpr int BM = 128;                   // query rows per CTA (the MMA's M)
    static constexpr int DP = (D + 63) / 64 * 64;    // row width in shared memory
    static constexpr int BK = (DP == 64) ? 128 : 64; // keys per stage (a stage of 16 KB or more)
    static constexpr int NCH = DP / 64;              // 128-byte swizzle chunks per row
    static constexpr int STAGES = 5;
    static constexpr uint32_t Q_CHUNK = BM * 128;
    static constexpr uint32_t KV_CHUNK = BK * 128;
    static constexpr uint32_t Q_BYTES = BM * DP * 2;
    static constexpr uint32_t KV_BYTES = BK * DP * 2;      // one of K_j, V_j
    static constexpr uint32_t STAGE_BYTES = 2 * KV_BYTES;  // K_j, then V_j
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_KV = Q_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_KV + STAGES * STAGE_BYTES;
    // q_full, full[STAGES], empty[STAGES], s_full[2], p_full[2], pv_done, o_full, mma_done
    static constexpr int NBAR = 1 + 2 * STAGES + 2 + 2 + 3;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    static constexpr uint32_t TM_O = 2 * BK;  // S slots at columns 0 and BK, then O (d columns)
    static constexpr uint32_t TM_COLS = (TM_O + D <= 256) ? 256 : 512;
    static constexpr int THREADS = 192;
    static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(Q_CHUNK % 1024 == 0 && KV_CHUNK % 1024 == 0 && KV_BYTES % 1024 == 0,
                  "swizzle atoms must stay aligned");
};

constexpr int kDecMmaMinRows = 2;

template <int D>
__global__ void __launch_bounds__(DecMmaTile<D>::THREADS, 1)
    fa_decode_mma_kernel(const __grid_constant__ DecodeParams p) {
    using T = DecMmaTile<D>;
    griddep_launch_dependents();  // the merge kernel may launch while the ranges run
    constexpr int BK = T::BK, STAGES = T::STAGES;
    extern __shared__ uint8_t dec_smem_raw[];
    const uint32_t raw = smem_u32(dec_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = dec_smem_raw + (base - raw);
    const uint32_t sQ = base + T::OFF_Q, sKV = base + T::OFF_KV;
    const uint32_t bar_q = base + T::OFF_BAR;
    const uint32_t bar_full = bar_q + 8;                  // [STAGES]
    const uint32_t bar_empty = bar_full + 8 * STAGES;     // [STAGES]
    const uint32_t bar_s = bar_empty + 8 * STAGES;        // [2]
    const uint32_t bar_p = bar_s + 16;                    // [2]
    const uint32_t bar_pv = bar_p + 16, bar_o = bar_pv + 8, bar_done = bar_o + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + T::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // One CTA per (key/value head, key range, block of 128 of its R rows).  The R
    // rows of key/value head kvh are consecutive in q, o and lse: the Nq rows of
    // each of its `group` query heads in turn.
    const int kvh = blockIdx.x, split = blockIdx.y;
    const int R = p.group * p.Nq;
    const int r0 = blockIdx.z * T::BM;
    const int nrows = min(T::BM, R - r0);
    const int b = kvh / p.Hkv;
    const long long row_base =
        ((long long)b * p.H + (long long)(kvh % p.Hkv) * p.group) * p.Nq + r0;
    const int k0 = split * p.keys_per_split;
    const int k1 = min(p.Nk, k0 + p.keys_per_split);
    const int n_tiles = k1 > k0 ? (k1 - k0 + BK - 1) / BK : 0;  // 0: an empty range
    const int n_sw = (nrows + 31) / 32;                           // softmax warps with rows

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(bar_s + 8 * u, 1);
            mbar_init(bar_p + 8 * u, 32 * n_sw);  // per S slot, one arrival per softmax thread
        }
        mbar_init(bar_pv, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(tmem_slot), T::TM_COLS);
        tmem_relinquish();
    }
    if (warp == 5 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Guard g{p.status, abort_flag, p.limit_ns};

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            int issued = 0;
            // the CTA's 128 rows of q: rows past this head's R belong to other heads
            // (or read as zeros past the tensor) and are computed and dropped
            mbar_arrive_expect_tx(bar_q, T::Q_BYTES);
            for (int c = 0; c < T::NCH; ++c)
                tma_load_3d(sQ + c * T::Q_CHUNK, &p.tm_q, bar_q, c * 64, (int)row_base, 0);
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % STAGES;
                if (t >= STAGES &&
                    !mbar_wait(bar_empty + 8 * st, ((t / STAGES) - 1) & 1, g, SITE_DEC_EMPTY))
                    break;
                const uint32_t dst = sKV + st * T::STAGE_BYTES;
                const uint32_t fb = bar_full + 8 * st;
                const int key = k0 + t * BK;  // keys past Nk read as zeros and are masked
                mbar_arrive_expect_tx(fb, T::STAGE_BYTES);
                for (int c = 0; c < T::NCH; ++c) {
                    tma_load_3d(dst + c * T::KV_CHUNK, &p.tm_k, fb, c * 64, key, kvh);
                    tma_load_3d(dst + T::KV_BYTES + c * T::KV_CHUNK, &p.tm_v, fb, c * 64, key, kvh);
                }
                ++issued;
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits
                volatile int never = 0;
                const Guard g2{p.status, &never, kWaitLimitNs};
                mbar_wait(bar_q, 0, g2, SITE_DEC_DRAIN);
                for (int t = (issued > STAGES ? issued - STAGES : 0); t < issued; ++t)
                    mbar_wait(bar_full + 8 * (t % STAGES), (t / STAGES) & 1, g2, SITE_DEC_DRAIN);
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (warp-uniform); one elected lane issues.
        constexpr uint32_t kIdescS = idesc_bf16_f32(128, BK, false, false);
        constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
        auto issue_s = [&](int u, int st) {  // S slot u = Q K^T from stage st
            const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk = sdesc_sw128(sKV + st * T::STAGE_BYTES, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t koff = (ks & 3) * 32;
                mma_ss_elect(tmem + BK * u, desc_add(dq, (ks >> 2) * T::Q_CHUNK + koff),
                             desc_add(dk, (ks >> 2) * T::KV_CHUNK + koff), kIdescS, ks > 0 ? 1u : 0u);
            }
            tc_commit_elect(bar_s + 8 * u);
        };
        auto issue_pv = [&](int u, int st, bool first) {  // O += P(slot u) V(stage st)
            const uint64_t dv = sdesc_sw128(sKV + st * T::STAGE_BYTES + T::KV_BYTES, T::KV_CHUNK, 1024);
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
                mma_ts_elect(tmem + T::TM_O, tmem + BK * u + ks * 8, desc_add(dv, ks * 2048), kIdescO,
                             (!first || ks > 0) ? 1u : 0u);
        };
        auto wait_full = [&](int t) {
            const bool r = mbar_wait_warp(bar_full + 8 * (t % STAGES), (t / STAGES) & 1, g, SITE_DEC_FULL);
            tc_fence_after();
            return r;
        };
        bool ok = n_tiles > 0;
        if (ok) {
            ok = mbar_wait_warp(bar_q, 0, g, SITE_DEC_MMA);
            tc_fence_after();
        }
        for (int t = 0; ok && t < 2 && t < n_tiles; ++t)
            if ((ok = wait_full(t))) issue_s(t & 1, t % STAGES);
        for (int j = 0; ok && j < n_tiles; ++j) {
            ok = mbar_wait_warp(bar_p + 8 * (j & 1), (j >> 1) & 1, g, SITE_DEC_MMA);
            tc_fence_after();
            if (!ok) break;
            issue_pv(j & 1, j % STAGES, j == 0);
            tc_commit_elect(bar_pv);
            tc_commit_elect(bar_empty + 8 * (j % STAGES));  // S(j) and PV(j) have read the stage
            if (j + 2 < n_tiles) {
                if (!(ok = wait_full(j + 2))) break;
                issue_s(j & 1, (j + 2) % STAGES);
            }
        }
        if (ok && n_tiles > 0) tc_commit_elect(bar_o);
        // fires once every MMA issued above has completed (normal or aborted run)
        tc_commit_elect(bar_done);
        volatile int never = 0;
        const Guard g2{p.status, &never, kWaitLimitNs};
        mbar_wait_warp(bar_done, 0, g2, SITE_DEC_DRAIN);
    } else if (warp < n_sw) {
        // ------------------------------------------------------------ softmax
        const int r = warp * 32 + lane;  // row of this CTA (TMEM lane r)
        const bool valid = r < nrows;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t t_o = tmem + lane_base + T::TM_O;
        const float c_s = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int u = j & 1;
            const uint32_t t_s = tmem + lane_base + BK * u;
            if (!(ok = mbar_wait_warp(bar_s + 8 * u, (j >> 1) & 1, g, SITE_DEC_MMA))) break;
            tc_fence_after();
            uint32_t sr[BK / 32][32];
#pragma unroll
            for (int c = 0; c < BK / 32; ++c) tmem_ld32(t_s + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < BK / 32; ++c) tmem_wait_ld(sr[c]);
            float s[BK];
#pragma unroll
            for (int c = 0; c < BK / 32; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(sr[c][e]);
            const int key0 = k0 + j * BK;
            if (key0 + BK > k1) {  // the range's last tile: keys from k1 on are not this CTA's
#pragma unroll
                for (int c = 0; c < BK; ++c)
                    if (key0 + c >= k1) s[c] = -INFINITY;
            }
            float mp0 = -INFINITY, mp1 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BK; c += 4) {
                mp0 = fmax3(mp0, s[c], s[c + 1]);
                mp1 = fmax3(mp1, s[c + 2], s[c + 3]);
            }
            const float m_tile = fmaxf(mp0, mp1) * c_s;  // finite: tile j has a key of the range
            float alpha = 1.f;
            const bool move = m_tile > m_ref + kRescaleLog2Dec;
            if (move) {
                alpha = ex2(m_ref - m_tile);
                m_ref = m_tile;
            }
            float sp0 = 0.f, sp1 = 0.f;
            const uint64_t c2 = f32x2_splat(c_s), nm2 = f32x2_splat(-m_ref);
#pragma unroll
            for (int c = 0; c < BK; c += 2) {
                fma_f32x2(s[c], s[c + 1], c2, nm2);
                s[c] = ex2(s[c]);
                s[c + 1] = ex2(s[c + 1]);
                add_f32x2(sp0, sp1, s[c], s[c + 1]);
            }
            l = l * alpha + (sp0 + sp1);
#pragma unroll
            for (int c = 0; c < BK / 64; ++c) {  // P as bf16 pairs over the slot's first BK/2 columns
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(s[64 * c + 2 * e], s[64 * c + 2 * e + 1]);
                tmem_st32(t_s + c * 32, pk);
            }
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                // O <- alpha O once PV(j-1) is complete (PV(j) waits for the arrive below)
                if (!(ok = mbar_wait_warp(bar_pv, (j - 1) & 1, g, SITE_DEC_MMA))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld(o);
                    const uint64_t a2 = f32x2_splat(alpha);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0 = __uint_as_float(o[e]), x1 = __uint_as_float(o[e + 1]);
                        mul_f32x2(x0, x1, a2);
                        o[e] = __float_as_uint(x0);
                        o[e + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(t_o + c * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_p + 8 * u);
        }
        if (ok && n_tiles > 0) ok = mbar_wait_warp(bar_o, 0, g, SITE_DEC_MMA);
        tc_fence_after();
        if (ok && !*abort_flag) {
            // an empty key range contributes L = -inf and O = 0 to the merge
            const bool empty = n_tiles == 0;
            const float inv = empty ? 0.f : 1.f / l;
            const float l_nat = empty ? -INFINITY : (m_ref + lg2(l)) * kLn2;
            const long long row = row_base + r;
            const long long prow = ((long long)kvh * p.S + split) * R + r0 + r;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (!empty) {
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld(o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (!valid) continue;
                if (p.S == 1) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) +
                                                           (size_t)row * D + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.part_o + (size_t)prow * D + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_uint4(__float_as_uint(__uint_as_float(o[4 * e]) * inv),
                                            __float_as_uint(__uint_as_float(o[4 * e + 1]) * inv),
                                            __float_as_uint(__uint_as_float(o[4 * e + 2]) * inv),
                                            __float_as_uint(__uint_as_float(o[4 * e + 3]) * inv));
                }
            }
            if (valid) {
                if (p.S == 1)
                    p.lse[row] = l_nat;
                else
                    p.part_l[prow] = l_nat;
            }
        }
        tmem_wait_st();  // an aborted step may leave a store in flight
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TM_COLS);
    }
}

template <int D>
int launch_decode_mma(const DecodeParams &p, cudaStream_t stream) {
    using T = DecMmaTile<D>;
    auto kern = fa_decode_mma_kernel<D>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)T::SMEM_BYTES) != FA_OK)
        return FA_ERR_CUDA;
    const int R = p.group * p.Nq;
    const dim3 grid((unsigned)(p.BH / p.group), (unsigned)p.S, (unsigned)((R + T::BM - 1) / T::BM));
    kern<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    return launch_decode_combine<D>(p, stream);
}

template <int D>
int launch_decode_d(const DecodeParams &p, cudaStream_t stream) {
    constexpr int QB = dec_qblock<D>();
    if constexpr (D <= 128) {
        if (decode_uses_mma(D, p.group * p.Nq, p.paged != 0)) return launch_decode_mma<D>(p, stream);
    }
    const bool one = p.group * p.Nq == 1;  // one query row per key/value head
    if (p.paged)
        return one ? launch_decode_t<D, 1, true>(p, stream) : launch_decode_t<D, QB, true>(p, stream);
    return one ? launch_decode_t<D, 1, false>(p, stream) : launch_decode_t<D, QB, false>(p, stream);
}

// Resident CTAs per SM of the split kernel, asked of the runtime once per
// (instantiation, device) and remembered.
template <int D, int QB>
int ctas_per_sm_t() {
    static std::atomic<int> cached[kMaxCachedDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const bool cacheable = dev >= 0 && dev < kMaxCachedDevices;
    if (cacheable) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    auto kern = fa_decode_split_kernel<D, QB, false>;
    int n = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)DecTile<D>::SMEM_BYTES) != FA_OK ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, DecTile<D>::THREADS,
                                                      DecTile<D>::SMEM_BYTES) != cudaSuccess)
        return 1;
    n = n > 0 ? n : 1;
    if (cacheable) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <int D>
int ctas_per_sm_d(int Nq) {
    return Nq == 1 ? ctas_per_sm_t<D, 1>() : ctas_per_sm_t<D, dec_qblock<D>()>();
}

}  // namespace

// Several query rows per key/value head, contiguous cache, d <= 128: the tensor-core
// kernel.  (Paged caches and d = 256 stay on the CUDA-core kernel.)
bool decode_uses_mma(int d, int R, bool paged) {
    return !paged && d <= 128 && R >= kDecMmaMinRows;
}

int decode_block_keys(int d, int R, bool paged) {
    if (decode_uses_mma(d, R, paged)) return d == 64 ? DecMmaTile<64>::BK : DecMmaTile<128>::BK;
    return d == 256 ? DecTile<256>::BK : DecTile<128>::BK;
}

int decode_query_block(int d, int R, bool paged) {
    if (decode_uses_mma(d, R, paged)) return DecMmaTile<128>::BM;
    if (R == 1) return 1;
    return d == 256 ? dec_qblock<256>() : dec_qblock<128>();
}

int decode_ctas_per_sm(int d, int R, bool paged) {
    if (decode_uses_mma(d, R, paged)) return 1;  // ~190 KB of shared memory per CTA
    switch (d) {
        case 64: return ctas_per_sm_d<64>(R);
        case 96: return ctas_per_sm_d<96>(R);
        case 128: return ctas_per_sm_d<128>(R);
        case 256: return ctas_per_sm_d<256>(R);
        default: return 1;
    }
}

int launch_decode(const DecodeParams &p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_decode_d<64>(p, stream);
        case 96: return launch_decode_d<96>(p, stream);
        case 128: return launch_decode_d<128>(p, stream);
        case 256: return launch_decode_d<256>(p, stream);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
