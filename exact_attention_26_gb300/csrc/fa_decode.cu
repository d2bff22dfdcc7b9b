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

template <int D>
int launch_decode_d(const DecodeParams &p, cudaStream_t stream) {
    constexpr int QB = dec_qblock<D>();
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

int decode_block_keys(int d) { return d == 256 ? DecTile<256>::BK : DecTile<128>::BK; }

int decode_query_block(int d, int Nq) {
    if (Nq == 1) return 1;
    return d == 256 ? dec_qblock<256>() : dec_qblock<128>();
}

int decode_ctas_per_sm(int d, int Nq) {
    switch (d) {
        case 64: return ctas_per_sm_d<64>(Nq);
        case 96: return ctas_per_sm_d<96>(Nq);
        case 128: return ctas_per_sm_d<128>(Nq);
        case 256: return ctas_per_sm_d<256>(Nq);
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
