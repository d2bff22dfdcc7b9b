// Forward pass of exact attention for sm_103a.
//
// One CTA owns one tile of 128 query rows of one (batch, head) and streams the
// K/V tiles of that head through shared memory ("FlashAttention-2: Why the
// Attention Bottleneck Wasn't Where Everyone Was Looking", section "FA2 change
// #2": outer loop over query blocks, inner loop over key/value blocks, the
// softmax state kept on chip).  Per K/V tile j:
//
//   S   = Q K_j^T                     tcgen05.mma, fp32 accumulator in TMEM
//   m'  = max(m, rowmax(S) * scale)   one thread per row, the whole row in registers
//   P   = exp(S * scale - m')         written back to TMEM as bf16 over S
//   l'  = exp(m - m') l + rowsum(P)
//   O~  = exp(m - m') O~ + P V_j      rescale in TMEM, then tcgen05.mma (A = P from TMEM)
//
// which is the online-softmax update of "FlashAttention: Move Less, Not Compute
// Less", section "Tiling Is Easy; Softmax Couples the Entire Row", with the
// division by l deferred to the end ("FA2 change #1").  Exponentials run in base
// 2 with scale*log2(e) folded into one FMA.  The reference maximum m only moves
// when the new row maximum exceeds it by more than 2^8 (kRescaleLog2); a stale
// reference cancels exactly in O~/l and in L, and keeps every P <= 256.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); rescale of O~;
//              epilogue O = O~/l -> bf16, L = (m + log2 l) ln 2
//   warp 4     TMA producer (lane 0): Q once, then K_j/V_j into a 2-stage ring
//   warp 5     TMEM allocator; lane 0 issues every MMA and commit
//
// Causal tiles above the diagonal are never loaded; the diagonal and the ragged
// tail (keys >= N) are masked to -inf element by element, other tiles take no
// mask work ("The causal masking freebie").  Rows past N compute on zero-filled
// Q rows and are not stored.
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdTile {
    static constexpr int BM = 128;                  // query rows per tile
    static constexpr int BN = (D == 256) ? 64 : 128;  // keys per K/V tile
    static constexpr int STAGES = 2;
    static constexpr int NCH = D / 64;              // 128-byte swizzle chunks per row
    static constexpr uint32_t Q_CHUNK = BM * 128;
    static constexpr uint32_t KV_CHUNK = BN * 128;
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    // tensor memory columns
    static constexpr uint32_t TM_S = 0;             // S (fp32, BN cols), P (bf16) over it
    static constexpr uint32_t TM_O = 128;           // O~ (fp32, D cols)
    static constexpr uint32_t TM_COLS = (128 + D <= 256) ? 256 : 512;
    // shared memory layout (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
    // barriers: q_full, kv_full[STAGES], kv_empty[STAGES], s_full, p_full, o_full
    static constexpr int NBAR = 1 + 2 * STAGES + 3;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int THREADS = 192;

    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(Q_CHUNK % 1024 == 0 && KV_CHUNK % 1024 == 0, "swizzle atoms must stay aligned");
    static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
    static_assert(BN % 64 == 0, "P is packed 64 keys per tcgen05.st");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ out,
                  float *__restrict__ lse, int N, int BH, int n_qblocks, float scale_log2,
                  int *status, unsigned long long limit_ns) {
    using T = FwdTile<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t sQ = base + T::OFF_Q;
    const uint32_t sK = base + T::OFF_K;
    const uint32_t sV = base + T::OFF_V;
    const uint32_t bar_q = base + T::OFF_BAR;
    const uint32_t bar_kv_full = bar_q + 8;
    const uint32_t bar_kv_empty = bar_kv_full + 8 * T::STAGES;
    const uint32_t bar_s_full = bar_kv_empty + 8 * T::STAGES;
    const uint32_t bar_p_full = bar_s_full + 8;
    const uint32_t bar_o_full = bar_p_full + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + T::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Tile of this CTA.  Causal: the longest rows (largest q-block) go first.
    const int bh = blockIdx.x % BH;
    const int qb = CAUSAL ? (n_qblocks - 1 - (int)(blockIdx.x / BH)) : (int)(blockIdx.x / BH);
    const int n_kv_all = (N + T::BN - 1) / T::BN;
    const int n_kv = CAUSAL ? min(n_kv_all, ((qb + 1) * T::BM + T::BN - 1) / T::BN) : n_kv_all;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(bar_kv_full + 8 * s, 1);
            mbar_init(bar_kv_empty + 8 * s, 1);
        }
        mbar_init(bar_s_full, 1);
        mbar_init(bar_p_full, 128);
        mbar_init(bar_o_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), T::TM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Guard g{status, abort_flag, limit_ns};

    if (warp == 4) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, T::Q_BYTES);
            for (int c = 0; c < T::NCH; ++c)
                tma_load_3d(sQ + c * T::Q_CHUNK, &tm_q, bar_q, c * 64, qb * T::BM, bh);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % T::STAGES;
                if (j >= T::STAGES &&
                    !mbar_wait(bar_kv_empty + 8 * s, ((j / T::STAGES) - 1) & 1, g,
                               SITE_FWD_LOAD_KV_EMPTY))
                    break;
                mbar_arrive_expect_tx(bar_kv_full + 8 * s, 2 * T::KV_BYTES);
                for (int c = 0; c < T::NCH; ++c) {
                    tma_load_3d(sK + s * T::KV_BYTES + c * T::KV_CHUNK, &tm_k, bar_kv_full + 8 * s,
                                c * 64, j * T::BN, bh);
                    tma_load_3d(sV + s * T::KV_BYTES + c * T::KV_CHUNK, &tm_v, bar_kv_full + 8 * s,
                                c * 64, j * T::BN, bh);
                }
                ++issued;
            }
            if (*abort_flag) {
                // Let the copies already in flight land before the CTA exits.
                volatile int never = 0;
                const Guard g2{status, &never, limit_ns / 4};
                mbar_wait(bar_q, 0, g2, SITE_FWD_DRAIN);
                for (int j = (issued > T::STAGES ? issued - T::STAGES : 0); j < issued; ++j)
                    mbar_wait(bar_kv_full + 8 * (j % T::STAGES), (j / T::STAGES) & 1, g2,
                              SITE_FWD_DRAIN);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, T::BN, false, false);
            constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
            bool ok = mbar_wait(bar_q, 0, g, SITE_FWD_MMA_Q);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % T::STAGES;
                if (!mbar_wait(bar_kv_full + 8 * s, (j / T::STAGES) & 1, g, SITE_FWD_MMA_KV_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t k_tile = sK + s * T::KV_BYTES;
                // S = Q K_j^T: M = 128, N = BN, K = D in steps of 16 (32 bytes).
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks & 3) * 32;  // 16 bf16 = 32 bytes per K step
                    const uint64_t a = sdesc_sw128(sQ + (ks >> 2) * T::Q_CHUNK + koff, 16, 1024);
                    const uint64_t b = sdesc_sw128(k_tile + (ks >> 2) * T::KV_CHUNK + koff, 16, 1024);
                    mma_ss(tmem + T::TM_S, a, b, kIdescS, ks > 0 ? 1u : 0u);
                }
                tc_commit(bar_s_full);
                if (!mbar_wait(bar_p_full, j & 1, g, SITE_FWD_MMA_P_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // O~ += P V_j: M = 128, N = D, K = BN; P from TMEM, V MN-major in smem.
                const uint32_t v_tile = sV + s * T::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < T::BN / 16; ++ks) {
                    const uint64_t b = sdesc_sw128(v_tile + ks * 2048, T::KV_CHUNK, 1024);
                    mma_ts(tmem + T::TM_O, tmem + T::TM_S + ks * 8, b, kIdescO,
                           (j > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(bar_kv_empty + 8 * s);
            }
            // Fires once every MMA issued above has completed (normal or aborted run).
            tc_commit(bar_o_full);
            volatile int never = 0;
            const Guard g2{status, &never, limit_ns};
            mbar_wait(bar_o_full, 0, g2, SITE_FWD_DRAIN);
        }
    } else {
        // ------------------------------------------------------- softmax warps
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t t_s = tmem + lane_base + T::TM_S;
        const uint32_t t_o = tmem + lane_base + T::TM_O;
        const int row = threadIdx.x;
        const int q_idx = qb * T::BM + row;
        float m_ref = -INFINITY;  // reference max, base-2 scaled units
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            ok = mbar_wait_warp(bar_s_full, j & 1, g, SITE_FWD_SOFTMAX_S_FULL);
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[T::BN / 32][32];
#pragma unroll
            for (int c = 0; c < T::BN / 32; ++c) tmem_ld32(t_s + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < T::BN / 32; ++c) tmem_wait_ld(sr[c]);
            float s[T::BN];
#pragma unroll
            for (int c = 0; c < T::BN / 32; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(sr[c][e]);

            const int kv0 = j * T::BN;
            const bool need_mask = (kv0 + T::BN > N) || (CAUSAL && kv0 + T::BN - 1 > qb * T::BM);
            if (need_mask) {
                const int lim = CAUSAL ? min(N, q_idx + 1) : N;  // keys [0, lim) are visible
#pragma unroll
                for (int c = 0; c < T::BN; ++c)
                    if (kv0 + c >= lim) s[c] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < T::BN; ++c) mx = fmaxf(mx, s[c]);
            const float m_tile = mx * scale_log2;
            float alpha = 1.f;
            const bool move = m_tile > m_ref + kRescaleLog2;
            if (move) {
                alpha = ex2(m_ref - m_tile);
                m_ref = m_tile;
            }
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                // O~ <- alpha O~ for this warp's 32 rows (alpha = 1 on rows that kept m).
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(t_o + c * 32, o);
                }
            }
            const float neg_m = -m_ref;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < T::BN; ++c) {
                s[c] = ex2(fmaf(s[c], scale_log2, neg_m));
                sum += s[c];
            }
            l = l * alpha + sum;
            // P as bf16 pairs into the first BN/2 columns of S.
#pragma unroll
            for (int c = 0; c < T::BN / 64; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(s[c * 64 + 2 * e], s[c * 64 + 2 * e + 1]);
                tmem_st32(t_s + c * 32, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_p_full);
        }
        // ------------------------------------------------------- epilogue
        ok = ok && mbar_wait_warp(bar_o_full, 0, g, SITE_FWD_EPILOGUE_O_FULL);
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            __nv_bfloat16 *orow = out + ((size_t)bh * (size_t)N + (size_t)q_idx) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_o + c * 32, o);
                tmem_wait_ld(o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l,
                                      __uint_as_float(o[2 * e + 1]) * inv_l);
                if (q_idx < N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (q_idx < N) lse[(size_t)bh * (size_t)N + q_idx] = (m_ref + lg2(l)) * kLn2;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TM_COLS);
    }
}

template <int D, bool CAUSAL>
int launch_fwd_t(const FwdParams &p, cudaStream_t stream) {
    using T = FwdTile<D>;
    auto kern = fa_fwd_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)T::SMEM_BYTES);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    const int n_qblocks = (p.N + T::BM - 1) / T::BM;
    const long long grid = (long long)n_qblocks * p.BH;
    if (grid > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    kern<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(
        p.tm_q, p.tm_k, p.tm_v, reinterpret_cast<__nv_bfloat16 *>(p.o), p.lse, p.N, p.BH,
        n_qblocks, p.scale_log2, p.status, p.limit_ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_fwd(const FwdParams &p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return p.causal ? launch_fwd_t<64, true>(p, stream) : launch_fwd_t<64, false>(p, stream);
        case 128: return p.causal ? launch_fwd_t<128, true>(p, stream) : launch_fwd_t<128, false>(p, stream);
        case 256: return p.causal ? launch_fwd_t<256, true>(p, stream) : launch_fwd_t<256, false>(p, stream);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
