// Backward pass of exact attention for sm_103a.
//
// The pages fix the structure ("FlashAttention-2: Why the Attention Bottleneck
// Wasn't Where Everyone Was Looking", section "FA2 change #2", backward: one
// worker per K/V column block owns dK_j and dV_j, dQ takes additive updates;
// "FlashAttention: Move Less, Not Compute Less", section "Why More Arithmetic Can
// Finish Sooner": S and P are rebuilt on chip from the saved row statistics).
// The formulas are the chain rule of O = softmax(scale QK^T + mask) V:
//
//   P   = exp(scale S - L)                  (S = Q K^T, L the forward's log-sum-exp)
//   dV  = P^T dO
//   dP  = dO V^T
//   dS  = P o (dP - D),   D_i = dO_i . O_i
//   dQ  = scale dS K,     dK = scale dS^T Q
//
// Kernel 1 (fa_bwd_pre_kernel): -D_i and -L_i log2(e), negated so the main kernel
// adds them (padded rows get 0 and -inf, so their P is exactly 0), and dQ := 0.
//
// Kernel 2 (fa_bwd_kernel): one CTA per (batch * key/value head, block of 128
// keys), looping over blocks of 64 query rows.  All products are tcgen05 MMAs
// with fp32 accumulators in tensor memory, computed in the transposed orientation
// so that a TMEM lane is a key:
//
//   S^T  = K_j Q_i^T        (A = K  smem K-major,  B = Q  smem K-major)
//   dP^T = V_j dO_i^T       (A = V,  B = dO)
//   dV  += P^T dO_i         (A = P^T from TMEM,  B = dO smem MN-major)
//   dK  += dS^T Q_i         (A = dS^T from TMEM, B = Q  smem MN-major)
//   dQ_i^T = K_j^T dS^T     (A = K smem MN-major, B = dS^T smem MN-major)
//
// dQ_i leaves tensor memory through a shared-memory staging tile and one bulk
// asynchronous fp32 add (cp.reduce.async.bulk) into the global dQ rows.  At the
// end dK (times scale) and dV leave once, through shared memory and bulk copies.
//
// Warp roles (448 threads):
//   warps 0-7   P^T = exp2(S^T scale log2e - L log2e), dS^T = P^T o (dP^T - D)
//               (one key per thread, two warpgroups split a block's 64 queries),
//               written as bf16 to TMEM and dS^T to smem; final dK/dV epilogue
//   warps 8-11  dQ readout: TMEM -> staging smem -> bulk add into global dQ
//   warp 12     TMA producer: K_j, V_j once; Q_i, dO_i, L_i, D_i per ring stage
//   warp 13     TMEM allocator; one elected lane issues every MMA and commit
#include "fa_ptx.cuh"

namespace fa {
namespace {

// ---------------------------------------------------------------- preprocess

// VARLEN: o, dout, dq token-major [T][H][D], lse [H][T], sequence b = tokens
// cu_seqlens[b] .. cu_seqlens[b+1]-1 (N is then the maximum length); the workspace
// rows stay [B*H][Npad].  Rows of a sequence that breaks the bounds are treated
// as padding (the main kernel reports it).
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256)
    fa_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                      const float *__restrict__ lse, float *__restrict__ delta,
                      float *__restrict__ lse2, float *__restrict__ dq, int N, int Npad, int BH,
                      int H, const int *__restrict__ cu_seqlens, int total_tokens) {
    // A warp takes RPW consecutive rows at a time (Npad is a multiple of 128, so they
    // share a head) and issues all their loads before any arithmetic: the kernel is
    // bound by HBM, and one row of O and dO per warp leaves too few bytes in flight.
    constexpr int RPW = 4;
    constexpr int PER = D / 32;  // elements per lane
    griddep_launch_dependents();  // the main kernel may set up while this one runs
    constexpr int W = PER == 3 ? 3 : PER / 2;  // loaded words: bf16 pairs, or 3 halves at d = 96
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long groups = (long long)BH * Npad / RPW;
    constexpr float kLog2e = 1.4426950408889634074f;
    for (long long gidx = warp0; gidx < groups; gidx += nwarps) {
        const long long r0 = gidx * RPW;
        const int bh = (int)(r0 / Npad);
        const int i0 = (int)(r0 % Npad);
        int len = N;
        size_t row0, lse0;  // element offset of row i0, index of its L
        if constexpr (VARLEN) {
            const int b = bh / H, h = bh % H;
            const int a = cu_seqlens[b], e = cu_seqlens[b + 1];
            len = (a >= 0 && e >= a && e <= total_tokens && e - a <= N) ? e - a : 0;
            row0 = ((size_t)(a + i0) * H + h) * D;
            lse0 = (size_t)h * total_tokens + a + i0;
        } else {
            row0 = ((size_t)bh * N + i0) * D;
            lse0 = (size_t)bh * N + i0;
        }
        const size_t rstride = VARLEN ? (size_t)H * D : (size_t)D;  // between consecutive rows
        uint32_t ow[RPW][W], dw[RPW][W];
        float lv[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const bool on = i0 + k < len;
            const size_t row = row0 + (size_t)k * rstride;
            if constexpr (PER == 3) {
                // d = 96: lane takes columns lane, lane + 32, lane + 64 (each load of the
                // warp reads 64 contiguous bytes)
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    const size_t c = row + (size_t)(lane + 32 * e);
                    ow[k][e] = on ? (uint32_t)__bfloat16_as_ushort(o[c]) << 16 : 0u;
                    dw[k][e] = on ? (uint32_t)__bfloat16_as_ushort(dout[c]) << 16 : 0u;
                }
            } else if constexpr (PER == 4) {
                const size_t c = row + (size_t)lane * PER;
                const uint2 a = on ? *reinterpret_cast<const uint2 *>(o + c) : make_uint2(0u, 0u);
                const uint2 b = on ? *reinterpret_cast<const uint2 *>(dout + c) : make_uint2(0u, 0u);
                ow[k][0] = a.x; ow[k][1] = a.y;
                dw[k][0] = b.x; dw[k][1] = b.y;
            } else {
                static_assert(PER == 2, "head dim 64, 96 or 128");
                const size_t c = row + (size_t)lane * PER;
                ow[k][0] = on ? *reinterpret_cast<const uint32_t *>(o + c) : 0u;
                dw[k][0] = on ? *reinterpret_cast<const uint32_t *>(dout + c) : 0u;
            }
            lv[k] = (on && lane == 0) ? lse[lse0 + k] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const long long r = r0 + k;
            const size_t row = row0 + (size_t)k * rstride;
            float acc = 0.f;
            if constexpr (PER == 3) {
#pragma unroll
                for (int e = 0; e < 3; ++e)
                    acc = fmaf(__uint_as_float(ow[k][e]), __uint_as_float(dw[k][e]), acc);
            } else {
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    acc = fmaf(__uint_as_float(ow[k][e] << 16), __uint_as_float(dw[k][e] << 16), acc);
                    acc = fmaf(__uint_as_float(ow[k][e] & 0xffff0000u),
                               __uint_as_float(dw[k][e] & 0xffff0000u), acc);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (i0 + k < len) {
                if constexpr (PER == 3) {
#pragma unroll
                    for (int e = 0; e < 3; ++e) dq[row + lane + 32 * e] = 0.f;
                } else if constexpr (PER == 4) {
                    *reinterpret_cast<float4 *>(dq + row + lane * PER) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    *reinterpret_cast<float2 *>(dq + row + lane * PER) = make_float2(0.f, 0.f);
                }
                if (lane == 0) {
                    delta[r] = -acc;
                    lse2[r] = -(lv[k] * kLog2e);
                }
            } else if (lane == 0) {
                delta[r] = 0.f;
                lse2[r] = -INFINITY;
            }
        }
    }
}

// ---------------------------------------------------------------- main kernel
//
// The products are scheduled so the tensor core never waits for the P^T/dS^T
// warps.  Tensor memory (512 columns): dV [0,128), dK [128,256),
// S^T [256,320), dP^T [320,384), PD [384,448) holding bf16 P^T (first 32
// columns) and dS^T (last 32), dQ^T [448,512).  Because P^T and dS^T go to their
// own region, the next block's S^T and dP^T can be issued as soon as the compute
// warps have READ the current ones (st_free), and they run on the tensor core
// while the compute warps work; the dV/dK products of block i release PD for
// block i+1 (pd_free).  Per block the MMA thread issues
//   S^T(i+1), dP^T(i+1)  |  dV(i), dK(i)  |  dQ^T(i)
// Two compute warpgroups split the 64 query columns of a block.
//
// d = 96 keeps the d = 128 layout: rows are two 64-column swizzle chunks whose
// columns past d the copies zero-fill, S^T and dP^T run D/16 K steps, dV and dK
// have N = D, and dQ^T keeps M = 128 (its rows past d come out zero and are not
// read).  d = 64 has rows of one chunk; dQ^T still has M = 128, its rows 64..127
// read the next 64-row chunk of shared memory (the V tile) and are not read back.
template <int D_>
struct BwdTile {
    static constexpr int D = D_;
    static constexpr int DP = D <= 64 ? 64 : 128;       // row width in shared memory
    static constexpr int BN = 128;
    static constexpr int BQ = 64;
    static constexpr int NCH = DP / 64;
    static constexpr int QS = 3;                        // Q/dO/L/D ring stages
    static constexpr uint32_t K_CHUNK = BN * 128;
    static constexpr uint32_t Q_CHUNK = BQ * 128;
    static constexpr uint32_t KV_BYTES = BN * DP * 2;
    static constexpr uint32_t Q_BYTES = BQ * DP * 2;
    static constexpr uint32_t DS_BYTES = BQ * BN * 2;   // dS^T, [128 keys][64 queries] bf16
    static constexpr uint32_t STAGE_BYTES = BQ * D * 4; // dQ tile, fp32
    static constexpr uint32_t VEC_BYTES = BQ * 4;
    static constexpr uint32_t TM_DV = 0, TM_DK = 128, TM_ST = 256, TM_DPT = 320, TM_PD = 384,
                              TM_DQ = 448, TM_COLS = 512;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
    static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;
    static constexpr uint32_t OFF_DO = OFF_Q + QS * Q_BYTES;
    static constexpr uint32_t OFF_DS = OFF_DO + QS * Q_BYTES;
    static constexpr uint32_t OFF_STAGE = OFF_DS + DS_BYTES;  // one dS^T buffer
    static constexpr uint32_t OFF_L2 = OFF_STAGE + STAGE_BYTES;
    static constexpr uint32_t OFF_DELTA = OFF_L2 + QS * VEC_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_DELTA + QS * VEC_BYTES;
    // kv_full, q_full[QS], q_empty[QS], s_full, st_free, ds_full, pd_free, dq_full,
    // dq_empty, stg_free, stg_full, done (dq_full also tells the compute warps that
    // the dS^T buffer is free)
    static constexpr int NBAR = 1 + 2 * QS + 9;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int THREADS = 448;  // compute 0-7, dQ readout 8-11, TMA 12, MMA 13
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(Q_CHUNK % 1024 == 0 && DS_BYTES % 1024 == 0, "swizzle atoms must stay aligned");
    static_assert(D == 64 || D == 96 || D == 128, "head dim");
};

template <int D, bool CAUSAL, bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(448, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq,
                       const float *__restrict__ ws_lse2, const float *__restrict__ ws_delta,
                       float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv, int N,
                       int Npad, int BHkv, int H, int group, int head_group,
                       const int *__restrict__ cu_seqlens,
                  int total_tokens, float scale, float scale_log2, int *status,
                       unsigned long long limit_ns) {
    using T = BwdTile<D>;
    constexpr int BQ = T::BQ, QS = T::QS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t sK = base + T::OFF_K, sV = base + T::OFF_V;
    const uint32_t sQ = base + T::OFF_Q, sDO = base + T::OFF_DO;
    const uint32_t sDS = base + T::OFF_DS, sStage = base + T::OFF_STAGE;
    const uint32_t sL2 = base + T::OFF_L2, sDelta = base + T::OFF_DELTA;
    const uint32_t bar = base + T::OFF_BAR;
    const uint32_t bar_kv_full = bar;
    const uint32_t bar_q_full = bar + 8;                 // [QS]
    const uint32_t bar_q_empty = bar_q_full + 8 * QS;     // [QS]
    const uint32_t bar_s_full = bar_q_empty + 8 * QS;
    const uint32_t bar_st_free = bar_s_full + 8;
    const uint32_t bar_ds_full = bar_s_full + 16;
    const uint32_t bar_pd_free = bar_s_full + 24;
    const uint32_t bar_dq_full = bar_s_full + 32;
    const uint32_t bar_dq_empty = bar_s_full + 40;
    const uint32_t bar_stg_free = bar_s_full + 48;  // staging tile may be overwritten
    const uint32_t bar_stg_full = bar_s_full + 56;  // staging tile written by all 128 threads
    const uint32_t bar_done = bar_s_full + 64;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + T::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 4);
    float *stage_f = reinterpret_cast<float *>(gbase + T::OFF_STAGE);
    const float *l2_f = reinterpret_cast<const float *>(gbase + T::OFF_L2);
    const float *delta_f = reinterpret_cast<const float *>(gbase + T::OFF_DELTA);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTAs walk the key/value heads in groups of head_group (whose Q/dO then stay in
    // L2 together) and, within a group, the key blocks first: with a causal mask key
    // block 0 has the most query blocks, so low blockIdx = longest first.
    // Grouped-query attention: this CTA owns key/value head kvh (= b * Hkv + hk)
    // and accumulates dK, dV over the `group` query heads that read it, walking
    // their query blocks one head after the other.
    // SPLIT (small grids): two consecutive CTAs share a key block, each taking a
    // contiguous half of its query blocks, and add their dK, dV into zeroed outputs.
    const int part = SPLIT ? (int)(blockIdx.x & 1u) : 0;
    const unsigned bid = SPLIT ? blockIdx.x >> 1 : blockIdx.x;
    int kvh, kv0;
    if (!(VARLEN || !CAUSAL) || head_group >= BHkv) {
        kvh = bid % BHkv;
        kv0 = (bid / BHkv) * T::BN;
    } else {
        const int n_kb = (N + T::BN - 1) / T::BN;
        const int hgrp = (int)bid / (head_group * n_kb);
        const int hrem = (int)bid % (head_group * n_kb);
        const int hcnt = min(head_group, BHkv - hgrp * head_group);  // heads in this group
        kvh = hgrp * head_group + hrem % hcnt;
        kv0 = (hrem / hcnt) * T::BN;
    }
    // Keys and queries of this head: N, or with packed sequences (VARLEN: token-major
    // q, k, v, o, dO, dq, dk, dv, and N is the maximum length) the sequence's own
    // length, checked on the device.  A key block past the sequence's end has no work.
    const int hk = kvh % (H / group);
    int len = N, tok0 = 0;
    if constexpr (VARLEN) {
        const int b = kvh / (H / group);
        const int a = cu_seqlens[b], e = cu_seqlens[b + 1];
        if (a < 0 || e < a || e > total_tokens || e - a > N) {
            if (threadIdx.x == 0 && kv0 == 0 && hk == 0) {
                atomicCAS(status + 1, 0, SITE_BWD_BAD_SEQ);
                atomicExch(status, FA_ERR_BAD_INDEX);
            }
            len = 0;
        } else {
            len = e - a;
            tok0 = a;
        }
    }
    if (kv0 >= len) return;  // uniform across the CTA, before any barrier or TMEM use
    const int n_qb = (len + BQ - 1) / BQ;
    const int i_start = CAUSAL ? kv0 / BQ : 0;
    const int n_qit = n_qb - i_start;  // query blocks per query head
    const int n_all = group * n_qit;
    const int it0 = part ? n_all / 2 : 0;  // this CTA's blocks: [it0, it0 + n_it)
    const int n_it = SPLIT ? (part ? n_all - n_all / 2 : n_all / 2) : n_all;
    if (SPLIT && n_it == 0) return;  // uniform across the CTA, before any barrier or TMEM use
    const int qb_first = SPLIT ? it0 % n_qit : 0, gq_first = SPLIT ? it0 / n_qit : 0;
    const int bhq0 = (kvh / (H / group)) * H + (kvh % (H / group)) * group;
    // Block it is query block qb = it % n_qit of query head bhq0 + it / n_qit; the
    // loops below carry (qb, gq) as counters instead of dividing every block.

    if (threadIdx.x == 0) {
        mbar_init(bar_kv_full, 1);
        for (int s = 0; s < QS; ++s) {
            mbar_init(bar_q_full + 8 * s, 1);
            mbar_init(bar_q_empty + 8 * s, 1);
        }
        mbar_init(bar_s_full, 1);
        mbar_init(bar_st_free, 256);
        mbar_init(bar_ds_full, 256);
        mbar_init(bar_pd_free, 1);
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_empty, 128);
        mbar_init(bar_stg_free, 1);
        mbar_init(bar_stg_full, 128);
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), T::TM_COLS);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        if (VARLEN) tma_prefetch_desc(&tm_dq);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Guard g{status, abort_flag, limit_ns};

    if (warp == 12) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_kv_full, 2 * T::KV_BYTES);
            for (int c = 0; c < T::NCH; ++c) {
                tma_load_3d(sK + c * T::K_CHUNK, &tm_k, bar_kv_full, c * 64, VARLEN ? hk : kv0,
                            VARLEN ? tok0 + kv0 : kvh);
                tma_load_3d(sV + c * T::K_CHUNK, &tm_v, bar_kv_full, c * 64, VARLEN ? hk : kv0,
                            VARLEN ? tok0 + kv0 : kvh);
            }
            // the -L log2e and -D vectors come from the preprocess kernel
            griddep_wait();
            int issued = 0;
            for (int it = 0, qb = qb_first, gq = gq_first; it < n_it;
             ++it, (++qb == n_qit) ? (qb = 0, ++gq) : 0) {
                const int s = it % QS;
                const int q0 = (i_start + qb) * BQ;
                if (it >= QS && !mbar_wait(bar_q_empty + 8 * s, ((it / QS) - 1) & 1, g,
                                           SITE_BWD_LOAD_EMPTY))
                    break;
                const uint32_t fb = bar_q_full + 8 * s;
                mbar_arrive_expect_tx(fb, 2 * T::Q_BYTES + 2 * T::VEC_BYTES);
                for (int c = 0; c < T::NCH; ++c) {
                    tma_load_3d(sQ + s * T::Q_BYTES + c * T::Q_CHUNK, &tm_q, fb, c * 64, VARLEN ? (bhq0 + gq) % H : q0,
                                VARLEN ? tok0 + q0 : bhq0 + gq);
                    tma_load_3d(sDO + s * T::Q_BYTES + c * T::Q_CHUNK, &tm_do, fb, c * 64, VARLEN ? (bhq0 + gq) % H : q0,
                                VARLEN ? tok0 + q0 : bhq0 + gq);
                }
                const size_t voff = (size_t)(bhq0 + gq) * Npad + q0;
                bulk_load(sL2 + s * T::VEC_BYTES, ws_lse2 + voff, T::VEC_BYTES, fb);
                bulk_load(sDelta + s * T::VEC_BYTES, ws_delta + voff, T::VEC_BYTES, fb);
                ++issued;
            }
            if (*abort_flag) {
                volatile int never = 0;
                const Guard g2{status, &never, kWaitLimitNs};
                mbar_wait(bar_kv_full, 0, g2, SITE_BWD_DRAIN);
                for (int it = (issued > QS ? issued - QS : 0); it < issued; ++it)
                    mbar_wait(bar_q_full + 8 * (it % QS), (it / QS) & 1, g2, SITE_BWD_DRAIN);
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs this loop (warp-uniform); one elected lane issues.
        {
            constexpr uint32_t kIdescT = idesc_bf16_f32(128, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);   // dV, dK
            constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, BQ, true, true);    // dQ^T
            const uint64_t dK_k = sdesc_sw128(sK, 16, 1024);           // K, K-major (A of S^T)
            const uint64_t dV_k = sdesc_sw128(sV, 16, 1024);           // V, K-major (A of dP^T)
            const uint64_t dK_mn = sdesc_sw128(sK, T::K_CHUNK, 1024);  // K, MN-major (A of dQ^T)
            const uint64_t dDS = sdesc_sw128(sDS, T::DS_BYTES, 1024);  // dS^T, MN-major
            auto issue_st_dpt = [&](int it) {
                const int s = it % QS;
                const uint64_t dQ_k = sdesc_sw128(sQ + s * T::Q_BYTES, 16, 1024);
                const uint64_t dDO_k = sdesc_sw128(sDO + s * T::Q_BYTES, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks & 3) * 32, kc = ks >> 2;
                    mma_ss_elect(tmem + T::TM_ST, desc_add(dK_k, kc * T::K_CHUNK + koff),
                                 desc_add(dQ_k, kc * T::Q_CHUNK + koff), kIdescT, ks > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks & 3) * 32, kc = ks >> 2;
                    mma_ss_elect(tmem + T::TM_DPT, desc_add(dV_k, kc * T::K_CHUNK + koff),
                                 desc_add(dDO_k, kc * T::Q_CHUNK + koff), kIdescT, ks > 0 ? 1u : 0u);
                }
                tc_commit_elect(bar_s_full);
            };
            bool ok = mbar_wait_warp(bar_kv_full, 0, g, SITE_BWD_MMA_KV) &&
                      mbar_wait_warp(bar_q_full, 0, g, SITE_BWD_MMA_Q_FULL);
            tc_fence_after();
            if (ok) issue_st_dpt(0);
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % QS;
                // 1. S^T, dP^T of the next block, once the compute warps have read this one.
                if (it + 1 < n_it) {
                    ok = mbar_wait_warp(bar_st_free, it & 1, g, SITE_BWD_MMA_DS_FULL) &&
                         mbar_wait_warp(bar_q_full + 8 * ((it + 1) % QS), ((it + 1) / QS) & 1, g,
                                        SITE_BWD_MMA_Q_FULL);
                    if (!ok) break;
                    tc_fence_after();
                    issue_st_dpt(it + 1);
                }
                // 2. dV += P^T dO_i, dK += dS^T Q_i (K = 64 queries, 16 per step).
                if (!(ok = mbar_wait_warp(bar_ds_full, it & 1, g, SITE_BWD_MMA_DS_FULL))) break;
                tc_fence_after();
                const uint64_t dQ_mn = sdesc_sw128(sQ + s * T::Q_BYTES, T::Q_CHUNK, 1024);
                const uint64_t dDO_mn = sdesc_sw128(sDO + s * T::Q_BYTES, T::Q_CHUNK, 1024);
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks)
                    mma_ts_elect(tmem + T::TM_DV, tmem + T::TM_PD + ks * 8, desc_add(dDO_mn, ks * 2048),
                                 kIdescAcc, (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks)
                    mma_ts_elect(tmem + T::TM_DK, tmem + T::TM_PD + 32 + ks * 8,
                                 desc_add(dQ_mn, ks * 2048), kIdescAcc, (it > 0 || ks > 0) ? 1u : 0u);
                tc_commit_elect(bar_pd_free);
                tc_commit_elect(bar_q_empty + 8 * s);
                // 3. dQ^T[d][q] = sum_k K[k][d] dS^T[k][q] (K = 128 keys, 16 per step).
                if (it >= 1 &&
                    !(ok = mbar_wait_warp(bar_dq_empty, (it - 1) & 1, g, SITE_BWD_MMA_DQ_FREE)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < T::BN / 16; ++ks)
                    mma_ss_elect(tmem + T::TM_DQ, desc_add(dK_mn, ks * 2048), desc_add(dDS, ks * 2048),
                                 kIdescDQ, ks > 0 ? 1u : 0u);
                tc_commit_elect(bar_dq_full);
            }
            tc_commit_elect(bar_done);
            volatile int never = 0;
            const Guard g2{status, &never, kWaitLimitNs};
            mbar_wait_warp(bar_done, 0, g2, SITE_BWD_DRAIN);
        }
    } else if (warp < 8) {
        // ------------------------------------------------------- P^T and dS^T
        const int h = warp >> 2;          // query columns [32h, 32h + 32) of each block
        const int r = threadIdx.x & 127;  // key row within the block (TMEM lane)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int key = kv0 + r;
        bool ok = true;
        for (int it = 0, qb = qb_first, gq = gq_first; it < n_it;
             ++it, (++qb == n_qit) ? (qb = 0, ++gq) : 0) {
            const int s = it % QS;
            const int q0 = (i_start + qb) * BQ;
            ok = mbar_wait_warp(bar_s_full, it & 1, g, SITE_BWD_SOFTMAX_S_FULL);
            if (!ok) break;
            tc_fence_after();
            uint32_t sv[32], dpv[32];
            tmem_ld32(tmem + lane_base + T::TM_ST + 32 * h, sv);
            tmem_ld32(tmem + lane_base + T::TM_DPT + 32 * h, dpv);
            tmem_wait_ld(sv);
            tmem_wait_ld(dpv);
            tc_fence_before();
            mbar_arrive(bar_st_free);  // S^T / dP^T may now be overwritten
            const bool need_mask = (kv0 + T::BN > len) || (CAUSAL && q0 < kv0 + T::BN - 1);
            const float *l2v = l2_f + s * BQ + 32 * h;
            const float *dlv = delta_f + s * BQ + 32 * h;
            uint32_t pk[16], dk_[16];
            const uint64_t c2 = f32x2_splat(scale_log2);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                // the workspace holds -L log2e and -D, so both steps are packed pair
                // operations (the same roundings as s*c - L and dP - D)
                const float4 l4 = *reinterpret_cast<const float4 *>(l2v + e);
                const float4 d4 = *reinterpret_cast<const float4 *>(dlv + e);
                float p[4], ds[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    p[u] = __uint_as_float(sv[e + u]);
                    ds[u] = __uint_as_float(dpv[e + u]);
                }
                fma_f32x2(p[0], p[1], c2, l4.x, l4.y);
                fma_f32x2(p[2], p[3], c2, l4.z, l4.w);
                add_f32x2(ds[0], ds[1], d4.x, d4.y);
                add_f32x2(ds[2], ds[3], d4.z, d4.w);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    p[u] = ex2(p[u]);
                    if (need_mask) {
                        const int q = q0 + 32 * h + e + u;
                        if (key >= len || (CAUSAL && q < key)) p[u] = 0.f;
                    }
                }
                mul_f32x2(ds[0], ds[1], p[0], p[1]);
                mul_f32x2(ds[2], ds[3], p[2], p[3]);
                pk[e / 2] = pack_bf16(p[0], p[1]);
                pk[e / 2 + 1] = pack_bf16(p[2], p[3]);
                dk_[e / 2] = pack_bf16(ds[0], ds[1]);
                dk_[e / 2 + 1] = pack_bf16(ds[2], ds[3]);
            }
            // dS^T row r, queries [32h, 32h + 32): 4 swizzled 16-byte units (MN-major).
            // The single dS^T buffer is free once dQ^T of the previous block is done.
            if (it > 0 && !(ok = mbar_wait_warp(bar_dq_full, (it - 1) & 1, g,
                                                SITE_BWD_SOFTMAX_S_FULL)))
                break;
            uint8_t *ds_row = gbase + T::OFF_DS + r * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int unit = 4 * h + u;
                *reinterpret_cast<uint4 *>(ds_row + ((unit ^ (r & 7)) * 16)) =
                    make_uint4(dk_[4 * u], dk_[4 * u + 1], dk_[4 * u + 2], dk_[4 * u + 3]);
            }
            // PD is free once dV/dK of the previous block have read it.
            if (it > 0 && !(ok = mbar_wait_warp(bar_pd_free, (it - 1) & 1, g,
                                                SITE_BWD_SOFTMAX_S_FULL)))
                break;
            tc_fence_after();
            tmem_st16(tmem + lane_base + T::TM_PD + 16 * h, pk);
            tmem_st16(tmem + lane_base + T::TM_PD + 32 + 16 * h, dk_);
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_ds_full);
        }
        // ------------------------------------------------------- dK, dV epilogue
        // dK and dV are final once the last block's dV/dK products are done
        // (pd_free); the last dQ^T product, which reads only K and dS^T, still runs
        // while they leave through the Q/dO ring.
        ok = ok && mbar_wait_warp(bar_pd_free, (n_it - 1) & 1, g, SITE_BWD_EPILOGUE);
        if (ok) {
            tc_fence_after();
            // Each thread owns half a key row (d columns [64h, min(64h + 64, D))).  Rows are
            // staged in shared memory at a 528-byte pitch (16-byte writes without bank
            // conflicts; the Q/dO area is free once every MMA is done) and leave with
            // one bulk copy per half-row, so global writes are 256 contiguous bytes.
            constexpr uint32_t kPitch = T::DP * 4 + 16;  // 16-byte units shift by one per row
            static_assert(128 * kPitch <= T::OFF_DS - T::OFF_Q, "epilogue staging fits Q/dO area");
            uint8_t *stg = gbase + T::OFF_Q + r * kPitch + 256 * h;
            const uint32_t stg_s = sQ + r * kPitch + 256 * h;
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {  // 0: dV, 1: dK (times scale)
                const uint32_t tcol = (pass == 0 ? T::TM_DV : T::TM_DK) + 64 * h;
                const float mul = pass == 0 ? 1.f : scale;
                if (pass == 1) bulk_wait_group_read<0>();  // own staging row is reused
                constexpr int kHalf1 = (D - 64) / 32;  // 32-column loads of the second half
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (h == 1 && c >= kHalf1) break;
                    uint32_t a[32];
                    tmem_ld32(tmem + lane_base + tcol + 32 * c, a);
                    tmem_wait_ld(a);
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(stg + (32 * c + e) * 4) = make_float4(
                            __uint_as_float(a[e]) * mul, __uint_as_float(a[e + 1]) * mul,
                            __uint_as_float(a[e + 2]) * mul, __uint_as_float(a[e + 3]) * mul);
                }
                fence_proxy_async_smem();
                if (key < len && (h == 0 || D > 64)) {
                    const size_t krow =
                        VARLEN ? (size_t)(tok0 + key) * (H / group) + hk : (size_t)kvh * N + key;
                    float *dst = (pass == 0 ? dv : dk) + krow * D + 64 * h;
                    const uint32_t nb = h == 0 ? 256u : (uint32_t)(D - 64) * 4;
                    if constexpr (SPLIT)
                        bulk_reduce_add_f32(dst, stg_s, nb);
                    else
                        bulk_store(dst, stg_s, nb);
                }
                bulk_commit_group();
            }
            bulk_wait_group_read<0>();
        }
        tmem_wait_st();
    } else {
        // ------------------------------------------------------- dQ readout (warps 8-11)
        const int t = threadIdx.x - 256;  // TMEM lane = column d of dQ
        if (warp == 8) griddep_wait();    // dQ was zeroed by the preprocess kernel
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        for (int it = 0, qb = qb_first, gq = gq_first; it < n_it;
             ++it, (++qb == n_qit) ? (qb = 0, ++gq) : 0) {
            const int q0 = (i_start + qb) * BQ;
            ok = mbar_wait_warp(bar_dq_full, it & 1, g, SITE_BWD_DQ_FULL);
            if (!ok) break;
            tc_fence_after();
            uint32_t x0[32], x1[32];
            tmem_ld32(tmem + lane_base + T::TM_DQ, x0);
            tmem_ld32(tmem + lane_base + T::TM_DQ + 32, x1);
            tmem_wait_ld(x0);
            tmem_wait_ld(x1);
            tc_fence_before();
            mbar_arrive(bar_dq_empty);
            // dQ^T column t of the block's 64 rows -> row-major fp32 staging tile ->
            // one bulk asynchronous add into the block's contiguous global dQ rows.
            // The tile is free once the previous bulk add has read it; every sync here
            // is a bounded mbarrier wait, so an abort cannot strand a warp.
            if (warp == 8) {
                bulk_wait_group_read<0>();  // every lane's adds of the previous block
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_stg_free);
            }
            ok = mbar_wait_warp(bar_stg_free, it & 1, g, SITE_BWD_DQ_FULL);
            if (!ok) break;
            if (t < D) {  // rows of dQ^T past d are zero padding
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    stage_f[e * D + t] = __uint_as_float(x0[e]) * scale;
                    stage_f[(e + 32) * D + t] = __uint_as_float(x1[e]) * scale;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_stg_full);
            if (warp == 8) {
                bool ok0 = true;
                const int rows = min(BQ, len - q0);
                if constexpr (VARLEN) {
                    // token-major dQ: the block's rows of this head are H * D floats
                    // apart; one tiled add through the (d, heads, T) tensor map writes
                    // all of them.  Rows of the block past the sequence's end hold exact
                    // zeros (their P is 0), so adding them into the next sequence's rows
                    // leaves those unchanged; rows past T are skipped by the copy.
                    if (lane == 0) {
                        ok0 = mbar_wait(bar_stg_full, it & 1, g, SITE_BWD_DQ_FULL);
                        if (ok0) {
                            tma_reduce_add_3d(&tm_dq, sStage, 0, (bhq0 + gq) % H, tok0 + q0);
                            bulk_commit_group();
                        }
                    }
                } else {
                    if (lane == 0) {
                        ok0 = mbar_wait(bar_stg_full, it & 1, g, SITE_BWD_DQ_FULL);
                        if (ok0) {
                            bulk_reduce_add_f32(dq + ((size_t)(bhq0 + gq) * N + q0) * D, sStage,
                                                (uint32_t)(rows * D * 4));
                            bulk_commit_group();
                        }
                    }
                }
                ok0 = __shfl_sync(0xffffffffu, ok0 ? 1 : 0, 0) != 0;
                if (!ok0) {
                    ok = false;
                    break;
                }
            }
        }
        // Only the shared-memory reads of the last bulk add must finish before the
        // CTA retires; its global writes complete before the kernel does.
        if (warp == 8) bulk_wait_group_read<0>();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TM_COLS);
    }
}

template <int D, bool CAUSAL, bool VARLEN>
int launch_bwd_t(const BwdParams &p, cudaStream_t stream) {
    using W = BwdTile<D>;
    long long grid = (long long)((p.N + W::BN - 1) / W::BN) * (p.BH / p.group);
    // Small grids (single sequences with few heads; fixed layout): two CTAs per key
    // block, each over half of its query blocks, adding dK and dV into outputs
    // zeroed here, stream-ordered ahead of the preprocess kernel (so the main kernel
    // stays a programmatic dependent of the preprocess).  Causal: whenever the grid
    // is under one wave, since halving the longest key blocks shortens the critical
    // path; non-causal: only when the doubled grid still fits one wave (the CTAs are
    // all equally long, and a second wave of halves costs as much as the whole).
    const bool split = !VARLEN && (CAUSAL ? grid < p.num_sms : 2 * grid <= p.num_sms);
    if (split) {
        grid *= 2;
        const size_t kv_bytes = (size_t)(p.BH / p.group) * p.N * D * sizeof(float);
        if (cudaMemsetAsync(p.dk, 0, kv_bytes, stream) != cudaSuccess ||
            cudaMemsetAsync(p.dv, 0, kv_bytes, stream) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    {
        const long long rows = (long long)p.BH * p.Npad;
        long long blocks = (rows / 4 * 32 + 255) / 256;  // a warp per group of four rows
        const long long cap = (long long)p.num_sms * 16;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        fa_bwd_pre_kernel<D, VARLEN><<<(unsigned)blocks, 256, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16 *>(p.o),
            reinterpret_cast<const __nv_bfloat16 *>(p.dout), p.lse, p.ws_delta, p.ws_lse2, p.dq,
            p.N, p.Npad, p.BH, p.H, p.cu_seqlens, p.total_tokens);
        if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    }

    // Packed sequences and non-causal masks: groups of 8 key/value heads (measured:
    // varlen length mix 3.58 -> 2.55 ms, B8 H16 N2048 d64 non-causal +4.7%, B2 H16
    // N4096 d128 non-causal -0.5%).  Causal fixed layouts: one group, i.e. key block
    // major, which keeps the longest CTAs first (the kernel then skips the grouping
    // arithmetic; grouping measured -0.5% on B2 H16 N4096 d128 causal).
    const int head_group = (VARLEN || !CAUSAL) ? min(8, p.BH / p.group) : p.BH / p.group;
    if (grid > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    auto launch = [&](auto kern) -> int {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)W::SMEM_BYTES) != cudaSuccess)
            return FA_ERR_CUDA;
        // Launched as a programmatic dependent of the preprocess kernel: its CTAs set
        // up (barriers, tensor memory, K/V loads) while the preprocess finishes, and
        // wait for it only where they read its results.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(W::THREADS);
        cfg.dynamicSmemBytes = W::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p.tm_q, p.tm_k, p.tm_v, p.tm_do, p.tm_dq, p.ws_lse2,
                               p.ws_delta, p.dq, p.dk, p.dv, p.N, p.Npad, p.BH / p.group, p.H,
                               p.group, head_group, p.cu_seqlens, p.total_tokens, p.scale,
                               p.scale_log2, p.status, p.limit_ns) != cudaSuccess)
            return FA_ERR_CUDA;
        return FA_OK;
    };
    int rc;
    if constexpr (VARLEN)
        rc = launch(fa_bwd_kernel<D, CAUSAL, true, false>);
    else
        rc = split ? launch(fa_bwd_kernel<D, CAUSAL, false, true>)
                   : launch(fa_bwd_kernel<D, CAUSAL, false, false>);
    if (rc != FA_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
int launch_bwd_d(const BwdParams &p, cudaStream_t stream) {
    if (p.cu_seqlens)
        return p.causal ? launch_bwd_t<D, true, true>(p, stream) : launch_bwd_t<D, false, true>(p, stream);
    return p.causal ? launch_bwd_t<D, true, false>(p, stream) : launch_bwd_t<D, false, false>(p, stream);
}

}  // namespace

int bwd_block_q(int) { return BwdTile<128>::BQ; }

int launch_bwd(const BwdParams &p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_bwd_d<64>(p, stream);
        case 96: return launch_bwd_d<96>(p, stream);
        case 128: return launch_bwd_d<128>(p, stream);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
