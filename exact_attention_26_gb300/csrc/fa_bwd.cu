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
// adds them (padded rows get 0 and -inf, so their P is exactly 0), dQ := 0, and
// the main kernel's work counter := 0.
//
// Kernel 2 (fa_bwd_kernel): persistent CTAs (one per SM) over work items, an item
// being (batch * key/value head, block of 128 keys), each looping over blocks of
// 128 query rows; small grids instead give each item to two CTAs, one per half of
// its query blocks.  All products are tcgen05 MMAs
// with fp32 accumulators in tensor memory, computed in the transposed orientation
// so that a TMEM lane is a key:
//
//   S^T  = K_j Q_i^T        (A = K  smem K-major,  B = Q  smem K-major)
//   dP^T = V_j dO_i^T       (A = V,  B = dO)
//   dV  += P^T dO_i         (A = P^T from TMEM,  B = dO smem MN-major)
//   dK  += dS^T Q_i         (A = dS^T from TMEM, B = Q  smem MN-major)
//   dQ_i^T = K_j^T dS^T     (A = K smem MN-major, B = dS^T smem MN-major)
//
// dQ_i leaves tensor memory into registers and goes through shared memory into
// tiled bulk fp32 adds on the global dQ rows.  At the end of an item dK (times
// scale) and dV leave once, turned around in shared memory into whole-line stores.
//
// Warp roles (640 threads):
//   warps 0-7   P^T = exp2(S^T scale log2e - L log2e), dS^T = P^T o (dP^T - D)
//               (one key per thread, two warpgroups split a block's 128 queries),
//               written as bf16 to TMEM and dS^T to smem; the dV epilogue
//   warps 8-15  the dQ read-out and adds; the dK epilogue
//   warp 16     TMA producer: claims the items; K_j, Q_0, V_j, then Q_i (with L_i,
//               D_i) and dO_i per ring stage
//   warp 17     TMEM allocator; one elected lane issues every MMA and commit
//   warps 18-19 idle (the register pool is allocated per warpgroup)
#include <algorithm>

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
                      int H, const int *__restrict__ cu_seqlens, int total_tokens,
                      int *__restrict__ item_counter, float *__restrict__ zero_k,
                      float *__restrict__ zero_v, long long kv_elems) {
    // A warp takes RPW consecutive rows at a time (Npad is a multiple of 128, so they
    // share a head) and issues all their loads before any arithmetic: the kernel is
    // bound by HBM, and one row of O and dO per warp leaves too few bytes in flight.
    constexpr int RPW = 4;
    constexpr int PER = D / 32;  // elements per lane
    griddep_launch_dependents();  // the main kernel may set up while this one runs
    if (blockIdx.x == 0 && threadIdx.x == 0) *item_counter = 0;  // the main kernel's items
    // split key blocks: dK and dV := 0 (both parts of a key block add into them)
    for (long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < kv_elems;
         e += (long long)gridDim.x * blockDim.x * 4) {
        *reinterpret_cast<float4 *>(zero_k + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(zero_v + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
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
// A CTA owns 128 keys (one per TMEM lane) and walks blocks of 128 query rows, so
// every product is an M = 128, N = 128 tcgen05 MMA.  (With both operands in shared
// memory an MMA reads (M + N) x 32 bytes per K step, and at N = 64 that operand
// fetch, not the arithmetic, sets its time: 48 cycles instead of 32.  At N = 128
// the fetch and the arithmetic take the same 64 cycles.)
//
// Tensor memory (512 columns, d = 128): dV [0,128), dK [128,256), X [256,384),
// Y [384,512).  X holds S^T, then P^T as bf16 over its first half; Y holds dP^T,
// then dS^T as bf16, then dQ^T.  (d = 64: dV [0,64), dK [64,128), X [128,256),
// Y [256,384), and dQ^T in Z [384,512) of its own.)  Per block i the MMA thread
// issues
//
//   dP^T(i)     = V dO(i)^T   -> Y        once dQ^T(i-1) has been read out of Y
//                                         (d = 64: without waiting)
//   dV(i)      += P^T(i) dO(i)            A = P^T in X
//   S^T(i+1)    = K Q(i+1)^T  -> X        X is free once dV(i) has read P^T(i)
//   dK(i)      += dS^T(i) Q(i)            A = dS^T in Y
//   dQ^T(i)     = K^T dS^T(i) -> Y        B = dS^T from shared memory (d = 64: -> Z,
//                                         once dQ^T(i-1) has been read out of it)
//
// Warpgroups 0-1 compute dS(i) while dV(i) and S^T(i+1) run and P(i+1) while
// dK(i), dQ^T(i) and dP^T(i+1) run.  Warpgroups 2-3 read dQ^T(i) out of Y into
// registers (the tensor core waits only for that) and then add it into global dQ
// through tiled bulk adds.  The adds are bound by the L2's reduction rate (about
// 24 bytes per SM clock with every SM adding, by bulk copies or vector
// reductions; scalar per-thread reductions reach about 19), which is why they
// have warps of their own: their 64 KB per block then overlap the exponentials
// and the products instead of following them.
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
    static constexpr int BN = 128;                      // keys per CTA
    static constexpr int BQ = 128;                      // query rows per block
    static constexpr int NCH = DP / 64;
    static constexpr int QS = D <= 64 ? 4 : 2;          // Q ring stages (Q, -L log2e, -D)
    // dO ring stages.  dO(i) serves only dP^T(i) and dV(i), issued back to back, so
    // one stage leaves the copy of dO(i+1) the rest of the block's products.
    static constexpr int OS = D <= 64 ? 2 : 1;
    static constexpr uint32_t K_CHUNK = BN * 128;       // 64 columns of every key row
    static constexpr uint32_t Q_CHUNK = BQ * 128;
    static constexpr uint32_t KV_BYTES = BN * DP * 2;
    static constexpr uint32_t Q_BYTES = BQ * DP * 2;
    static constexpr uint32_t DS_CHUNK = BN * 128;      // dS^T: 64 queries of every key
    static constexpr uint32_t DS_BYTES = BN * BQ * 2;
    static constexpr uint32_t VEC_BYTES = BQ * 4;
    static constexpr uint32_t TM_DV = 0, TM_DK = DP, TM_X = 2 * DP, TM_Y = 2 * DP + 128,
                              TM_COLS = 512;
    // d = 64 leaves 128 columns spare: dQ^T gets its own (Z), so the next block's
    // dP^T need not wait for the dQ warps to read dQ^T out of Y; the next dQ^T waits
    // instead, a block later.  Wider heads share Y.
    static constexpr bool SEPQ = DP == 64;
    static constexpr uint32_t TM_QT = SEPQ ? TM_Y + 128 : TM_Y;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
    static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;
    static constexpr uint32_t OFF_DO = OFF_Q + QS * Q_BYTES;
    static constexpr uint32_t OFF_DS = OFF_DO + OS * Q_BYTES;  // dS^T (B of dQ^T)
    static constexpr uint32_t OFF_STG = OFF_DS + DS_BYTES;     // dQ staging, 4 KB per dQ warp
    static constexpr uint32_t STG_BYTES = 8 * 4096;
    static constexpr uint32_t OFF_L2 = OFF_STG + STG_BYTES;
    static constexpr uint32_t OFF_DELTA = OFF_L2 + QS * VEC_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_DELTA + QS * VEC_BYTES;
    // k_full, q_full[QS], q_empty[QS], o_full[OS], o_empty[OS], s_full, p_full,
    // dp_full, ds_full, dq_full, dq_empty, done, v_full, kv_empty, dv_free, dk_free,
    // item[2], item_read[2]
    static constexpr int NBAR = 1 + 2 * QS + 2 * OS + 15;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // TMEM base, abort flag, item[2]
    static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
    // The tiles need 1024-byte alignment (128-byte swizzle atoms).  At d = 128 the
    // layout leaves no room to align the start by hand: the kernel then requires
    // the dynamic shared memory to start aligned, and checks it.
    static constexpr uint32_t kMaxSmem = 227 * 1024;
    static constexpr uint32_t SMEM_BYTES =
        SMEM_USED + 1024 <= kMaxSmem ? SMEM_USED + 1024 : SMEM_USED;
    static constexpr int THREADS = 640;  // P/dS 0-7, dQ 8-15, TMA 16, MMA 17, 18-19 idle
    // Registers per thread after the warpgroups rebalance (launch: 96 each, a pool
    // of 5 x 128 x 96): P/dS warpgroups hold 64 fp32 P values per thread.  Chosen by
    // timing (B8 H16 N2048 d64 causal 0.290 ms vs 0.295 at 136 / 80; B4 H16 N4096
    // d96 causal 0.569 ms vs 0.581 at 144 / 72).
    static constexpr int LAUNCH_REGS = 96, REG_PDS = D == 96 ? 136 : 144, REG_DQ = D == 96 ? 80 : 72,
                         REG_MISC = 48;
    static_assert(2 * REG_PDS + 2 * REG_DQ + REG_MISC <= 5 * LAUNCH_REGS, "register pool");
    static_assert(REG_PDS % 8 == 0 && REG_DQ % 8 == 0 && REG_MISC % 8 == 0, "register targets");
    static_assert(SMEM_USED <= kMaxSmem, "shared memory budget");
    static_assert(Q_CHUNK % 1024 == 0 && DS_CHUNK % 1024 == 0 && KV_BYTES % 1024 == 0,
                  "swizzle atoms must stay aligned");
    static_assert(TM_Y + 128 <= TM_COLS && TM_QT + 128 <= TM_COLS, "tensor memory budget");
    static_assert(D == 64 || D == 96 || D == 128, "head dim");
};

template <int D, bool CAUSAL, bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(640, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq,
                  const float *__restrict__ ws_lse2, const float *__restrict__ ws_delta,
                  float *__restrict__ dk, float *__restrict__ dv, int N, int Npad, int BHkv,
                  int H, int group, int head_group, const int *__restrict__ cu_seqlens,
                  int total_tokens, float scale, float scale_log2, int *status,
                  unsigned long long limit_ns, int *__restrict__ item_counter) {
    using T = BwdTile<D>;
    constexpr int BQ = T::BQ, QS = T::QS, OS = T::OS;
    extern __shared__ __align__(1024) uint8_t smem_bwd[];
    const uint32_t raw = smem_u32(smem_bwd);
    const uint32_t base = (raw + 1023u) & ~1023u;
    if (base - raw + T::SMEM_USED > T::SMEM_BYTES) {
        // uniform across the CTA, before any barrier or TMEM use
        if (threadIdx.x == 0) {
            atomicCAS(status + 1, 0, SITE_BWD_SMEM_ALIGN);
            atomicExch(status, FA_ERR_UNSUPPORTED);
        }
        return;
    }
    uint8_t *gbase = smem_bwd + (base - raw);

    const uint32_t sK = base + T::OFF_K, sV = base + T::OFF_V;
    const uint32_t sQ = base + T::OFF_Q, sDO = base + T::OFF_DO;
    const uint32_t sDS = base + T::OFF_DS;
    const uint32_t sL2 = base + T::OFF_L2, sDelta = base + T::OFF_DELTA;
    const uint32_t bar = base + T::OFF_BAR;
    const uint32_t bar_k_full = bar;
    const uint32_t bar_q_full = bar + 8;               // [QS]
    const uint32_t bar_q_empty = bar_q_full + 8 * QS;  // [QS]
    const uint32_t bar_o_full = bar_q_empty + 8 * QS;  // [OS]
    const uint32_t bar_o_empty = bar_o_full + 8 * OS;  // [OS]
    const uint32_t bar_s_full = bar_o_empty + 8 * OS;
    const uint32_t bar_p_full = bar_s_full + 8;
    const uint32_t bar_dp_full = bar_s_full + 16;
    const uint32_t bar_ds_full = bar_s_full + 24;
    const uint32_t bar_dq_full = bar_s_full + 32;
    const uint32_t bar_dq_empty = bar_s_full + 40;
    const uint32_t bar_done = bar_s_full + 48;
    const uint32_t bar_v_full = bar_s_full + 56;
    const uint32_t bar_kv_empty = bar_s_full + 64;  // an item's last products are done
    const uint32_t bar_dv_free = bar_s_full + 72;   // the epilogue has read dV from TMEM
    const uint32_t bar_dk_free = bar_s_full + 80;   // ... dK
    const uint32_t bar_item = bar_s_full + 88;      // [2] the next item is published
    const uint32_t bar_item_read = bar_s_full + 104; // [2] every reading warp has read it
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + T::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 4);
    volatile int *item_slot = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 8);  // [2]
    const float *l2_f = reinterpret_cast<const float *>(gbase + T::OFF_L2);
    const float *delta_f = reinterpret_cast<const float *>(gbase + T::OFF_DELTA);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kTmaWarp = 16, kMmaWarp = 17;

    // CTAs walk the key/value heads in groups of head_group (whose Q/dO then stay in
    // L2 together) and, within a group, the key blocks first: with a causal mask key
    // block 0 has the most query blocks, so low blockIdx = longest first.
    // Grouped-query attention: this CTA owns key/value head kvh (= b * Hkv + hk)
    // and accumulates dK, dV over the `group` query heads that read it, walking
    // their query blocks one head after the other.
    // SPLIT (small grids): two consecutive CTAs share a key block, each taking a
    // contiguous half of its query blocks, and add their dK, dV into zeroed outputs.
    // Work items: key blocks of key/value heads, numbered as the grid used to be.
    // CTAs walk the key/value heads in groups of head_group (whose Q/dO then stay in
    // L2 together) and, within a group, the key blocks first: with a causal mask key
    // block 0 has the most query blocks, so a low item number is a long item.
    // Without SPLIT the CTAs are persistent (one per SM): CTA c starts with item c and
    // then takes the next unclaimed item from a counter in global memory (zeroed by
    // the preprocess kernel), so the CTAs finish together as if the hardware had
    // scheduled one CTA per item, and the next item's K/V loads and first products
    // overlap the previous item's dK/dV epilogue instead of a CTA's launch and setup.
    // The TMA warp claims the items and publishes each in a two-entry ring that every
    // role reads; all barrier phases are running counts across the items.
    // SPLIT (small grids): one item per CTA; two consecutive CTAs share a key block,
    // each taking a contiguous half of its query blocks, and add their dK, dV into
    // zeroed outputs.
    const int part = SPLIT ? (int)(blockIdx.x & 1u) : 0;
    const int n_kb = (N + T::BN - 1) / T::BN;
    const int n_items = SPLIT ? 1 : n_kb * BHkv;
    struct Item {
        int kvh, kv0, hk, len, tok0;
        int n_it;             // query blocks of this item (0: no work)
        int i_start, n_qit;   // first query block; query blocks per query head
        int qb_first, gq_first, bhq0;
    };
    auto decode_item = [&](int bid) -> Item {
        Item it;
        if (!(VARLEN || !CAUSAL) || head_group >= BHkv) {
            it.kvh = bid % BHkv;
            it.kv0 = (bid / BHkv) * T::BN;
        } else {
            const int hgrp = bid / (head_group * n_kb);
            const int hrem = bid % (head_group * n_kb);
            const int hcnt = min(head_group, BHkv - hgrp * head_group);  // heads in this group
            it.kvh = hgrp * head_group + hrem % hcnt;
            it.kv0 = (hrem / hcnt) * T::BN;
        }
        // Keys and queries of this head: N, or with packed sequences (VARLEN: token-
        // major q, k, v, o, dO, dq, dk, dv, and N is the maximum length) the
        // sequence's own length, checked on the device.  A key block past the
        // sequence's end has no work.
        it.hk = it.kvh % (H / group);
        it.len = N;
        it.tok0 = 0;
        if constexpr (VARLEN) {
            const int b = it.kvh / (H / group);
            const int a = cu_seqlens[b], e = cu_seqlens[b + 1];
            if (a < 0 || e < a || e > total_tokens || e - a > N) {
                // reported once, by the TMA thread that claims the sequence's first item
                if (threadIdx.x == kTmaWarp * 32 && it.kv0 == 0 && it.hk == 0) {
                    atomicCAS(status + 1, 0, SITE_BWD_BAD_SEQ);
                    atomicExch(status, FA_ERR_BAD_INDEX);
                }
                it.len = 0;
            } else {
                it.len = e - a;
                it.tok0 = a;
            }
        }
        const int n_qb = (it.len + BQ - 1) / BQ;
        it.i_start = CAUSAL ? it.kv0 / BQ : 0;
        it.n_qit = n_qb - it.i_start;
        const int n_all = it.kv0 < it.len ? group * it.n_qit : 0;
        const int it0 = part ? n_all / 2 : 0;  // this CTA's blocks: [it0, it0 + n_it)
        it.n_it = SPLIT ? (part ? n_all - n_all / 2 : n_all / 2) : n_all;
        it.qb_first = (SPLIT && it.n_qit > 0) ? it0 % it.n_qit : 0;
        it.gq_first = (SPLIT && it.n_qit > 0) ? it0 / it.n_qit : 0;
        it.bhq0 = (it.kvh / (H / group)) * H + (it.kvh % (H / group)) * group;
        // Block i of the item is query block qb = i % n_qit of query head
        // bhq0 + i / n_qit; the loops below carry (qb, gq) as counters.
        return it;
    };
    if constexpr (SPLIT) {
        // uniform across the CTA, before any barrier or TMEM use
        if (decode_item((int)(blockIdx.x >> 1)).n_it == 0) return;
    }

    if (threadIdx.x == 0) {
        mbar_init(bar_k_full, 1);
        mbar_init(bar_v_full, 1);
        mbar_init(bar_kv_empty, 1);
        for (int s = 0; s < QS; ++s) {
            mbar_init(bar_q_full + 8 * s, 1);
            mbar_init(bar_q_empty + 8 * s, 1);
        }
        for (int s = 0; s < OS; ++s) {
            mbar_init(bar_o_full + 8 * s, 1);
            mbar_init(bar_o_empty + 8 * s, 1);
        }
        mbar_init(bar_s_full, 1);
        mbar_init(bar_p_full, 256);
        mbar_init(bar_dp_full, 1);
        mbar_init(bar_ds_full, 256);
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_empty, 256);
        mbar_init(bar_done, 1);
        mbar_init(bar_dv_free, 256);
        mbar_init(bar_dk_free, 256);
        mbar_init(bar_item, 1);
        mbar_init(bar_item + 8, 1);
        // readers: the MMA warp, the 8 P/dS warps and the 8 dQ warps, one arrival each
        mbar_init(bar_item_read, 17);
        mbar_init(bar_item_read + 8, 17);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), T::TM_COLS);
        tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Guard g{status, abort_flag, limit_ns};
    // Item ri of this CTA (a running count): its number, or -1 after the last.  Each
    // reading warp marks the entry read (item_read), and the TMA warp rewrites the
    // entry of ri - 2 with ri only after all 17 have: no other chain orders the dQ
    // warps' read of an item with one block before the TMA warp runs two items on.
    auto next_item = [&](int ri, int &w) -> bool {
        if (!mbar_wait_warp<true>(bar_item + 8 * (ri & 1), (ri >> 1) & 1, g, SITE_BWD_ITEM)) return false;
        w = item_slot[ri & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_item_read + 8 * (ri & 1));
        return true;
    };
    // Each role rebalances its registers first thing in its own branch, so that the
    // compiler allocates the role's code within that role's budget.
    if (warp == kTmaWarp) {
        setmaxnreg_dec<T::REG_MISC>();
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int issued_q = 0, issued_o = 0;  // running over the CTA's items
            int n_k = 0, n_v = 0;            // items whose K, V were issued
            bool ok = true;
            // The CTA's next item with work (-1: none left).
            auto claim = [&](int ri) -> int {
                if constexpr (SPLIT) return ri == 0 ? (int)(blockIdx.x >> 1) : -1;
                int w = ri == 0 ? (int)blockIdx.x : -1;
                for (;;) {
                    if (w < 0) {
                        griddep_wait();  // the counter is zeroed by the preprocess kernel
                        w = (int)gridDim.x + atomicAdd(item_counter, 1);
                    }
                    if (w >= n_items) return -1;
                    if (decode_item(w).n_it > 0) return w;
                    w = -1;
                }
            };
            for (int ri = 0; ok; ) {
                const int w = claim(ri);
                // the entry's previous item (ri - 2) has been read by every role
                if (ri >= 2 && !(ok = mbar_wait<true>(bar_item_read + 8 * (ri & 1), ((ri - 2) >> 1) & 1, g,
                                                      SITE_BWD_ITEM)))
                    break;
                item_slot[ri & 1] = w;
                mbar_arrive(bar_item + 8 * (ri & 1));
                if (w < 0) break;
                const Item itm = decode_item(w);
                // K, then Q(0), then V: S^T(0) needs K and Q(0), and V is first read by
                // dP^T(0) after it, so an item's first product waits for two tiles.  K and V
                // of the previous item are free once its last dQ^T is done.
                if (ri > 0 && !(ok = mbar_wait<true>(bar_kv_empty, (ri - 1) & 1, g, SITE_BWD_LOAD_EMPTY)))
                    break;
                mbar_arrive_expect_tx(bar_k_full, T::KV_BYTES);
                for (int c = 0; c < T::NCH; ++c)
                    tma_load_3d(sK + c * T::K_CHUNK, &tm_k, bar_k_full, c * 64, VARLEN ? itm.hk : itm.kv0,
                                VARLEN ? itm.tok0 + itm.kv0 : itm.kvh);
                ++n_k;
                // the -L log2e and -D vectors come from the preprocess kernel
                if (ri == 0) griddep_wait();
                bool v_issued = false;
                for (int i = 0, qb = itm.qb_first, gq = itm.gq_first; i < itm.n_it;
                     ++i, (++qb == itm.n_qit) ? (qb = 0, ++gq) : 0) {
                    const int q0 = (itm.i_start + qb) * BQ;
                    const int yq = VARLEN ? (itm.bhq0 + gq) % H : q0;
                    const int zq = VARLEN ? itm.tok0 + q0 : itm.bhq0 + gq;
                    // Q(i) goes first: S^T(i) is issued a block ahead of dP^T(i) and dV(i),
                    // the products of dO(i).
                    // Q(i) with its -L log2e and -D: free once dK of the block QS before is done
                    const int gi = issued_q, qs = gi % QS;
                    if (gi >= QS && !(ok = mbar_wait<true>(bar_q_empty + 8 * qs, ((gi / QS) - 1) & 1, g,
                                                          SITE_BWD_LOAD_EMPTY)))
                        break;
                    const uint32_t fb = bar_q_full + 8 * qs;
                    mbar_arrive_expect_tx(fb, T::Q_BYTES + 2 * T::VEC_BYTES);
                    for (int c = 0; c < T::NCH; ++c)
                        tma_load_3d(sQ + qs * T::Q_BYTES + c * T::Q_CHUNK, &tm_q, fb, c * 64, yq, zq);
                    const size_t voff = (size_t)(itm.bhq0 + gq) * Npad + q0;
                    bulk_load(sL2 + qs * T::VEC_BYTES, ws_lse2 + voff, T::VEC_BYTES, fb);
                    bulk_load(sDelta + qs * T::VEC_BYTES, ws_delta + voff, T::VEC_BYTES, fb);
                    ++issued_q;
                    if (!v_issued) {
                        mbar_arrive_expect_tx(bar_v_full, T::KV_BYTES);
                        for (int c = 0; c < T::NCH; ++c)
                            tma_load_3d(sV + c * T::K_CHUNK, &tm_v, bar_v_full, c * 64,
                                        VARLEN ? itm.hk : itm.kv0, VARLEN ? itm.tok0 + itm.kv0 : itm.kvh);
                        v_issued = true;
                        ++n_v;
                    }
                    // dO(i): free once dV and dP^T of the block OS before are done
                    const int go = issued_o, os = go % OS;
                    if (go >= OS && !(ok = mbar_wait<true>(bar_o_empty + 8 * os, ((go / OS) - 1) & 1, g,
                                                          SITE_BWD_LOAD_EMPTY)))
                        break;
                    mbar_arrive_expect_tx(bar_o_full + 8 * os, T::Q_BYTES);
                    for (int c = 0; c < T::NCH; ++c)
                        tma_load_3d(sDO + os * T::Q_BYTES + c * T::Q_CHUNK, &tm_do, bar_o_full + 8 * os,
                                    c * 64, yq, zq);
                    ++issued_o;
                }
                ++ri;
            }
            if (*abort_flag) {
                // every copy this warp started lands before the CTA exits
                volatile int never = 0;
                const Guard g2{status, &never, kWaitLimitNs};
                if (n_k > 0) mbar_wait<true>(bar_k_full, (n_k - 1) & 1, g2, SITE_BWD_DRAIN);
                if (n_v > 0) mbar_wait<true>(bar_v_full, (n_v - 1) & 1, g2, SITE_BWD_DRAIN);
                for (int i = (issued_q > QS ? issued_q - QS : 0); i < issued_q; ++i)
                    mbar_wait<true>(bar_q_full + 8 * (i % QS), (i / QS) & 1, g2, SITE_BWD_DRAIN);
                for (int i = (issued_o > OS ? issued_o - OS : 0); i < issued_o; ++i)
                    mbar_wait<true>(bar_o_full + 8 * (i % OS), (i / OS) & 1, g2, SITE_BWD_DRAIN);
            }
        }
    } else if (warp == kMmaWarp) {
        setmaxnreg_dec<T::REG_MISC>();
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs this loop (warp-uniform); one elected lane issues.
        constexpr uint32_t kIdescT = idesc_bf16_f32(128, BQ, false, false);   // S^T, dP^T
        constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);   // dV, dK
        constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, BQ, true, true);    // dQ^T
        const uint64_t dK_k = sdesc_sw128(sK, 16, 1024);           // K, K-major (A of S^T)
        const uint64_t dV_k = sdesc_sw128(sV, 16, 1024);           // V, K-major (A of dP^T)
        const uint64_t dK_mn = sdesc_sw128(sK, T::K_CHUNK, 1024);  // K, MN-major (A of dQ^T)
        const uint64_t dDS = sdesc_sw128(sDS, T::DS_CHUNK, 1024);  // dS^T, MN-major (B of dQ^T)
        // S^T = K Q^T or dP^T = V dO^T: A (keys) and B (queries) both K-major.
        auto issue_t = [&](uint32_t dst, uint64_t a, uint32_t b_tile) {
            const uint64_t b = sdesc_sw128(b_tile, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t koff = (ks & 3) * 32, kc = ks >> 2;
                mma_ss_elect(tmem + dst, desc_add(a, kc * T::K_CHUNK + koff),
                             desc_add(b, kc * T::Q_CHUNK + koff), kIdescT, ks > 0 ? 1u : 0u);
            }
        };
        // dV += P^T dO or dK += dS^T Q: A (bf16, K = queries) from TMEM, where
        // warpgroup h put queries [64h, 64h + 64) at columns 64h .. 64h + 31; B MN-major.
        auto issue_acc = [&](uint32_t dst, uint32_t a_col, uint32_t b_tile, bool first) {
            const uint64_t b = sdesc_sw128(b_tile, T::Q_CHUNK, 1024);
#pragma unroll
            for (int ks = 0; ks < BQ / 16; ++ks)
                mma_ts_elect(tmem + dst, tmem + a_col + 64 * (ks >> 2) + 8 * (ks & 3),
                             desc_add(b, ks * 2048), kIdescAcc, (!first || ks > 0) ? 1u : 0u);
        };
        bool ok = true;
        int gb = 0;  // blocks of the CTA's earlier items
        for (int ri = 0; ok;) {
            int w = -1;
            if (!(ok = next_item(ri, w)) || w < 0) break;
            const Item itm = decode_item(w);
            const int n_it = itm.n_it;
            ok = mbar_wait_warp<true>(bar_k_full, ri & 1, g, SITE_BWD_MMA_KV) &&
                 mbar_wait_warp<true>(bar_q_full + 8 * (gb % QS), (gb / QS) & 1, g, SITE_BWD_MMA_Q_FULL);
            tc_fence_after();
            if (!ok) break;
            issue_t(T::TM_X, dK_k, sQ + (gb % QS) * T::Q_BYTES);
            tc_commit_elect(bar_s_full);
            for (int i = 0; ok && i < n_it; ++i) {
                const int it = gb + i;  // the block's running index
                const int qs = it % QS, os = it % OS;
                // 1. dP^T(it) into Y once dQ^T(it - 1) has been read out of it (shared Y)
                if (i == 0 && !(ok = mbar_wait_warp<true>(bar_v_full, ri & 1, g, SITE_BWD_MMA_KV))) break;
                if (!(ok = mbar_wait_warp<true>(bar_o_full + 8 * os, (it / OS) & 1, g, SITE_BWD_MMA_Q_FULL)))
                    break;
                if (!T::SEPQ && it > 0 &&
                    !(ok = mbar_wait_warp<true>(bar_dq_empty, (it - 1) & 1, g, SITE_BWD_MMA_DQ_FREE)))
                    break;
                tc_fence_after();
                issue_t(T::TM_Y, dV_k, sDO + os * T::Q_BYTES);
                tc_commit_elect(bar_dp_full);
                // 2. dV += P^T(it) dO(it); dO(it) is then done with.  The item's first dV
                //    overwrites the accumulator once the previous item's epilogue read it.
                if (!(ok = mbar_wait_warp<true>(bar_p_full, it & 1, g, SITE_BWD_MMA_DS_FULL))) break;
                if (i == 0 && ri > 0 &&
                    !(ok = mbar_wait_warp<true>(bar_dv_free, (ri - 1) & 1, g, SITE_BWD_MMA_DS_FULL)))
                    break;
                tc_fence_after();
                issue_acc(T::TM_DV, T::TM_X, sDO + os * T::Q_BYTES, i == 0);
                tc_commit_elect(bar_o_empty + 8 * os);
                // 3. S^T(it + 1) into X (P^T(it) is read by dV(it), issued before)
                if (i + 1 < n_it) {
                    const int qn = (it + 1) % QS;
                    if (!(ok = mbar_wait_warp<true>(bar_q_full + 8 * qn, ((it + 1) / QS) & 1, g,
                                                    SITE_BWD_MMA_Q_FULL)))
                        break;
                    tc_fence_after();
                    issue_t(T::TM_X, dK_k, sQ + qn * T::Q_BYTES);
                    tc_commit_elect(bar_s_full);
                }
                // 4. dK += dS^T(it) Q(it); Q(it) and its vectors are then done with.
                if (!(ok = mbar_wait_warp<true>(bar_ds_full, it & 1, g, SITE_BWD_MMA_DS_FULL))) break;
                if (i == 0 && ri > 0 &&
                    !(ok = mbar_wait_warp<true>(bar_dk_free, (ri - 1) & 1, g, SITE_BWD_MMA_DS_FULL)))
                    break;
                tc_fence_after();
                issue_acc(T::TM_DK, T::TM_Y, sQ + qs * T::Q_BYTES, i == 0);
                tc_commit_elect(bar_q_empty + 8 * qs);
                // 5. dQ^T(it)[d][q] = sum_k K[k][d] dS^T[k][q] into Y, or Z once dQ^T(it - 1)
                //    has been read out of it (K = 128 keys, 16 per step).  The next dP^T is
                //    issued after it, so the tensor pipe, in order, has read the dS^T tile
                //    before the P/dS warps (waiting for that dP^T) overwrite it.
                if (T::SEPQ && it > 0) {
                    if (!(ok = mbar_wait_warp<true>(bar_dq_empty, (it - 1) & 1, g, SITE_BWD_MMA_DQ_FREE)))
                        break;
                    tc_fence_after();
                }
#pragma unroll
                for (int ks = 0; ks < T::BN / 16; ++ks)
                    mma_ss_elect(tmem + T::TM_QT, desc_add(dK_mn, ks * 2048), desc_add(dDS, ks * 2048),
                                 kIdescDQ, ks > 0 ? 1u : 0u);
                tc_commit_elect(bar_dq_full);
            }
            // K and V are free for the next item once this item's products are done
            if (ok) tc_commit_elect(bar_kv_empty);
            gb += n_it;
            ++ri;
        }
        tc_commit_elect(bar_done);
        volatile int never = 0;
        const Guard g2{status, &never, kWaitLimitNs};
        mbar_wait_warp<true>(bar_done, 0, g2, SITE_BWD_DRAIN);
    } else if (warp >= 16) {
        setmaxnreg_dec<T::REG_MISC>();  // warps 18-19: no role
    } else {
        // ------------------------------------------------------- warps 0-15
        // Thread = key row r (TMEM lane).  Warpgroup wg: 0-1 compute P and dS of
        // query columns [64h, 64h + 64) of every block (h = wg): P = exp2(S^T scale
        // log2e - L log2e) into X, dS = P o (dP - D) into Y and into shared memory.
        // 2-3 read dQ^T columns [64h, 64h + 64) (h = wg - 2) out of Y and add them
        // into global dQ.  At the end of an item, 0-1 write dV and 2-3 dK.
        const int wg = warp >> 2;
        const int h = wg & 1;
        const int qt = warp & 3;          // TMEM lane quarter
        const int r = threadIdx.x & 127;  // key row within the block
        const uint32_t lane_base = (uint32_t)(qt * 32) << 16;
        bool ok = true;
        // ------------------------------------------------------- dK, dV epilogue
        auto epilogue = [&](const Item &itm) {
            // Every product of the item is done: dK and dV are final.  Warpgroups 0-1
            // take dV, 2-3 dK (times scale); each thread owns half a key row (d columns
            // [64h, min(64h + 64, D))).  A warp turns each 32-key by 32-column tile
            // around in a 4 KB buffer of its own (128-byte swizzle: 16-byte unit j of
            // row x at unit j ^ (x & 7), so both the row-wise writes and the transposed
            // reads are free of bank conflicts) and stores it with plain 16-byte stores,
            // eight lanes to a 128-byte row segment, so every store instruction writes
            // four whole lines.  The buffers are the warp's own quarter of its half of
            // the dS^T tile (P/dS warps: the item's last dQ^T is done, and the same warps
            // write the next item's dS^T) or its own dQ staging tile (dQ warps, after
            // their adds have read it): nothing waits on the epilogue but its own warp,
            // and the stores stay out of the bulk-copy queue the dQ adds keep busy.
            // The accumulator is free for the next item's first product once it is read.
            const int pass = wg >> 1;  // 0: dV, 1: dK
            const uint32_t tcol = (pass == 0 ? T::TM_DV : T::TM_DK) + 64 * h;
            const float mul = pass == 0 ? 1.f : scale;
            constexpr int kHalf1 = (D - 64) / 32;  // 32-column groups of the second half
            const int ncol = h == 0 ? 2 : kHalf1;
            uint8_t *wbuf = gbase + (pass == 0 ? T::OFF_DS + h * T::DS_CHUNK + qt * 4096u
                                               : T::OFF_STG + (warp - 8) * 4096u);
            const int tr = lane >> 3, tu = lane & 7;  // transposed: row 4k + tr, unit tu
            float *out = pass == 0 ? dv : dk;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (c >= ncol) break;
                uint32_t a[32];
                tmem_ld32(tmem + lane_base + tcol + 32 * c, a);
                tmem_wait_ld(a);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4 *>(wbuf + lane * 128 + ((j ^ (lane & 7)) << 4)) = make_float4(
                        __uint_as_float(a[4 * j]) * mul, __uint_as_float(a[4 * j + 1]) * mul,
                        __uint_as_float(a[4 * j + 2]) * mul, __uint_as_float(a[4 * j + 3]) * mul);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int x = 4 * k + tr;  // row of the tile
                    const float4 v = *reinterpret_cast<const float4 *>(wbuf + x * 128 + ((tu ^ (x & 7)) << 4));
                    const int key = itm.kv0 + 32 * qt + x;
                    if (key < itm.len) {
                        const size_t krow = VARLEN ? (size_t)(itm.tok0 + key) * (H / group) + itm.hk
                                                   : (size_t)itm.kvh * N + key;
                        float *dst = out + krow * D + 64 * h + 32 * c + 4 * tu;
                        if constexpr (SPLIT) {
                            atomicAdd(dst, v.x);
                            atomicAdd(dst + 1, v.y);
                            atomicAdd(dst + 2, v.z);
                            atomicAdd(dst + 3, v.w);
                        } else {
                            *reinterpret_cast<float4 *>(dst) = v;
                        }
                    }
                }
                __syncwarp();  // the buffer's reads are done before the next tile's writes
            }
            tc_fence_before();
            mbar_arrive(pass == 0 ? bar_dv_free : bar_dk_free);
        };
        if (wg < 2) {
            setmaxnreg_inc<T::REG_PDS>();
            const uint64_t c2 = f32x2_splat(scale_log2);
            float p[64];  // P of this thread's 64 queries, kept for dS
            int key = 0, len = 0, kv0 = 0;  // of the current item

            // P(it) from S^T(it) in X, in two 32-column halves.
            auto p_stage = [&](int it, int q0) -> bool {
                if (!mbar_wait_warp<true>(bar_s_full, it & 1, g, SITE_BWD_SOFTMAX_S_FULL)) return false;
                tc_fence_after();
                const bool need_mask = (kv0 + T::BN > len) || (CAUSAL && q0 < kv0 + T::BN - 1);
                const float *l2v = l2_f + (it % QS) * BQ + 64 * h;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sv[32];
                    tmem_ld32(tmem + lane_base + T::TM_X + 64 * h + 32 * c, sv);
                    tmem_wait_ld(sv);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        // the workspace holds -L log2e, so this is one packed FMA per pair
                        const float4 l4 = *reinterpret_cast<const float4 *>(l2v + 32 * c + e);
                        float *pp = p + 32 * c + e;
#pragma unroll
                        for (int u = 0; u < 4; ++u) pp[u] = __uint_as_float(sv[e + u]);
                        fma_f32x2(pp[0], pp[1], c2, l4.x, l4.y);
                        fma_f32x2(pp[2], pp[3], c2, l4.z, l4.w);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            pp[u] = ex2(pp[u]);
                            if (need_mask) {
                                const int q = q0 + 64 * h + 32 * c + e + u;
                                if (key >= len || (CAUSAL && q < key)) pp[u] = 0.f;
                            }
                        }
                        pk[e / 2] = pack_bf16(pp[0], pp[1]);
                        pk[e / 2 + 1] = pack_bf16(pp[2], pp[3]);
                    }
                    // P of columns [32c, 32c + 32) lands on columns [16c, 16c + 16),
                    // whose S values this thread has already read
                    tmem_st16(tmem + lane_base + T::TM_X + 64 * h + 16 * c, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar_p_full);
                return true;
            };

            // dS(it) = P o (dP - D) from dP^T(it) in Y: bf16 into Y (A of dK) and into
            // the shared dS^T tile (B of dQ^T).
            auto ds_stage = [&](int it) -> bool {
                if (!mbar_wait_warp<true>(bar_dp_full, it & 1, g, SITE_BWD_SOFTMAX_S_FULL)) return false;
                tc_fence_after();
                const float *dlv = delta_f + (it % QS) * BQ + 64 * h;
                uint8_t *ds_row = gbase + T::OFF_DS + h * T::DS_CHUNK + r * 128;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t dpv[32];
                    tmem_ld32(tmem + lane_base + T::TM_Y + 64 * h + 32 * c, dpv);
                    tmem_wait_ld(dpv);
                    uint32_t dsk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        // the workspace holds -D, so dP - D is a packed add
                        const float4 d4 = *reinterpret_cast<const float4 *>(dlv + 32 * c + e);
                        const float *pp = p + 32 * c + e;
                        float ds[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) ds[u] = __uint_as_float(dpv[e + u]);
                        add_f32x2(ds[0], ds[1], d4.x, d4.y);
                        add_f32x2(ds[2], ds[3], d4.z, d4.w);
                        mul_f32x2(ds[0], ds[1], pp[0], pp[1]);
                        mul_f32x2(ds[2], ds[3], pp[2], pp[3]);
                        dsk[e / 2] = pack_bf16(ds[0], ds[1]);
                        dsk[e / 2 + 1] = pack_bf16(ds[2], ds[3]);
                    }
                    tmem_st16(tmem + lane_base + T::TM_Y + 64 * h + 16 * c, dsk);
                    // dS^T row r, queries [64h + 32c, +32): 4 swizzled 16-byte units
                    // of the 64-query chunk h (MN-major)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int unit = 4 * c + u;
                        *reinterpret_cast<uint4 *>(ds_row + ((unit ^ (r & 7)) * 16)) = make_uint4(
                            dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar_ds_full);
                return true;
            };


            int gb = 0;  // blocks of the CTA's earlier items
            for (int ri = 0; ok; ++ri) {
                int w = -1;
                if (!(ok = next_item(ri, w)) || w < 0) break;
                const Item itm = decode_item(w);
                const int n_it = itm.n_it;
                kv0 = itm.kv0;
                len = itm.len;
                key = kv0 + r;
                ok = p_stage(gb, (itm.i_start + itm.qb_first) * BQ);
                for (int i = 0, qb = itm.qb_first; ok && i < n_it; ++i, (++qb == itm.n_qit) ? (qb = 0) : 0) {
                    ok = ds_stage(gb + i);
                    if (ok && i + 1 < n_it)
                        ok = p_stage(gb + i + 1, (itm.i_start + (qb + 1 == itm.n_qit ? 0 : qb + 1)) * BQ);
                }
                // every product of the item is done once its last dQ^T is
                ok = ok && mbar_wait_warp<true>(bar_dq_full, (gb + n_it - 1) & 1, g, SITE_BWD_EPILOGUE);
                if (!ok) break;
                tc_fence_after();
                // split: dV adds into the zeros the preprocess kernel wrote
                if constexpr (SPLIT) griddep_wait();
                epilogue(itm);
                gb += n_it;
            }
        } else {
            setmaxnreg_dec<T::REG_DQ>();
            griddep_wait();  // dQ is zeroed by the preprocess kernel before any add below
            // dQ(it): dQ^T rows [32 qt, +32) (d = 32 qt + lane) of queries [64h, 64h + 64)
            // leave Y into registers; then, scaled, each 32-query half goes through this
            // warp's 4 KB staging tile ([32 queries][32 columns] fp32) and one tiled
            // bulk add into global dQ (rows past the end of the sequence are skipped
            // by the copy, or hold exact zeros).
            const uint32_t s_stage = base + T::OFF_STG + (warp - 8) * 4096u;
            float *stage_f = reinterpret_cast<float *>(gbase + T::OFF_STG + (warp - 8) * 4096u);
            int tok0 = 0;  // of the current item
            auto stage_add = [&](const uint32_t(&x)[32], int row, int head) {
                if (lane == 0) bulk_wait_group_read<0>();  // the tile's previous add has read it
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 32; ++e) stage_f[e * 32 + lane] = __uint_as_float(x[e]) * scale;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (VARLEN)
                        tma_reduce_add_3d(&tm_dq, s_stage, 32 * qt, head, tok0 + row);
                    else
                        tma_reduce_add_3d(&tm_dq, s_stage, 32 * qt, row, head);
                    bulk_commit_group();
                }
            };
            int gb = 0, ri = 0;  // blocks and items of the CTA's earlier items
            for (; ok;) {
                int w = -1;
                if (!(ok = next_item(ri, w)) || w < 0) break;
                const Item itm = decode_item(w);
                const int n_it = itm.n_it;
                tok0 = itm.tok0;
                for (int i = 0, qb = itm.qb_first, gq = itm.gq_first; i < n_it;
                     ++i, (++qb == itm.n_qit) ? (qb = 0, ++gq) : 0) {
                    const int it = gb + i;
                    if (!(ok = mbar_wait_warp<true>(bar_dq_full, it & 1, g, SITE_BWD_DQ_FULL))) break;
                    tc_fence_after();
                    if (i == n_it - 1) {
                        // Every product of the item is done: dK leaves first (through the
                        // warp's staging tile, once its last add has read it), so the next
                        // item's first dK product need not wait for these dQ adds; the MMA
                        // warp's next dP^T waits for Y below instead, which is sooner.
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                        epilogue(itm);
                    }
                    uint32_t x0[32], x1[32];
                    tmem_ld32(tmem + lane_base + T::TM_QT + 64 * h, x0);
                    tmem_ld32(tmem + lane_base + T::TM_QT + 64 * h + 32, x1);
                    tmem_wait_ld(x0);
                    tmem_wait_ld(x1);
                    tc_fence_before();
                    mbar_arrive(bar_dq_empty);
                    if (32 * qt >= D) continue;  // rows of dQ^T past d are padding
                    const int row0 = (itm.i_start + qb) * BQ + 64 * h;
                    const int head = VARLEN ? (itm.bhq0 + gq) % H : itm.bhq0 + gq;
                    stage_add(x0, row0, head);
                    stage_add(x1, row0 + 32, head);
                }
                if (!ok) break;
                gb += n_it;
                ++ri;
            }
        }
        // The shared-memory reads of this thread's bulk copies and adds finish before
        // the CTA retires; their global writes complete before the kernel does.
        bulk_wait_group_read<0>();
        tmem_wait_st();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TM_COLS);
    }
}

template <int D, bool CAUSAL, bool VARLEN>
int launch_bwd_t(const BwdParams &p, cudaStream_t stream) {
    using W = BwdTile<D>;
    long long grid = (long long)((p.N + W::BN - 1) / W::BN) * (p.BH / p.group);
    // Small grids (single sequences with few heads; fixed layout): two CTAs per key
    // block, each over half of its query blocks, adding dK and dV into outputs the
    // preprocess kernel zeroes (the main kernel waits for it before its first add).
    // Zeroing there instead of two memsets ahead of it saves two launches on these
    // latency-bound shapes.  Causal: whenever the grid
    // is under one wave, since halving the longest key blocks shortens the critical
    // path; non-causal: only when the doubled grid still fits one wave (the CTAs are
    // all equally long, and a second wave of halves costs as much as the whole).
    const bool split = !VARLEN && (CAUSAL ? grid < p.num_sms : 2 * grid <= p.num_sms);
    // split: the preprocess kernel zeroes dK and dV (elements, a multiple of 4)
    const long long kv_elems = split ? (long long)(p.BH / p.group) * p.N * D : 0;
    if (split) grid *= 2;
    {
        const long long rows = (long long)p.BH * p.Npad;
        long long blocks = (rows / 4 * 32 + 255) / 256;  // a warp per group of four rows
        const long long cap = (long long)p.num_sms * 16;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        fa_bwd_pre_kernel<D, VARLEN><<<(unsigned)blocks, 256, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16 *>(p.o),
            reinterpret_cast<const __nv_bfloat16 *>(p.dout), p.lse, p.ws_delta, p.ws_lse2, p.dq,
            p.N, p.Npad, p.BH, p.H, p.cu_seqlens, p.total_tokens, p.ws_counter, p.dk, p.dv,
            kv_elems);
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
        if (ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)W::SMEM_BYTES) != FA_OK)
            return FA_ERR_CUDA;
        // The warpgroups' register budgets add up to the launch allocation; a build
        // that launches with any other count could leave a warpgroup waiting for
        // registers forever, so it is refused here.
        if (kernel_num_regs(reinterpret_cast<const void *>(kern)) != W::LAUNCH_REGS)
            return FA_ERR_UNSUPPORTED;
        // Launched as a programmatic dependent of the preprocess kernel: its CTAs set
        // up (barriers, tensor memory, K/V loads) while the preprocess finishes, and
        // wait for it only where they read its results.
        cudaLaunchConfig_t cfg = {};
        // Persistent CTAs (one per SM) over the items, or one CTA per half item (split).
        cfg.gridDim = dim3((unsigned)(split ? grid : std::min<long long>(grid, p.num_sms)));
        cfg.blockDim = dim3(W::THREADS);
        cfg.dynamicSmemBytes = W::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p.tm_q, p.tm_k, p.tm_v, p.tm_do, p.tm_dq, p.ws_lse2,
                               p.ws_delta, p.dk, p.dv, p.N, p.Npad, p.BH / p.group, p.H,
                               p.group, head_group, p.cu_seqlens, p.total_tokens, p.scale,
                               p.scale_log2, p.status, p.limit_ns, p.ws_counter) != cudaSuccess)
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
