// Forward pass of exact attention for sm_103a.
//
// One CTA owns NT tiles of 128 query rows of one (batch, head) (NT = 2 for
// d <= 128, 1 for d = 256) and streams the K/V tiles of that head through shared
// memory once for all of them ("FlashAttention-2: Why the Attention Bottleneck
// Wasn't Where Everyone Was Looking", section "FA2 change #2": outer loop over
// query blocks, inner loop over key/value blocks, the softmax state kept on chip).
// Per K/V tile j and query tile t:
//
//   S_t = Q_t K_j^T                   tcgen05.mma, fp32 accumulator in TMEM
//   m'  = max(m, rowmax(S_t) * scale) one thread per row, the whole row in registers
//   P_t = exp(S_t * scale - m')       written back to TMEM as bf16 over S_t
//   l'  = exp(m - m') l + rowsum(P_t)
//   O_t = exp(m - m') O_t + P_t V_j   rescale in TMEM, then tcgen05.mma (A = P_t from TMEM)
//
// which is the online-softmax update of "FlashAttention: Move Less, Not Compute
// Less", section "Tiling Is Easy; Softmax Couples the Entire Row", with the
// division by l deferred to the end ("FA2 change #1").  Exponentials run in base
// 2 with scale*log2(e) folded into one FMA.  The reference maximum m only moves
// when the new row maximum exceeds it by more than 2^8 (kRescaleLog2); a stale
// reference cancels exactly in O/l and in L, and keeps every P <= 256.
//
// With two tiles the MMA issue order per K/V tile is PV_0(j), S_0(j+1), PV_1(j),
// S_1(j+1): while the softmax warps of one tile work, the tensor core runs the
// other tile's products (the ping-pong of the course page "10 FlashAttention",
// section 6, mapped onto one MMA-issuing thread and two softmax warpgroups).
//
// Warp roles (NH softmax warpgroups per tile: 2 with two tiles at d <= 96, else 1):
//   warpgroup w < NT NH   softmax of tile t = w / NH over keys [h CB, h CB + CB) of
//                         each S row (h = w % NH, CB = BN / NH): thread r owns query
//                         row r (TMEM lane r); the two halves of a row trade their
//                         maxima once per K/V tile and their sums once per item
//                         through shared memory, so both take the same reference
//                         max; rescale of O_t and the epilogue O = O_t/l -> bf16, L
//                         split over the halves by 32-column chunks
//   warp 4 NT NH          TMEM allocator; one elected lane issues every MMA and
//                         commit (the whole warp runs the loop, warp-uniform)
//   warp 4 NT NH + 1      TMA producer (lane 0): Q tiles, then K_j/V_j into a ring
// Halving the row per thread halves the serial chain of each tile's softmax (load
// S, max, exponentials, pack P), the part of the per-tile step that the tensor core
// waits on; the exponential unit's throughput is unchanged.
//
// CTAs are persistent (one per SM): each walks a list of work items (NT query
// tiles of one head) longest first in snake order, with barrier phases carried
// across items.  The e4m3 variant (F8) runs the same pipeline with 8-bit operands
// in both products and P rounded to e4m3; packed sequences (VARLEN) read
// token-major tensors through (d, heads, tokens) tensor maps.
//
// Causal tiles above the diagonal are never loaded or multiplied; the diagonal
// and the ragged tail (keys >= N) are masked to -inf element by element, other
// tiles take no mask work ("The causal masking freebie").  A tile whose first row
// is past N is skipped; rows past N inside a tile compute on zero-filled Q rows
// and are not stored.
#include <algorithm>
#include <array>
#include <memory>
#include <type_traits>
#include <mutex>
#include <vector>

#include "fa_ptx.cuh"

namespace fa {
namespace {

// One 32-byte global store (sm_100+), a full L2 sector per thread; dst 32-byte
// aligned.  The epilogue writes each thread's O row with these: a warp's 16-byte
// stores to 32 different rows leave every sector half written.
__device__ __forceinline__ void st_global_v8(void *dst, const uint32_t *w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

// F8: Q, K and V arrive as e4m3 bytes (one scale per 128-row block of Q and of K,
// one per head of V) and P is rounded to e4m3 for the PV product; V comes
// transposed ([d][keys]) so that both products read K-major operands.
// ONE: a single 128-row tile per CTA (two S slots), for launches whose two-tile
// items would leave SMs idle; its per-step chain is shorter, so with more CTAs in
// flight the longest item finishes sooner.
template <int D, bool F8 = false, bool ONE = false>
struct FwdTile {
    static constexpr int EB = F8 ? 1 : 2;             // bytes per element
    static constexpr int NT = (D <= 128 && !ONE) ? 2 : 1;  // 128-row query tiles per CTA
    // keys per K/V tile: 64 at d = 256 (tensor memory).  (Two tiles at d = 64 with
    // 64-key tiles, which leaves room for two S slots per tile so that each tile's
    // next S is computed while its softmax runs, measured 4% slower non-causal and
    // 2% faster causal: both tiles' softmaxes then run in step and contend for the
    // exponential unit.)
    static constexpr int BN = (D == 256) ? 64 : 128;
    static constexpr int SB = (NT == 1) ? 2 : 1;      // S slots per tile
    static constexpr int NS = NT * SB;                // S slots in TMEM
    static constexpr int BM = 128;
    static constexpr int ROWS = NT * BM;              // query rows per CTA
    static constexpr int KV_BOX = fwd_kv_box_rows(D); // rows per K/V TMA box
    static constexpr int KS = (F8 || D == 64) ? 4 : 3;  // K ring stages
    static constexpr int VS = (F8 || D == 64) ? 4 : 2;  // V ring stages
    // Rows sit in shared memory as 128-byte swizzle chunks (64 bf16 or 128 e4m3
    // columns); d = 96 takes two bf16 chunks, the columns past d zero-filled by the
    // copy and never read by a product (S runs D/16 K steps, PV has N = D).
    static constexpr int CW = 128 / EB;               // columns per swizzle chunk
    static constexpr int DP = (D + CW - 1) / CW * CW; // row width in shared memory
    static constexpr int NCH = DP / CW;               // 128-byte swizzle chunks per row
    static constexpr int KSTEP = 32 / EB;             // K elements per MMA (32 bytes)
    static constexpr uint32_t Q_CHUNK = BM * 128;
    static constexpr uint32_t KV_CHUNK = BN * 128;
    static constexpr uint32_t Q_BYTES = BM * DP * EB;  // one query tile
    static constexpr uint32_t KV_BYTES = BN * DP * EB; // one of K_j, V_j (F8: V_j^T)
    // tensor memory columns: S slot u at BN u (fp32; the P of the keys of softmax
    // half h as bf16 pairs or e4m3 quadruples from column h CB of the slot on), then
    // O_t (fp32, D columns) at BN NS + D t
    static constexpr uint32_t TM_O0 = BN * NS;
    static constexpr uint32_t TM_COLS = 512;
    // shared memory layout (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + NT * Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KS * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + VS * KV_BYTES;
    // With two tiles and d <= 96 (bf16) each tile's softmax runs on NH = 2
    // warpgroups, one per half of the BN keys of an S row (CB columns each); the
    // halves trade their row maxima and row sums through a shared-memory exchange
    // guarded by bar_x[t].  (At d = 128 and in e4m3, whose tensor work per step is
    // larger, the split measured 2% and 6% slower: the MMA warp then shares its
    // scheduler with four busy softmax warps instead of two and issues late.)
    static constexpr int NH = (NT == 2 && D <= 96 && !F8) ? 2 : 1;  // softmax warpgroups per tile
    static constexpr int CB = BN / NH;                // S columns per softmax thread
    static constexpr int NWG = NT * NH;               // softmax warpgroups
    // q_full[NT], q_empty[NT], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    // s_full[NS], p_full[NS], o_full[NT], o_free[NT], pv_done[NT], mma_done, x[NT]
    static constexpr int NBAR = 2 * NT + 2 * KS + 2 * VS + 2 * NS + 4 * NT + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    // half exchange: fp32 [XB][NT][NH][BM]; two buffers, alternating by phase, where
    // the S slots are double-buffered (a half may then run a step ahead) and room
    // allows
    static constexpr int XB = (NH > 1 && SB == 2) ? 2 : 1;
    static constexpr uint32_t OFF_XCH = OFF_MISC + 16;
    static constexpr uint32_t SMEM_USED = OFF_XCH + (NH > 1 ? XB * NT * NH * BM * 4 : 0);
    // The tiles need 1024-byte alignment (128-byte swizzle atoms).  Where the layout
    // leaves no room to align the start by hand (d = 96 with two tiles) the
    // kernel requires the dynamic shared memory to start aligned, and checks it.
    static constexpr uint32_t kMaxSmem = 227 * 1024;
    static constexpr uint32_t SMEM_BYTES =
        SMEM_USED + 1024 <= kMaxSmem ? SMEM_USED + 1024 : SMEM_USED;
    static constexpr int WARP_MMA = 4 * NWG;
    static constexpr int WARP_LOAD = 4 * NWG + 1;
    // Two tiles (RB): a last warpgroup holds the MMA and TMA warps (and two idle
    // ones), and the warpgroups rebalance registers from the launch's even split
    // (registers are granted per four warps, so a 10-warp CTA would get no more per
    // thread than a 12-warp one): softmax threads hold CB fp32 scores and the P
    // they pack, the MMA and TMA warps little.
    static constexpr bool RB = (NT == 2);
    static constexpr int THREADS = 128 * NWG + (RB ? 128 : 64);
    static constexpr int LAUNCH_REGS = NH > 1 ? 96 : 168;
    static constexpr int REG_SOFTMAX = NH == 1 ? 224 : CB == 32 ? 104 : 112;
    static constexpr int REG_MISC = NH == 1 ? 56 : CB == 32 ? 64 : 32;
    static_assert(!RB || NWG * REG_SOFTMAX + REG_MISC <= (NWG + 1) * LAUNCH_REGS, "register pool");

    static_assert(D == 64 || D == 96 || D == 128 || D == 256, "head dim");
    static_assert(!F8 || (D == 128 && BN == 128), "e4m3 path: d = 128");
    static_assert(Q_CHUNK % 1024 == 0 && KV_CHUNK % 1024 == 0, "swizzle atoms must stay aligned");
    static_assert(TM_O0 + NT * D <= TM_COLS, "tensor memory budget");
    static_assert(BN % 64 == 0, "K/V tiles of whole 64-key groups");
    static_assert(SMEM_USED <= kMaxSmem, "shared memory budget");
    static_assert(CB == 32 || CB == 64 || CB == 128, "S columns per thread");
};

// VARLEN: packed sequences of different lengths, token-major: q, o [T][H][d],
// k, v [T][Hkv][d], lse [H][T]; sequence b holds tokens [cu_seqlens[b],
// cu_seqlens[b+1]).  The tensor maps are then (d, heads, T), so a box of 128 tokens
// of one head lands in shared memory exactly like a box of the fixed layout.
//
// F8: q_descale [BH][nqb] and k_descale [B*Hkv][nqb] hold one scale per 128-row
// block, v_descale [B*Hkv] one per head (nqb = ceil(N / 128)); S_t(j) is scaled
// by scale * q_descale(t) * k_descale(j) inside the exponent's FMA and O by
// v_descale / l in the epilogue.
//
// SPLIT (one query tile per CTA, fixed layout, bf16): the key range of every row
// block is cut into chunks of `chunk` K/V tiles ("FlashAttention-2: ...", section
// "FA2 change #2: Parallelize over sequence length": a single long sequence must
// still fill the GPU; the merge rule is the one of the course page "10
// FlashAttention", section "The decode variant: FlashDecoding").  A work item is
// then one chunk; a row block with one chunk writes O and L as usual, the others
// write their normalised partial O_s (fp32, ws_o [BH][N][s_max][D]) and
// L_s = m_s + ln l_s (ws_l [BH][N][s_max]), which fa_fwd_merge_kernel combines.
// Kernel argument carrying the balanced plan (n_cta = 0: none); launches that
// cannot cut key ranges take a one-int stand-in.
struct SegNone {
    int n_cta;
};
template <bool SPLIT>
using SegArg = typename std::conditional<SPLIT, FwdSegTable, SegNone>::type;

template <int D, bool CAUSAL, bool VARLEN, bool F8, bool ONE, bool SPLIT>
__global__ void __launch_bounds__(FwdTile<D, F8, ONE>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ out,
                  float *__restrict__ lse, int N, int BH, int H, int group, int n_cblocks,
                  const int *__restrict__ cu_seqlens, int total_tokens, float scale_log2,
                  const float *__restrict__ q_descale, const float *__restrict__ k_descale,
                  const float *__restrict__ v_descale, int nqb, int chunk,
                  float *__restrict__ ws_o, float *__restrict__ ws_l, int s_max, int *status,
                  unsigned long long limit_ns, const __grid_constant__ SegArg<SPLIT> tab) {
    using T = FwdTile<D, F8, ONE>;
    constexpr int NT = T::NT;
    constexpr int KS = T::KS;
    constexpr int VS = T::VS;
    // warpgroups with different register budgets cannot share a called function:
    // the waits' slow path is inlined where they rebalance
    constexpr bool kIn = T::RB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    if (base - raw + T::SMEM_USED > T::SMEM_BYTES) {
        // uniform across the CTA, before any barrier or TMEM use
        if (threadIdx.x == 0) {
            atomicCAS(status + 1, 0, SITE_FWD_SMEM_ALIGN);
            atomicExch(status, FA_ERR_UNSUPPORTED);
        }
        return;
    }
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t sQ = base + T::OFF_Q;
    const uint32_t sK = base + T::OFF_K;
    const uint32_t sV = base + T::OFF_V;
    const uint32_t bar_q_full = base + T::OFF_BAR;      // [NT]
    const uint32_t bar_q_empty = bar_q_full + 8 * NT;    // [NT]
    const uint32_t bar_k_full = bar_q_empty + 8 * NT;    // [KS]
    const uint32_t bar_k_empty = bar_k_full + 8 * KS;    // [KS]
    const uint32_t bar_v_full = bar_k_empty + 8 * KS;    // [VS]
    const uint32_t bar_v_empty = bar_v_full + 8 * VS;    // [VS]
    const uint32_t bar_s_full = bar_v_empty + 8 * VS;    // [NS]
    const uint32_t bar_p_full = bar_s_full + 8 * T::NS;  // [NS], per S slot like s_full
    const uint32_t bar_o_full = bar_p_full + 8 * T::NS;  // [NT]
    const uint32_t bar_o_free = bar_o_full + 8 * NT;     // [NT]
    const uint32_t bar_pv_done = bar_o_free + 8 * NT;    // [NT] two S slots per tile only
    const uint32_t bar_mma_done = bar_pv_done + 8 * NT;
    const uint32_t bar_x = bar_mma_done + 8;             // [NT] softmax half exchange
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + T::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + T::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Persistent schedule.  Work item w = ROWS query rows of one head; w runs over
    // (batch*head) fastest and, when causal, over row blocks from the last (longest)
    // to the first.  CTA c takes item r*G + c in even rounds r and r*G + G-1-c in
    // odd ones (G = gridDim.x), which visits every item once and evens out the
    // longest-first sizes.  Every role walks the same sequence; barrier phases are
    // running counts carried from one item to the next.
    static_assert(!SPLIT || (T::NT == 1 && !VARLEN && !F8), "split key ranges: one tile, bf16");
    const int n_kv_all = (N + T::BN - 1) / T::BN;  // fixed layout (SPLIT)
    const int ratio = T::ROWS / T::BN;               // K/V tiles per row block on the diagonal
    // SPLIT: chunks of the row blocks [0, c] together (c < n_cblocks - 1, whose key
    // ranges are not cut by N): sum over y = 1..c+1 of ceil(y ratio / chunk), chunk a
    // multiple of ratio.
    auto chunks_upto = [&](int c) -> int {
        const int cc = chunk / ratio, n = c + 1, q = n / cc, rr = n % cc;
        return cc * q * (q + 1) / 2 + (q + 1) * rr;
    };
    auto n_kv_of = [&](int cb) -> int {
        return CAUSAL ? min(n_kv_all, ((cb + 1) * T::ROWS + T::BN - 1) / T::BN) : n_kv_all;
    };
    // balanced plan (SPLIT, tab.n_cta > 0): CTA c runs the table's segments
    // [start[c], start[c + 1]) in order instead of the snake over even chunks
    const bool use_tab = SPLIT && tab.n_cta > 0;
    int per_bh = n_cblocks;  // work items per (batch, head)
    int last_chunks = 1;     // SPLIT: chunks of the last row block
    if constexpr (SPLIT) {
        if (!use_tab) {
            last_chunks = (n_kv_of(n_cblocks - 1) + chunk - 1) / chunk;
            per_bh = CAUSAL ? (n_cblocks > 1 ? chunks_upto(n_cblocks - 2) : 0) + last_chunks
                            : n_cblocks * last_chunks;
        }
    }
    const int n_items = per_bh * BH;
    const int G = (int)gridDim.x;
    int n_rounds = (n_items + G - 1) / G;
    if constexpr (SPLIT)
        if (use_tab) n_rounds = tab.max_per_cta;
    auto item_of = [&](int rnd) -> int {
        if constexpr (SPLIT) {
            if (use_tab) {
                const int idx = (int)tab.start[blockIdx.x] + rnd;
                return idx < (int)tab.start[blockIdx.x + 1] ? idx : -1;
            }
        }
        const int idx = rnd * G + ((rnd & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
        return idx < n_items ? idx : -1;
    };
    struct Item {
        int bh, kvh, cb, n_kv[NT], n_max;
        int len, tok0;  // rows of this head's sequence; its first token (packed layout)
        int kv_lo;      // first K/V tile of the item's key range
        int s, ns;      // SPLIT: chunk index, chunks of this row block
        int n_seg;      // SPLIT: K/V tiles of the item's key range (at most)
    };
    auto decode = [&](int w) {
        Item it;
        it.bh = w % BH;
        // grouped-query attention: query head h reads key/value head h / group
        it.kvh = (it.bh / H) * (H / group) + (it.bh % H) / group;
        it.cb = CAUSAL ? (n_cblocks - 1 - w / BH) : (w / BH);
        it.len = N;
        it.tok0 = 0;
        it.kv_lo = 0;
        it.s = 0;
        it.ns = 1;
        it.n_seg = chunk;
        if constexpr (SPLIT) {
          if (use_tab) {
            const uint32_t w0 = tab.seg[w][0], w1 = tab.seg[w][1];
            it.bh = (int)(w0 & 0xffffu);
            it.cb = (int)(w0 >> 16);
            it.kvh = (it.bh / H) * (H / group) + (it.bh % H) / group;
            it.kv_lo = (int)(w1 & 0xfffu);
            it.n_seg = (int)((w1 >> 12) & 0xfffu);
            it.s = (int)((w1 >> 24) & 0xfu);
            it.ns = (int)(w1 >> 28);
          } else {
            // items run row block by row block, the longest (last) first, chunks in
            // key order within a row block
            int r = w / BH;
            if (!CAUSAL) {
                it.cb = r / last_chunks;
                it.s = r % last_chunks;
                it.ns = last_chunks;
            } else if (r < last_chunks) {
                it.cb = n_cblocks - 1;
                it.s = r;
                it.ns = last_chunks;
            } else {
                // row blocks n_cblocks - 2 down to 0: row block c's chunks follow the
                // total - chunks_upto(c) chunks of the row blocks above it, so the item
                // lies in the smallest c whose count above is at most r (bisection)
                r -= last_chunks;
                const int total = chunks_upto(n_cblocks - 2);
                int lo = 0, hi = n_cblocks - 2;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (total - chunks_upto(mid) <= r) hi = mid; else lo = mid + 1;
                }
                it.cb = lo;
                const int before = total - chunks_upto(lo);
                it.s = r - before;
                it.ns = (n_kv_of(lo) + chunk - 1) / chunk;
            }
            it.kv_lo = it.s * chunk;
          }
        }
        if constexpr (VARLEN) {
            // cu_seqlens lives on the device, so it is checked here: a sequence that is
            // not inside [0, total_tokens) or is longer than the launch's maximum is
            // skipped and reported
            const int b = it.bh / H;
            const int a = cu_seqlens[b], e = cu_seqlens[b + 1];
            if (a < 0 || e < a || e > total_tokens || e - a > N) {  // N: the maximum length
                if (threadIdx.x == 0 && it.cb == 0 && (it.bh % H) == 0) {
                    atomicCAS(status + 1, 0, SITE_FWD_BAD_SEQ);
                    atomicExch(status, FA_ERR_BAD_INDEX);
                }
                it.len = 0;
            } else {
                it.len = e - a;
                it.tok0 = a;
            }
        }
        const int n_kv_seq = (it.len + T::BN - 1) / T::BN;
        it.n_max = 0;
#pragma unroll
        for (int t = 0; t < NT; ++t) {  // K/V tiles query tile t visits (0: past the end)
            const int row0 = it.cb * T::ROWS + t * T::BM;
            if (row0 >= it.len)
                it.n_kv[t] = 0;
            else
                it.n_kv[t] = CAUSAL ? min(n_kv_seq, (row0 + T::BM + T::BN - 1) / T::BN) : n_kv_seq;
            if constexpr (SPLIT) it.n_kv[t] = max(0, min(it.n_kv[t] - it.kv_lo, it.n_seg));
            it.n_max = max(it.n_max, it.n_kv[t]);
        }
        return it;
    };

    if (threadIdx.x == 0) {
        for (int t = 0; t < NT; ++t) {
            mbar_init(bar_q_full + 8 * t, 1);
            mbar_init(bar_q_empty + 8 * t, 1);
            mbar_init(bar_o_full + 8 * t, 1);
            mbar_init(bar_o_free + 8 * t, 128 * T::NH);
            mbar_init(bar_x + 8 * t, 4 * T::NH);  // one arrival per softmax warp of the tile
        }
        for (int u = 0; u < T::NS; ++u) {
            mbar_init(bar_s_full + 8 * u, 1);
            // P of a slot: one arrival per softmax thread of the slot's tile.  Per slot,
            // not per tile: with two slots a tile's softmax may finish P(j) and P(j+1)
            // before the MMA warp looks for P(j), and one barrier would then be two
            // phases ahead of its waiter, which a parity wait cannot tell apart.
            mbar_init(bar_p_full + 8 * u, 128 * T::NH);
        }
        for (int s = 0; s < KS; ++s) {
            mbar_init(bar_k_full + 8 * s, 1);
            mbar_init(bar_k_empty + 8 * s, 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(bar_v_full + 8 * s, 1);
            mbar_init(bar_v_empty + 8 * s, 1);
        }
        for (int t = 0; t < NT; ++t) mbar_init(bar_pv_done + 8 * t, 1);
        mbar_init(bar_mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == T::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), T::TM_COLS);
        tmem_relinquish();
    }
    if (warp == T::WARP_LOAD && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Guard g{status, abort_flag, limit_ns};

    if (warp == T::WARP_LOAD) {
        if constexpr (T::RB) setmaxnreg_dec<T::REG_MISC>();
        // ------------------------------------------------------- TMA producer
        // Per item: Q tiles (each once the previous item's last S MMA on that tile
        // has read it), then K_i ahead of V_{i-1}, since S needs K one step before
        // PV needs V.  The K/V rings run on across items.
        if (lane == 0) {
            int k_issued = 0, v_issued = 0;  // running counts over all items
            int q_issued[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) q_issued[t] = 0;
            bool ok = true;
            for (int rnd = 0; ok && rnd < n_rounds; ++rnd) {
                const int w = item_of(rnd);
                if (w < 0) continue;
                const Item itm = decode(w);
                auto load_kv = [&](const CUtensorMap *map, uint32_t ring, uint32_t full, int stage,
                                   int j, bool is_v) {
                    mbar_arrive_expect_tx(full + 8 * stage, T::KV_BYTES);
                    if (F8 && is_v) {  // V_j^T: D rows of BN keys, one box
                        tma_load_3d(ring + stage * T::KV_BYTES, map, full + 8 * stage, j * T::BN, 0,
                                    itm.kvh);
                        return;
                    }
                    static_assert(T::BN % T::KV_BOX == 0, "K/V tile of whole boxes");
                    for (int c = 0; c < T::NCH; ++c)
                        for (int rr = 0; rr < T::BN; rr += T::KV_BOX) {
                            const uint32_t dst = ring + stage * T::KV_BYTES + c * T::KV_CHUNK + rr * 128;
                            if constexpr (VARLEN)
                                tma_load_3d(dst, map, full + 8 * stage, c * T::CW, (itm.bh % H) / group,
                                            itm.tok0 + j * T::BN + rr);
                            else
                                tma_load_3d(dst, map, full + 8 * stage, c * T::CW, j * T::BN + rr, itm.kvh);
                        }
                };
                for (int t = 0; ok && t < NT; ++t) {
                    if (itm.n_kv[t] == 0) continue;
                    if (q_issued[t] > 0 && !(ok = mbar_wait<kIn>(bar_q_empty + 8 * t, (q_issued[t] - 1) & 1,
                                                            g, SITE_FWD_LOAD_KV_EMPTY)))
                        break;
                    mbar_arrive_expect_tx(bar_q_full + 8 * t, T::Q_BYTES);
                    for (int c = 0; c < T::NCH; ++c) {
                        const int row = itm.cb * T::ROWS + t * T::BM;
                        if constexpr (VARLEN)
                            tma_load_3d(sQ + t * T::Q_BYTES + c * T::Q_CHUNK, &tm_q,
                                        bar_q_full + 8 * t, c * T::CW, itm.bh % H, itm.tok0 + row);
                        else
                            tma_load_3d(sQ + t * T::Q_BYTES + c * T::Q_CHUNK, &tm_q,
                                        bar_q_full + 8 * t, c * T::CW, row, itm.bh);
                    }
                    ++q_issued[t];
                }
                for (int i = 0; ok && i <= itm.n_max; ++i) {
                    if (i < itm.n_max) {
                        const int gk = k_issued, ks = gk % KS;
                        if (gk >= KS && !(ok = mbar_wait<kIn>(bar_k_empty + 8 * ks, ((gk / KS) - 1) & 1, g,
                                                         SITE_FWD_LOAD_KV_EMPTY)))
                            break;
                        load_kv(&tm_k, sK, bar_k_full, ks, itm.kv_lo + i, false);
                        ++k_issued;
                    }
                    if (i >= 1) {
                        const int gv = v_issued, vs = gv % VS;
                        if (gv >= VS && !(ok = mbar_wait<kIn>(bar_v_empty + 8 * vs, ((gv / VS) - 1) & 1, g,
                                                         SITE_FWD_LOAD_KV_EMPTY)))
                            break;
                        load_kv(&tm_v, sV, bar_v_full, vs, itm.kv_lo + i - 1, true);
                        ++v_issued;
                    }
                }
            }
            if (*abort_flag) {
                // Let the copies already in flight land before the CTA exits.
                volatile int never = 0;
                const Guard g2{status, &never, kWaitLimitNs};
                for (int t = 0; t < NT; ++t)
                    if (q_issued[t] > 0)
                        mbar_wait<kIn>(bar_q_full + 8 * t, (q_issued[t] - 1) & 1, g2, SITE_FWD_DRAIN);
                for (int j = (k_issued > KS ? k_issued - KS : 0); j < k_issued; ++j)
                    mbar_wait<kIn>(bar_k_full + 8 * (j % KS), (j / KS) & 1, g2, SITE_FWD_DRAIN);
                for (int j = (v_issued > VS ? v_issued - VS : 0); j < v_issued; ++j)
                    mbar_wait<kIn>(bar_v_full + 8 * (j % VS), (j / VS) & 1, g2, SITE_FWD_DRAIN);
            }
        }
    } else if (warp == T::WARP_MMA) {
        if constexpr (T::RB) setmaxnreg_dec<T::REG_MISC>();
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs this loop (warp-uniform); one elected lane issues.
        {
            constexpr uint32_t kIdescS =
                F8 ? idesc_e4m3_f32(128, T::BN) : idesc_bf16_f32(128, T::BN, false, false);
            constexpr uint32_t kIdescO = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
            // S slot u = Q_t K_j^T from K stage ks: M = 128, N = BN, K = D.
            auto issue_s = [&](int t, int u, int ks_stage) {
                const uint64_t dq = sdesc_sw128(sQ + t * T::Q_BYTES, 16, 1024);
                const uint64_t dk = sdesc_sw128(sK + ks_stage * T::KV_BYTES, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / T::KSTEP; ++ks) {
                    const uint32_t koff = (ks & 3) * 32;  // 32 bytes of K per step
                    const uint64_t a = desc_add(dq, (ks >> 2) * T::Q_CHUNK + koff);
                    const uint64_t b = desc_add(dk, (ks >> 2) * T::KV_CHUNK + koff);
                    if constexpr (F8)
                        mma_ss_elect_f8(tmem + T::BN * u, a, b, kIdescS, ks > 0 ? 1u : 0u);
                    else
                        mma_ss_elect(tmem + T::BN * u, a, b, kIdescS, ks > 0 ? 1u : 0u);
                }
                tc_commit_elect(bar_s_full + 8 * u);
            };
            // O_t += P V from S slot u and V stage vs: M = 128, N = D, K = BN.  P sits
            // in TMEM as 32-bit columns of 2 bf16 or 4 e4m3 keys: 8 columns per step,
            // the keys of softmax half h from column h CB of the slot on.
            auto p_col = [&](int ks, int steps) -> uint32_t {
                const int per_half = steps / T::NH;
                return (uint32_t)((ks / per_half) * T::CB + (ks % per_half) * 8);
            };
            auto issue_pv = [&](int t, int u, int vs, bool first) {
                if constexpr (F8) {
                    // V_j^T is K-major: D rows of BN key bytes
                    const uint64_t dv = sdesc_sw128(sV + vs * T::KV_BYTES, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < T::BN / 32; ++ks)
                        mma_ts_elect_f8(tmem + T::TM_O0 + D * t, tmem + T::BN * u + p_col(ks, T::BN / 32),
                                        desc_add(dv, ks * 32), kIdescO, (!first || ks > 0) ? 1u : 0u);
                } else {
                    const uint64_t dv = sdesc_sw128(sV + vs * T::KV_BYTES, T::KV_CHUNK, 1024);
#pragma unroll
                    for (int ks = 0; ks < T::BN / 16; ++ks) {
                        const uint64_t b = desc_add(dv, ks * 2048);
                        mma_ts_elect(tmem + T::TM_O0 + D * t, tmem + T::BN * u + p_col(ks, T::BN / 16), b,
                                     kIdescO, (!first || ks > 0) ? 1u : 0u);
                    }
                }
            };
            auto wait_k = [&](int j) {
                const bool r = mbar_wait_warp<kIn>(bar_k_full + 8 * (j % KS), (j / KS) & 1, g,
                                         SITE_FWD_MMA_KV_FULL);
                tc_fence_after();
                return r;
            };
            auto wait_v = [&](int j) {
                const bool r = mbar_wait_warp<kIn>(bar_v_full + 8 * (j % VS), (j / VS) & 1, g,
                                         SITE_FWD_MMA_KV_FULL);
                tc_fence_after();
                return r;
            };
            bool ok = true;
            int kc = 0, vc = 0;  // K/V tiles consumed before the current item (running)
            int qc[NT], pc[NT], oc[NT];  // per tile: Q loads, P arrivals, items finished
#pragma unroll
            int gs[NT];  // per tile: S products issued before the current item (two slots)
#pragma unroll
            for (int t = 0; t < NT; ++t) qc[t] = pc[t] = oc[t] = gs[t] = 0;
            for (int rnd = 0; ok && rnd < n_rounds; ++rnd) {
                const int w = item_of(rnd);
                if (w < 0) continue;
                const Item itm = decode(w);
                if (itm.n_max == 0) continue;  // rows past a short sequence's end: no work
                if constexpr (T::SB == 1) {
                    // NT tiles, one S slot each: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ...
                    ok = wait_k(kc);
                    for (int t = 0; ok && t < NT; ++t) {
                        if (itm.n_kv[t] == 0) continue;
                        ok = mbar_wait_warp<kIn>(bar_q_full + 8 * t, qc[t] & 1, g, SITE_FWD_MMA_Q);
                        ++qc[t];
                        tc_fence_after();
                        if (!ok) break;
                        issue_s(t, t, kc % KS);
                        if (itm.n_kv[t] == 1) tc_commit_elect(bar_q_empty + 8 * t);
                    }
                    if (ok) tc_commit_elect(bar_k_empty + 8 * (kc % KS));
                    for (int j = 0; ok && j < itm.n_max; ++j) {
                        int last_pv = 0, last_s = -1;
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (j < itm.n_kv[t]) last_pv = t;
                            if (j + 1 < itm.n_kv[t]) last_s = t;
                        }
                        bool v_ready = false, k_ready = false;
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (!ok || j >= itm.n_kv[t]) continue;
                            ok = mbar_wait_warp<kIn>(bar_p_full + 8 * t, pc[t] & 1, g, SITE_FWD_MMA_P_FULL);
                            ++pc[t];
                            // The first PV of an item overwrites O_t: the previous item's
                            // epilogue must have read it.
                            if (ok && j == 0 && oc[t] > 0)
                                ok = mbar_wait_warp<kIn>(bar_o_free + 8 * t, (oc[t] - 1) & 1, g,
                                                    SITE_FWD_MMA_P_FULL);
                            tc_fence_after();
                            if (ok && !v_ready) ok = v_ready = wait_v(vc + j);
                            if (!ok) break;
                            issue_pv(t, t, (vc + j) % VS, j == 0);
                            if (t == last_pv) tc_commit_elect(bar_v_empty + 8 * ((vc + j) % VS));
                            if (j + 1 < itm.n_kv[t]) {
                                if (!k_ready) ok = k_ready = wait_k(kc + j + 1);
                                if (!ok) break;
                                issue_s(t, t, (kc + j + 1) % KS);
                                if (j + 2 == itm.n_kv[t]) tc_commit_elect(bar_q_empty + 8 * t);
                                if (t == last_s) tc_commit_elect(bar_k_empty + 8 * ((kc + j + 1) % KS));
                            } else {
                                tc_commit_elect(bar_o_full + 8 * t);  // O_t is final once this fires
                                ++oc[t];
                            }
                        }
                    }
                } else {
                    // Two S slots per tile (the g-th S of tile t in slot 2t + (g & 1)):
                    // S_t(j+2) is issued right after PV_t(j) frees its slot, so the tensor
                    // core computes it while the softmax works on S_t(j+1).  Per K/V step
                    // the tiles' products interleave: PV_0(j), S_0(j+2), PV_1(j), S_1(j+2).
                    auto slot = [&](int t, int gi) { return 2 * t + (gi & 1); };
                    for (int jj = 0; ok && jj < 2 && jj < itm.n_max; ++jj) {
                        if (!(ok = wait_k(kc + jj))) break;
                        for (int t = 0; ok && t < NT; ++t) {
                            if (jj >= itm.n_kv[t]) continue;
                            if (jj == 0) {
                                ok = mbar_wait_warp<kIn>(bar_q_full + 8 * t, qc[t] & 1, g, SITE_FWD_MMA_Q);
                                ++qc[t];
                                tc_fence_after();
                                if (!ok) break;
                            }
                            issue_s(t, slot(t, gs[t] + jj), (kc + jj) % KS);
                            if (jj + 1 == itm.n_kv[t]) tc_commit_elect(bar_q_empty + 8 * t);
                        }
                        if (ok) tc_commit_elect(bar_k_empty + 8 * ((kc + jj) % KS));
                    }
                    for (int j = 0; ok && j < itm.n_max; ++j) {
                        int last_pv = 0, last_s = -1;
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (j < itm.n_kv[t]) last_pv = t;
                            if (j + 2 < itm.n_kv[t]) last_s = t;
                        }
                        bool v_ready = false, k_ready = false;
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (!ok || j >= itm.n_kv[t]) continue;
                            const int gi = gs[t] + j;
                            ok = mbar_wait_warp<kIn>(bar_p_full + 8 * slot(t, gi), (gi >> 1) & 1, g,
                                                     SITE_FWD_MMA_P_FULL);
                            // The first PV of an item overwrites O_t: the previous item's
                            // epilogue must have read it.
                            if (ok && j == 0 && oc[t] > 0)
                                ok = mbar_wait_warp<kIn>(bar_o_free + 8 * t, (oc[t] - 1) & 1, g,
                                                         SITE_FWD_MMA_P_FULL);
                            tc_fence_after();
                            if (ok && !v_ready) ok = v_ready = wait_v(vc + j);
                            if (!ok) break;
                            issue_pv(t, slot(t, gi), (vc + j) % VS, j == 0);
                            tc_commit_elect(bar_pv_done + 8 * t);
                            if (t == last_pv) tc_commit_elect(bar_v_empty + 8 * ((vc + j) % VS));
                            if (j + 2 < itm.n_kv[t]) {
                                if (!k_ready) ok = k_ready = wait_k(kc + j + 2);
                                if (!ok) break;
                                issue_s(t, slot(t, gs[t] + j), (kc + j + 2) % KS);
                                if (j + 3 == itm.n_kv[t]) tc_commit_elect(bar_q_empty + 8 * t);
                                if (t == last_s) tc_commit_elect(bar_k_empty + 8 * ((kc + j + 2) % KS));
                            }
                            if (j + 1 == itm.n_kv[t]) {
                                tc_commit_elect(bar_o_full + 8 * t);  // O_t is final once this fires
                                ++oc[t];
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < NT; ++t) gs[t] += itm.n_kv[t];
                }
                kc += itm.n_max;
                vc += itm.n_max;
            }
            // Fires once every MMA issued above has completed (normal or aborted run).
            tc_commit_elect(bar_mma_done);
            volatile int never = 0;
            const Guard g2{status, &never, kWaitLimitNs};
            mbar_wait_warp<kIn>(bar_mma_done, 0, g2, SITE_FWD_DRAIN);
        }
    } else if (warp > T::WARP_LOAD) {
        if constexpr (T::RB) setmaxnreg_dec<T::REG_MISC>();  // warps with no role
    } else {
        if constexpr (T::RB) setmaxnreg_inc<T::REG_SOFTMAX>();
        // ------------------------------------------------------- softmax warpgroups
        // Warpgroup wg serves tile t = wg / NH and the CB keys [hc CB, hc CB + CB) of
        // every S row (hc = wg % NH); thread r owns TMEM lane r, query row r of the tile.
        const int wg = warp >> 2;
        const int t = wg / T::NH;
        const int hc = wg % T::NH;
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t t_o = tmem + lane_base + T::TM_O0 + D * t;
        // O rows are D * 2 bytes apart (a multiple of 32): 32-byte stores need only a
        // 32-byte aligned base (the boundary guarantees 16)
        const bool out_al32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
        // Half exchange (NH = 2): each thread publishes one value per phase of bar_x[t]
        // (its half's row maximum per K/V tile, its partial row sum per item) and reads
        // the other half's; both halves run the same sequence of phases.  A slot is
        // rewritten only after the other half has read it.  With two buffers (XB = 2,
        // alternating by phase) that holds by itself: a buffer is rewritten two phases
        // later, which the writer reaches only after the reader's next arrival.  With
        // one buffer (one S slot per tile) it holds within an item because the next
        // maximum follows S(j+1), which the MMA issues only after both halves' P(j);
        // across items a "read" phase after the row sums guards it.  Each half writes
        // its P over its own S columns, so the halves share no tensor memory.
        float *x_base = reinterpret_cast<float *>(gbase + T::OFF_XCH);
        auto x_slot = [&](int b, int h) { return x_base + ((b * NT + t) * T::NH + h) * T::BM + r; };
        uint32_t xph = 0;      // phases of bar_x[t] this thread has taken part in
        bool x_guard = false;  // one buffer: the last phase was a "read" mark not yet waited for
        auto x_arrive = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_x + 8 * t);
            ++xph;
        };
        auto x_wait_last = [&]() {
            return mbar_wait_warp<kIn>(bar_x + 8 * t, (xph - 1) & 1, g, SITE_FWD_SOFTMAX_S_FULL);
        };
        // publish v, wait for the other half's value of the same phase
        auto x_trade = [&](float v, float &other) -> bool {
            if (T::XB == 1 && x_guard && !x_wait_last()) return false;
            x_guard = false;
            const int b = (T::XB == 2) ? (int)(xph & 1) : 0;
            *x_slot(b, hc) = v;
            x_arrive();
            if (!x_wait_last()) return false;
            other = *x_slot(b, T::NH - 1 - hc);
            return true;
        };
        int sc = 0;  // S products of this tile consumed before the current item
        int oc = 0;  // items of this tile finished
        bool ok = true;
        for (int rnd = 0; ok && rnd < n_rounds; ++rnd) {
            const int w = item_of(rnd);
            if (w < 0) continue;
            const Item itm = decode(w);
            const int n_it = itm.n_kv[t];
            if (n_it == 0) continue;
            const int row0 = itm.cb * T::ROWS + t * T::BM;
            const int q_idx = row0 + r;
            float m_ref = -INFINITY;  // reference max, base-2 scaled units
            // Row sum in parts over keys [0, 64) and [64, 128) of each K/V tile, added
            // at the end: every layout (one thread or two halves per row) then rounds
            // the same way.  l: this thread's first part; l_hi: its second (CB = 128).
            float l = 0.f, l_hi = 0.f;
            // score -> base-2 exponent factor (F8: times the block scales of Q_t, K_j)
            float c_q = scale_log2;
            if constexpr (F8) c_q *= q_descale[(size_t)itm.bh * nqb + row0 / T::BM];
            for (int j = 0; j < n_it; ++j) {
                const int gsj = sc + j;                                     // running S index
                const int u = (T::SB == 1) ? t : (2 * t + (gsj & 1));       // S slot
                const uint32_t par = (T::SB == 1) ? (gsj & 1) : ((gsj >> 1) & 1);
                const uint32_t t_s = tmem + lane_base + T::BN * u;
                float c_s = c_q;
                if constexpr (F8) c_s *= __ldg(k_descale + (size_t)itm.kvh * nqb + itm.kv_lo + j);
                ok = mbar_wait_warp<kIn>(bar_s_full + 8 * u, par, g, SITE_FWD_SOFTMAX_S_FULL);
                if (!ok) break;
                tc_fence_after();
                constexpr int CB = T::CB;
                uint32_t sr[CB / 32][32];
#pragma unroll
                for (int c = 0; c < CB / 32; ++c) tmem_ld32(t_s + hc * CB + c * 32, sr[c]);
#pragma unroll
                for (int c = 0; c < CB / 32; ++c) tmem_wait_ld(sr[c]);
                float s[CB];
#pragma unroll
                for (int c = 0; c < CB / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(sr[c][e]);

                const int kv0 = (itm.kv_lo + j) * T::BN;  // first key of the tile
                const int len = itm.len;
                const bool need_mask = (kv0 + T::BN > len) || (CAUSAL && kv0 + T::BN - 1 > row0);
                if (need_mask) {
                    const int lim = CAUSAL ? min(len, q_idx + 1) : len;  // keys [0, lim) are visible
                    const int k0 = kv0 + hc * CB;
#pragma unroll
                    for (int c = 0; c < CB; ++c)
                        if (k0 + c >= lim) s[c] = -INFINITY;
                }
                // Row max and row sum as two independent partial chains: one thread
                // owns CB columns of the row, and a single chain of CB dependent
                // operations would be CB latencies long.  Three-input max and packed
                // fp32-pair FMA/add halve the instruction count (the issue slots of the
                // softmax warps are the scarce resource); the sums keep the even/odd
                // split per 64 keys, so the rounding is that of two scalar chains.
                // (d = 256, whose 64-key tiles leave the softmax less to do than the
                // tensor core, measured 1.4% faster with the scalar forms.)
                // Measured and not kept: exponentials against the previous reference
                // max with this tile's max found in the same pass (the pass repeated
                // from S in TMEM when the max moves): the pass grew by what the
                // separate max took, since the exponential pass is throughput-bound.
                constexpr bool kPacked = D != 256;
                float mp0 = -INFINITY, mp1 = -INFINITY;
                static_assert(CB % 4 == 0, "max chains take four columns per step");
#pragma unroll
                for (int c = 0; c < CB; c += 4) {
                    mp0 = fmax3(mp0, s[c], s[c + 1]);
                    mp1 = fmax3(mp1, s[c + 2], s[c + 3]);
                }
                float mx = fmaxf(mp0, mp1);
                if constexpr (T::NH > 1) {
                    // the row maximum over both halves; both then take the same steps
                    float mo;
                    if (!(ok = x_trade(mx, mo))) break;
                    mx = fmaxf(mx, mo);
                }
                const float m_tile = mx * c_s;
                float alpha = 1.f;
                const bool move = m_tile > m_ref + kRescaleLog2;
                if (move) {
                    alpha = ex2(m_ref - m_tile);
                    m_ref = m_tile;
                }
                float sp0 = 0.f, sp1 = 0.f, sq0 = 0.f, sq1 = 0.f;
                if constexpr (kPacked) {
                    const uint64_t c2 = f32x2_splat(c_s), nm2 = f32x2_splat(-m_ref);
#pragma unroll
                    for (int c = 0; c < CB; c += 2) {
                        fma_f32x2(s[c], s[c + 1], c2, nm2);
                        s[c] = ex2(s[c]);
                        s[c + 1] = ex2(s[c + 1]);
                        if (c < 64)
                            add_f32x2(sp0, sp1, s[c], s[c + 1]);
                        else
                            add_f32x2(sq0, sq1, s[c], s[c + 1]);
                    }
                } else {
                    const float neg_m = -m_ref;
#pragma unroll
                    for (int c = 0; c < CB; c += 2) {
                        s[c] = ex2(fmaf(s[c], c_s, neg_m));
                        s[c + 1] = ex2(fmaf(s[c + 1], c_s, neg_m));
                        sp0 += s[c];
                        sp1 += s[c + 1];
                    }
                }
                l = l * alpha + (sp0 + sp1);
                if constexpr (CB > 64) l_hi = l_hi * alpha + (sq0 + sq1);
                // P over the first columns of this thread's own CB S columns (keys in
                // order): e4m3 quadruples (P <= 2^8 with the reference max, inside
                // e4m3's range) or bf16 pairs
                if constexpr (F8) {
                    uint32_t pk[CB / 4];
#pragma unroll
                    for (int e = 0; e < CB / 4; ++e)
                        pk[e] = pack_e4m3x4(s[4 * e], s[4 * e + 1], s[4 * e + 2], s[4 * e + 3]);
                    if constexpr (CB / 4 == 32)
                        tmem_st32(t_s + hc * CB, pk);
                    else
                        tmem_st16(t_s + hc * CB, pk);
                } else if constexpr (CB >= 64) {
#pragma unroll
                    for (int c = 0; c < CB / 64; ++c) {
                        uint32_t pk[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            pk[e] = pack_bf16(s[c * 64 + 2 * e], s[c * 64 + 2 * e + 1]);
                        tmem_st32(t_s + hc * CB + c * 32, pk);
                    }
                } else {
                    uint32_t pk[CB / 2];
#pragma unroll
                    for (int e = 0; e < CB / 2; ++e) pk[e] = pack_bf16(s[2 * e], s[2 * e + 1]);
                    static_assert(CB / 2 == 16, "P words per thread");
                    tmem_st16(t_s + hc * CB, pk);
                }
                if (j > 0 && __any_sync(0xffffffffu, move)) {
                    // O_t <- alpha O_t for this warp's 32 rows (alpha = 1 on rows that kept
                    // m), after P is stored so the S registers are free; the halves take
                    // alternate 32-column chunks.  PV(j-1) must be complete: with one
                    // slot per tile S(j) was issued after it; with two slots it is
                    // awaited here.  PV(j) waits for the arrive below.
                    if (T::SB == 2 && !mbar_wait_warp<kIn>(bar_pv_done + 8 * t, (gsj - 1) & 1, g,
                                                      SITE_FWD_SOFTMAX_S_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = hc; c < D / 32; c += T::NH) {
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
                mbar_arrive(bar_p_full + 8 * u);
            }
            if (!ok) break;
            sc += n_it;
            // --------------------------------------------------- epilogue of this item
            ok = mbar_wait_warp<kIn>(bar_o_full + 8 * t, oc & 1, g, SITE_FWD_EPILOGUE_O_FULL);
            if (!ok) break;
            tc_fence_after();
            if constexpr (T::NH > 1) {
                // the whole row sum (the same sum, in the same order, in both halves),
                // then mark the other half's slot as read
                float lo;
                if (!(ok = x_trade(l, lo))) break;
                l = (hc == 0) ? l + lo : lo + l;
                if constexpr (T::XB == 1) {
                    x_arrive();
                    x_guard = true;
                }
            } else if constexpr (T::CB > 64) {
                l = l + l_hi;
            }
            const float inv_l = (F8 ? v_descale[itm.kvh] : 1.f) / l;
            __nv_bfloat16 *orow =
                VARLEN ? out + ((size_t)(itm.tok0 + q_idx) * H + (itm.bh % H)) * D
                       : out + ((size_t)itm.bh * (size_t)N + (size_t)q_idx) * D;
            if (SPLIT && itm.ns > 1) {
                // one chunk of a cut key range: the normalised partial O_s in fp32 and
                // its L_s, for the merge kernel
                const size_t prow = ((size_t)itm.bh * (size_t)N + (size_t)q_idx) * s_max + itm.s;
                float *prow_o = ws_o + prow * D;
#pragma unroll 1
                for (int c = hc; c < D / 32; c += T::NH) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld(o);
                    if (c + T::NH >= D / 32) {
                        tc_fence_before();
                        mbar_arrive(bar_o_free + 8 * t);
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
                    if (q_idx < itm.len) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) st_global_v8(prow_o + c * 32 + 8 * e, o + 8 * e);
                    }
                }
                if (hc == 0 && q_idx < itm.len) ws_l[prow] = (m_ref + lg2(l)) * kLn2;
                ++oc;
                continue;
            }
            // 32 columns of O: scaled, packed to bf16 and stored
            auto store_chunk = [&](int c, const uint32_t(&o)[32]) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l,
                                      __uint_as_float(o[2 * e + 1]) * inv_l);
                if (q_idx < itm.len) {
                    if (out_al32) {  // two full 32-byte sectors per thread
                        st_global_v8(orow + c * 32, pk);
                        st_global_v8(orow + c * 32 + 16, pk + 8);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    }
                }
            };
            if constexpr (T::NH == 1 && D == 128 && !F8) {
                // one softmax warpgroup per tile at d = 128 (bf16): the four 32-column
                // loads of O are in flight before one wait, and O is released before the
                // stores (measured: B2 H16 N4096 non-causal -1%, B1 H16 N16384 causal
                // -0.5%; the e4m3 kernel was 2% slower this way and keeps one load at a
                // time)
                uint32_t oall[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(t_o + c * 32, oall[c]);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_wait_ld(oall[c]);
                tc_fence_before();
                mbar_arrive(bar_o_free + 8 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c) store_chunk(c, oall[c]);
            } else {
#pragma unroll 1
                for (int c = hc; c < D / 32; c += T::NH) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld(o);
                    if (c + T::NH >= D / 32) {
                        // O_t has been read: the next item's first PV may overwrite it.
                        tc_fence_before();
                        mbar_arrive(bar_o_free + 8 * t);
                    }
                    store_chunk(c, o);
                }
            }
            if (hc == 0 && q_idx < itm.len) {
                const size_t li = VARLEN ? (size_t)(itm.bh % H) * total_tokens + itm.tok0 + q_idx
                                         : (size_t)itm.bh * (size_t)N + q_idx;
                lse[li] = (m_ref + lg2(l)) * kLn2;
            }
            ++oc;
        }
        tmem_wait_st();  // an aborted iteration may leave a store in flight
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == T::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TM_COLS);
    }
}

// Merge of the cut key ranges: one warp per query row whose row block was cut
// (rows of uncut row blocks were written by the attention kernel), lanes over the
// head dimension.  With L = ln sum_s e^{L_s}: O = sum_s e^{L_s - L} O_s, the
// online-softmax combination of the course page "10 FlashAttention", section "The
// decode variant: FlashDecoding".
template <int D>
__global__ void __launch_bounds__(256)
    fa_fwd_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_l,
                        __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, int N, int BH,
                        int causal, int rows_per_block, int n_kv_all, int keys_per_tile, int chunk,
                        int s_max, const __grid_constant__ FwdMergeNs mns, int n_cb_tab) {
    griddep_wait();  // the partials come from the attention kernel
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= (long long)BH * N) return;
    const int q = (int)(row % N);
    const int cb = q / rows_per_block;
    const int n_kv = causal ? min(n_kv_all, ((cb + 1) * rows_per_block + keys_per_tile - 1) /
                                                keys_per_tile)
                            : n_kv_all;
    // balanced plan (n_cb_tab > 0): the row block's segment count from its table
    const int ns = n_cb_tab > 0 ? (int)mns.ns[(row / N) * n_cb_tab + cb] : (n_kv + chunk - 1) / chunk;
    if (ns <= 1) return;
    const float *pl = ws_l + (size_t)row * s_max;
    float m = -INFINITY;
    for (int s = 0; s < ns; ++s) m = fmaxf(m, pl[s]);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float w = __expf(pl[s] - m);
        wsum += w;
        const float *po = ws_o + ((size_t)row * s_max + s) * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, po[lane + 32 * e], acc[e]);
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int e = 0; e < PER; ++e)
        out[(size_t)row * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
    if (lane == 0) lse[row] = m + __logf(wsum);
}

// Predicted time, in K/V-tile steps, of a one-tile launch whose row blocks are cut
// into chunks of `chunk` tiles (0: uncut): the persistent snake schedule of the
// kernel over min(items, SMs) CTAs, each item costing its tiles plus a fixed
// kItemCost (Q load, pipeline fill, epilogue), and a cut launch kMergeCost more for
// the merge kernel.  The constants come from fitting measured launches on this GPU
// (B1 H1 and H2 N16384, B1 H1 N32768 causal, B1 H1 N8192 non-causal, d = 128 and
// 256, chunks of 8, 16, 32 tiles and uncut): a tile step is ~0.86 us, an item's
// fixed cost ~6 steps.
constexpr double kItemCost = 6.0, kMergeCost = 5.0;

double fwd_split_cost(long long BH, long long n_cb, long long ratio, long long n_kv_all,
                      bool causal, long long chunk, int num_sms) {
    std::vector<long long> len;  // item lengths in the kernel's order (row block major)
    for (long long i = 0; i < n_cb; ++i) {
        const long long cb = causal ? n_cb - 1 - i : i;
        const long long nk = causal ? std::min(n_kv_all, (cb + 1) * ratio) : n_kv_all;
        const long long c = chunk > 0 ? chunk : nk;
        for (long long s = 0; s * c < nk; ++s)
            for (long long h = 0; h < BH; ++h) len.push_back(std::min(c, nk - s * c));
    }
    const long long n = (long long)len.size();
    const long long G = std::min<long long>(n, num_sms);
    std::vector<double> load((size_t)G, 0.0);
    for (long long r = 0; r * G < n; ++r)
        for (long long c = 0; c < G; ++c) {
            const long long idx = r * G + ((r & 1) ? G - 1 - c : c);
            if (idx < n) load[(size_t)c] += (double)len[(size_t)idx] + kItemCost;
        }
    double worst = 0.0;
    for (double x : load) worst = std::max(worst, x);
    return worst + (chunk > 0 ? kMergeCost : 0.0);
}

// Key-range chunk (in K/V tiles, a multiple of the row block's tiles on the
// diagonal) for a one-tile launch of B*H heads: 0 (no cut) unless the cost model
// above predicts a cut at least 5% faster; decisions are remembered per shape.
template <int D>
int fwd_split_chunk_t(int BH, int N, int causal, int num_sms, int forced) {
    using T = FwdTile<D, false, true>;
    const int ratio = T::ROWS / T::BN;
    if (forced > 0) return (forced + ratio - 1) / ratio * ratio;
    const long long n_cb = (N + T::ROWS - 1) / T::ROWS;
    const long long n_kv_all = (N + T::BN - 1) / T::BN;
    if (n_cb * BH >= num_sms) return 0;  // the row blocks alone fill the GPU
    static std::mutex m;
    static std::vector<std::array<int, 5>> memo;  // BH, N, causal, num_sms, chunk
    {
        std::lock_guard<std::mutex> lock(m);
        for (const auto &e : memo)
            if (e[0] == BH && e[1] == N && e[2] == causal && e[3] == num_sms) return e[4];
    }
    const long long longest = causal ? std::min(n_kv_all, n_cb * ratio) : n_kv_all;
    const double uncut = fwd_split_cost(BH, n_cb, ratio, n_kv_all, causal, 0, num_sms);
    double best = uncut * 0.95;
    int chunk = 0;
    for (long long c : {16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512}) {
        const long long ct = c * ratio;
        if (ct >= longest) break;
        const double cost = fwd_split_cost(BH, n_cb, ratio, n_kv_all, causal, ct, num_sms);
        if (cost < best) {
            best = cost;
            chunk = (int)ct;
        }
    }
    std::lock_guard<std::mutex> lock(m);
    if (memo.size() >= 256) memo.erase(memo.begin());
    memo.push_back({BH, N, causal, num_sms, chunk});
    return chunk;
}

// Balanced plan within a cap of `cap` steps per CTA (a segment costs its tiles plus
// kItemCost).  First the row blocks too long for one CTA's budget, longest first,
// are laid end to end from CTA 0 and cut where a CTA is full; no piece shorter than
// `min_seg` tiles is cut off unless the CTA is otherwise empty.  Then every other
// row block goes whole, longest first, to the CTA with the least room that still
// holds it, so only the long row blocks leave partials to merge.  Fills `out` (when
// given) and returns the CTAs used, or 0 when more than G CTAs, kSegMax segments or
// kSegMaxParts parts of one row block would be needed.
struct SegRow {
    int bh, cb;
    long long nk;
};

int seg_fill(const std::vector<SegRow> &rows, int n_cb, long long cap, long long min_seg, int G,
             FwdSegPlan *out) {
    const long long ic = (long long)kItemCost;
    struct Piece {
        int row, part;
        long long kv, n;
    };
    std::vector<std::vector<Piece>> per((size_t)G);
    std::vector<long long> load((size_t)G, 0);
    std::vector<int> parts_of(rows.size(), 1);
    int n = 0, cta = 0;
    for (size_t r = 0; r < rows.size(); ++r) {  // long row blocks, cut
        if (rows[r].nk + ic <= cap) continue;
        long long rem = rows[r].nk, kv = 0;
        int parts = 0;
        while (rem > 0) {
            if (cta >= G) return 0;
            const long long avail = cap - load[cta] - ic;
            long long take;
            if (rem <= avail) {
                take = rem;
            } else {
                take = rem - avail < min_seg ? rem - min_seg : avail;
                if (take < min_seg) take = load[cta] == 0 ? std::min(rem, std::max(avail, 1LL)) : 0;
            }
            if (take > 0) {
                if (n >= kSegMax || parts >= kSegMaxParts) return 0;
                per[cta].push_back({(int)r, parts, kv, take});
                ++n;
                ++parts;
                kv += take;
                rem -= take;
                load[cta] += take + ic;
            }
            if (rem > 0) ++cta;  // the CTA is full: the rest goes to the next
        }
        parts_of[r] = parts;
    }
    for (size_t r = 0; r < rows.size(); ++r) {  // the others, whole, best fit
        const long long need = rows[r].nk + ic;
        if (need > cap) continue;
        int best = -1;
        for (int c = 0; c < G; ++c)
            if (cap - load[c] >= need && (best < 0 || load[c] > load[best])) best = c;
        if (best < 0 || n >= kSegMax) return 0;
        per[best].push_back({(int)r, 0, 0, rows[r].nk});
        ++n;
        load[best] += need;
    }
    int used = 0, s_max = 1, k = 0;
    long long worst = 0;
    for (int c = 0; c < G; ++c) {
        if (per[c].empty()) continue;
        if (out) {
            out->tab.start[used] = (uint16_t)k;
            for (const Piece &pc : per[c]) {
                const SegRow &row = rows[pc.row];
                out->tab.seg[k][0] = (uint32_t)row.bh | ((uint32_t)row.cb << 16);
                out->tab.seg[k][1] = (uint32_t)pc.kv | ((uint32_t)pc.n << 12) | ((uint32_t)pc.part << 24) |
                                     ((uint32_t)parts_of[pc.row] << 28);
                ++k;
            }
        }
        worst = std::max(worst, load[c]);
        ++used;
    }
    for (size_t r = 0; r < rows.size(); ++r) {
        s_max = std::max(s_max, parts_of[r]);
        if (out) out->mns.ns[rows[r].bh * n_cb + rows[r].cb] = (uint8_t)parts_of[r];
    }
    if (out) {
        out->tab.n_cta = used;
        out->tab.start[used] = (uint16_t)n;
        int busiest = 0;
        for (int c = 0; c < used; ++c) busiest = std::max(busiest, out->tab.start[c + 1] - out->tab.start[c]);
        out->tab.max_per_cta = busiest;
        out->n_seg = n;
        out->s_max = s_max;
        out->cost = (double)worst + kMergeCost;
    }
    return used;
}

template <int D>
const FwdSegPlan *fwd_seg_plan_t(int BH, int N, int causal, int num_sms) {
    using T = FwdTile<D, false, true>;
    const long long ratio = T::ROWS / T::BN;
    const long long n_cb = (N + T::ROWS - 1) / T::ROWS;
    const long long n_kv_all = (N + T::BN - 1) / T::BN;
    const int G = std::min(num_sms, kSegMaxCta);
    if (n_cb * BH >= num_sms || n_cb * BH > kSegMaxRows || n_kv_all >= 4096 || n_cb > 65535 ||
        BH > 65535)
        return nullptr;
    struct Memo {
        int BH, N, causal, num_sms;
        std::unique_ptr<FwdSegPlan> plan;
    };
    static std::mutex m;
    static std::vector<Memo> memo;
    {
        std::lock_guard<std::mutex> lock(m);
        for (const Memo &e : memo)
            if (e.BH == BH && e.N == N && e.causal == causal && e.num_sms == num_sms) return e.plan.get();
    }
    std::vector<SegRow> rows;
    long long total = 0, longest = 0;
    for (long long i = 0; i < n_cb; ++i) {
        const long long cb = causal ? n_cb - 1 - i : i;
        const long long nk = causal ? std::min(n_kv_all, (cb + 1) * ratio) : n_kv_all;
        for (int h = 0; h < BH; ++h) rows.push_back({h, (int)cb, nk});
        total += BH * (nk + (long long)kItemCost);
        longest = std::max(longest, nk);
    }
    // Smallest cap the greedy fill meets with at most G CTAs (bisection); pieces of
    // at least eight row blocks' worth of diagonal tiles.  Only launches of at least
    // eight tiles per CTA: the cost model was fitted on long launches.
    const long long min_seg = 8 * ratio;
    if (total - BH * n_cb * (long long)kItemCost < 8LL * G) {
        std::lock_guard<std::mutex> lock(m);
        memo.push_back({BH, N, causal, num_sms, nullptr});
        return nullptr;
    }
    long long lo = std::max<long long>((total + G - 1) / G, (long long)kItemCost + 2 * min_seg);
    long long hi = lo + longest + (long long)kItemCost + 2 * min_seg;
    std::unique_ptr<FwdSegPlan> plan;
    if (seg_fill(rows, (int)n_cb, hi, min_seg, G, nullptr) > 0) {
        while (lo < hi) {
            const long long mid = (lo + hi) / 2;
            if (seg_fill(rows, (int)n_cb, mid, min_seg, G, nullptr) > 0) hi = mid; else lo = mid + 1;
        }
        plan.reset(new FwdSegPlan{});
        seg_fill(rows, (int)n_cb, lo, min_seg, G, plan.get());
        // kept only when predicted 5% faster than no cut and faster than even chunks
        const double uncut = fwd_split_cost(BH, n_cb, ratio, n_kv_all, causal, 0, num_sms);
        double even = uncut;
        for (long long c : {16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512}) {
            const long long ct = c * ratio;
            if (ct >= longest) break;
            even = std::min(even, fwd_split_cost(BH, n_cb, ratio, n_kv_all, causal, ct, num_sms));
        }
        if (!(plan->cost < 0.95 * uncut && plan->cost < even) || plan->s_max < 2) plan.reset();
    }
    // plans are kept for the life of the process (a few KB per shape), so the
    // pointers handed out stay valid
    std::lock_guard<std::mutex> lock(m);
    memo.push_back({BH, N, causal, num_sms, std::move(plan)});
    return memo.back().plan.get();
}

template <int D, bool CAUSAL, bool VARLEN, bool F8 = false, bool ONE = false, bool SPLIT = false>
int launch_fwd_t(const FwdParams &p, cudaStream_t stream) {
    using T = FwdTile<D, F8, ONE>;
    auto kern = fa_fwd_kernel<D, CAUSAL, VARLEN, F8, ONE, SPLIT>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), (int)T::SMEM_BYTES) != FA_OK)
        return FA_ERR_CUDA;
    // the warpgroups' register targets add up to the launch's pool only at this count
    if (T::RB && kernel_num_regs(reinterpret_cast<const void *>(kern)) != T::LAUNCH_REGS)
        return FA_ERR_UNSUPPORTED;
    // varlen: N is the longest sequence the caller allows
    const int n_cblocks = (p.N + T::ROWS - 1) / T::ROWS;
    long long items = (long long)n_cblocks * p.BH;
    const int n_kv_all = (p.N + T::BN - 1) / T::BN;
    if (SPLIT && p.seg) {
        items = p.seg->tab.n_cta;  // the plan's CTAs, each with its run of segments
    } else if (SPLIT) {
        const int ratio = T::ROWS / T::BN;
        long long per = 0;
        for (long long cb = 0; cb < n_cblocks; ++cb) {
            const long long nk = CAUSAL ? std::min<long long>(n_kv_all, (cb + 1) * ratio) : n_kv_all;
            per += (nk + p.kv_chunk - 1) / p.kv_chunk;
        }
        items = per * p.BH;
    }
    if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    // Persistent: one CTA per SM (the shared-memory footprint allows no more).
    const long long grid = items < p.num_sms ? items : p.num_sms;
    if (grid < 1) return FA_OK;
    SegArg<SPLIT> tab{};
    if constexpr (SPLIT)
        if (p.seg) tab = p.seg->tab;
    kern<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(
        p.tm_q, p.tm_k, p.tm_v, reinterpret_cast<__nv_bfloat16 *>(p.o), p.lse, p.N, p.BH, p.H,
        p.group, n_cblocks, p.cu_seqlens, p.total_tokens, p.scale_log2, p.q_descale, p.k_descale,
        p.v_descale, (p.N + 127) / 128, p.kv_chunk, p.ws_o, p.ws_l, p.s_max, p.status,
        p.limit_ns, tab);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
    if (SPLIT) {
        const long long rows = (long long)p.BH * p.N;
        const long long blocks = (rows * 32 + 255) / 256;
        if (blocks > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        FwdMergeNs mns{};
        if (p.seg) mns = p.seg->mns;
        if (cudaLaunchKernelEx(&cfg, fa_fwd_merge_kernel<D>, (const float *)p.ws_o,
                               (const float *)p.ws_l, reinterpret_cast<__nv_bfloat16 *>(p.o), p.lse,
                               p.N, p.BH, p.causal, T::ROWS, n_kv_all, T::BN, p.kv_chunk,
                               p.s_max, mns, p.seg ? n_cblocks : 0) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

template <int D>
int launch_fwd_d(const FwdParams &p, cudaStream_t stream) {
    if (p.cu_seqlens)
        return p.causal ? launch_fwd_t<D, true, true>(p, stream) : launch_fwd_t<D, false, true>(p, stream);
    if (p.kv_chunk > 0 || p.seg) {  // cut key ranges (one tile per CTA); the caller sized the workspace
        return p.causal ? launch_fwd_t<D, true, false, false, (D <= 128), true>(p, stream)
                        : launch_fwd_t<D, false, false, false, (D <= 128), true>(p, stream);
    }
    if constexpr (D <= 128) {
        // fewer two-tile items than SMs: one tile per CTA instead
        const long long items2 = (long long)((p.N + 255) / 256) * p.BH;
        if (items2 < p.num_sms)
            return p.causal ? launch_fwd_t<D, true, false, false, true>(p, stream)
                            : launch_fwd_t<D, false, false, false, true>(p, stream);
    }
    return p.causal ? launch_fwd_t<D, true, false>(p, stream) : launch_fwd_t<D, false, false>(p, stream);
}

const FwdSegPlan *fwd_seg_plan(int d, int BH, int N, int causal, int num_sms) {
    switch (d) {
        case 64: return fwd_seg_plan_t<64>(BH, N, causal, num_sms);
        case 96: return fwd_seg_plan_t<96>(BH, N, causal, num_sms);
        case 128: return fwd_seg_plan_t<128>(BH, N, causal, num_sms);
        case 256: return fwd_seg_plan_t<256>(BH, N, causal, num_sms);
        default: return nullptr;
    }
}

int fwd_split_chunk(int d, int BH, int N, int causal, int num_sms, int forced) {
    switch (d) {
        case 64: return fwd_split_chunk_t<64>(BH, N, causal, num_sms, forced);
        case 96: return fwd_split_chunk_t<96>(BH, N, causal, num_sms, forced);
        case 128: return fwd_split_chunk_t<128>(BH, N, causal, num_sms, forced);
        case 256: return fwd_split_chunk_t<256>(BH, N, causal, num_sms, forced);
        default: return 0;
    }
}

int launch_fwd(const FwdParams &p, cudaStream_t stream) {
    if (p.fp8) {
        if (p.d != 128 || p.cu_seqlens) return FA_ERR_UNSUPPORTED;
        return p.causal ? launch_fwd_t<128, true, false, true>(p, stream)
                        : launch_fwd_t<128, false, false, true>(p, stream);
    }
    switch (p.d) {
        case 64: return launch_fwd_d<64>(p, stream);
        case 96: return launch_fwd_d<96>(p, stream);
        case 128: return launch_fwd_d<128>(p, stream);
        case 256: return launch_fwd_d<256>(p, stream);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
