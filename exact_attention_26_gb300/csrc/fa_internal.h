// Declarations shared by the host API and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Where a bounded wait gave up (second word of the device status record).
enum WaitSite : int {
    SITE_NONE = 0,
    SITE_FWD_LOAD_KV_EMPTY = 1,
    SITE_FWD_MMA_Q = 2,
    SITE_FWD_MMA_KV_FULL = 3,
    SITE_FWD_MMA_P_FULL = 4,
    SITE_FWD_SOFTMAX_S_FULL = 5,
    SITE_FWD_EPILOGUE_O_FULL = 6,
    SITE_FWD_DRAIN = 7,
    SITE_FWD_BAD_SEQ = 8,
    SITE_BWD_LOAD_EMPTY = 11,
    SITE_BWD_MMA_KV = 12,
    SITE_BWD_MMA_Q_FULL = 13,
    SITE_BWD_MMA_DS_FULL = 14,
    SITE_BWD_MMA_DQ_FREE = 15,
    SITE_BWD_SOFTMAX_S_FULL = 16,
    SITE_BWD_DQ_FULL = 17,
    SITE_BWD_EPILOGUE = 18,
    SITE_BWD_DRAIN = 19,
    SITE_BWD_BAD_SEQ = 20,
    SITE_BWD_SMEM_ALIGN = 26,
    SITE_FWD_SMEM_ALIGN = 27,
    SITE_DEC_FULL = 21,
    SITE_DEC_EMPTY = 22,
    SITE_DEC_DRAIN = 23,
    SITE_DEC_BAD_LEN = 24,
    SITE_DEC_BAD_PAGE = 25,
    SITE_DEC_MMA = 28,
    SITE_BWD_ITEM = 29,
    SITE_SELFTEST = 30,
};

// Default limit of one in-kernel wait.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct FwdSegPlan;

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over [BH][N][d] (q) and [B*Hkv][N][d] (k, v) bf16
    void *o;                       // bf16 [BH][N][d]
    float *lse;                    // fp32 [BH][N]
    int N, BH, d, causal;
    int H, group;                  // query heads per batch; query heads per key/value head
    const int *cu_seqlens;         // varlen: [B+1] sequence starts (token-major layout), else null
    int total_tokens;              // varlen: T
    float scale_log2;              // scale * log2(e)
    int fp8;                       // e4m3 inputs: tm_q/tm_k over bytes, tm_v over V^T [B*Hkv][d][Np]
    const float *q_descale, *k_descale, *v_descale;  // fp8: [BH][nqb], [B*Hkv][nqb], [B*Hkv]
    int kv_chunk;                  // > 0: key ranges cut into chunks of this many K/V tiles
    const FwdSegPlan *seg;         // non-null: key ranges cut by this balanced plan
    float *ws_o, *ws_l;            // kv_chunk > 0: partial O [BH][N][s_max][d], L [BH][N][s_max]
    int s_max;                     // chunks of the longest key range
    int *status;                   // device status record (2 ints)
    unsigned long long limit_ns;
    int num_sms;
};

// Key-range chunk in K/V tiles of the one-tile forward for B*H heads of N rows
// (0: no cut); `forced` > 0 asks for that many tiles (rounded up to the tiles of a
// row block on the diagonal).
int fwd_split_chunk(int d, int BH, int N, int causal, int num_sms, int forced);

// Balanced cut of the one-tile forward's key ranges: the row blocks, longest first,
// are laid end to end and cut into segments (a row block's K/V tiles
// [kv_lo, kv_lo + n)) so that every CTA's run of consecutive segments costs about
// the same (its tiles plus a fixed cost per segment); the kernel reads its run from
// the table and the merge kernel the segment count of each row block.
constexpr int kSegMaxCta = 256, kSegMax = 640, kSegMaxRows = 256, kSegMaxParts = 15;
struct FwdSegTable {
    int n_cta, max_per_cta;           // CTAs of the launch; segments of the busiest
    uint16_t start[kSegMaxCta + 1];   // CTA c runs segments [start[c], start[c + 1])
    uint32_t seg[kSegMax][2];         // bh | cb << 16;  kv_lo | n << 12 | s << 24 | ns << 28
};
struct FwdMergeNs {
    uint8_t ns[kSegMaxRows];          // segments of row block bh * n_cb + cb
};
struct FwdSegPlan {
    FwdSegTable tab;
    FwdMergeNs mns;
    int n_seg, s_max;                 // segments; most segments of one row block
    double cost;                      // predicted K/V-tile steps, merge included
};
// The balanced plan for B*H heads of N rows, or null when the library does not cut
// this way (the cut is not predicted 5% faster than no cut and faster than even
// chunks).  Plans are remembered per shape; the pointer stays valid.
const FwdSegPlan *fwd_seg_plan(int d, int BH, int N, int causal, int num_sms);
// Rows per TMA box of the forward's K and V tensor maps (the kernel loads a K/V
// tile of BN keys as BN / box boxes).
constexpr int fwd_kv_box_rows(int d) { return d == 256 ? 64 : 128; }

// e4m3 block quantiser: x bf16 [BH][N][d] -> codes [BH][N][d] (or [BH][d][Np]).
struct QuantParams {
    const void *x;
    void *codes;
    float *descale;        // [BH][n_groups]
    float *partial;        // workspace: per 128-row chunk maxima, [BH][n_chunks]
    const float *signs;    // incoherent processing: d signs (+-1), or null
    int BH, N, d, block_rows, transpose, Np;
};

int launch_quant(const QuantParams &p, cudaStream_t stream);

// Query rows per backward block of the kernel that serves head dim d (the box
// height of the q and dO tensor maps).
int bwd_block_q(int d);

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // 3-D maps over [BH][N][d] (q, do), [B*Hkv][N][d] (k, v)
    CUtensorMap tm_dq;                    // fp32 dq: (d, N, BH) box (32, 32, 1), or packed
                                          // (d, heads, T) box (32, 1, 32); tiled bulk adds
    const void *o, *dout;                 // bf16 [BH][N][d]
    const float *lse;                     // fp32 [BH][N]
    float *dq, *dk, *dv;                  // fp32 [BH][N][d]
    float *ws_delta, *ws_lse2;            // workspace, [BH][Npad] each
    int *ws_counter;                      // workspace: the main kernel's next unclaimed item
    int N, Npad, BH, d, causal;
    int H, group;                         // query heads per batch; query heads per k/v head
    const int *cu_seqlens;                // varlen: [B+1] sequence starts (token-major), else null
    int total_tokens;                     // varlen: T
    float scale, scale_log2;
    int *status;
    unsigned long long limit_ns;
    int num_sms;
};

// Query rows per backward q-block and the padding unit of the workspace vectors.
constexpr int kBwdPad = 128;
// Bytes at the end of the backward workspace for the work-item counter.
constexpr size_t kBwdCounterBytes = 16;

struct DecodeParams {
    // tensor-core path only: q as [1][BH*Nq][d] (boxes of 128 rows), k and v as
    // [B*Hkv][Nk][d] (boxes of 64 keys)
    CUtensorMap tm_q, tm_k, tm_v;
    const void *q;            // bf16 [BH][Nq][d]
    const void *k, *v;        // bf16 [B*Hkv][Nk][d], or paged [num_pages][Hkv][page_size][d]
    void *o;                  // bf16 [BH][Nq][d]
    float *lse;               // fp32 [BH][Nq]
    float *part_o, *part_l;   // workspace when S > 1: [B*Hkv][S][group*Nq][d], [..][S][group*Nq]
    const int *block_table;   // paged: [B][max_pages] physical page of each logical page
    const int *seq_lens;      // paged: [B] cached tokens of each sequence
    int BH, H, Nq, Nk, d;     // Nk: keys per head (paged: page_size * max_pages, an upper bound)
    int Hkv, group;           // key/value heads; query heads per key/value head (H = Hkv*group)
    int S, keys_per_split;    // key ranges [s*keys_per_split, ...) per CTA
    int paged, page_size, max_pages, num_pages;
    float scale_log2;
    int *status;
    unsigned long long limit_ns;
};

// Devices the per-device caches of the host code cover (ordinals 0..63).
constexpr int kMaxCachedDevices = 64;

// Raise a kernel's dynamic shared memory limit to `bytes` once per (kernel,
// device): the attribute stays with the function in the device's context, so
// later launches skip the driver call.  FA_OK or FA_ERR_CUDA.
int ensure_smem_attr(const void *kernel, int bytes);

// Registers per thread a kernel is launched with (cached per kernel), or -1.
int kernel_num_regs(const void *kernel);

int launch_fwd(const FwdParams &p, cudaStream_t stream);
int launch_bwd(const BwdParams &p, cudaStream_t stream);
int launch_decode(const DecodeParams &p, cudaStream_t stream);
// Decode with R = (H / Hkv) * Nq query rows per key/value head: whether the
// tensor-core kernel serves it, and the launch shape of the kernel that does.
bool decode_uses_mma(int d, int R, bool paged);
int decode_block_keys(int d, int R, bool paged);   // keys per pipeline stage
int decode_query_block(int d, int R, bool paged);  // query rows per decode CTA
int decode_ctas_per_sm(int d, int R, bool paged);  // resident decode CTAs per SM

}  // namespace fa
