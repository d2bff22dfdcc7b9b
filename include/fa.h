/*
 * fa.h - C ABI of libfa.so: exact scaled-dot-product attention on GB300 (sm_103a).
 *
 * The operation ("FlashAttention: Move Less, Not Compute Less", section "The
 * Multiplication May Not Be the Slow Part"; the 1/sqrt(d) scale and causal rule
 * from the course page "10 FlashAttention", sections 1 and 4):
 *
 *     O = softmax(Q K^T * scale + mask) V,   per (batch b, head h),
 *     mask[i][j] = -inf where causal and j > i (query i sees keys 0..i), else 0,
 *     L[i] = m_i + ln(l_i) with m_i the row max of the scaled, masked scores and
 *            l_i = sum_j exp(s_ij - m_i)   ("FlashAttention-2: Why the Attention
 *            Bottleneck Wasn't Where Everyone Was Looking", section "FA2 change #1").
 *
 * The N x N score and probability matrices are never written to global memory:
 * the forward pass streams K/V tiles through on-chip memory with the online
 * softmax update and divides by l once at the end; the backward pass rebuilds S
 * and P tile by tile from L ("Why More Arithmetic Can Finish Sooner").
 *
 * Conventions shared by every entry point:
 *  - Tensors are DEVICE pointers in the caller's CUDA context, contiguous,
 *    row-major [B][H][N][d] for q, k, v, o, dout, dq, dk, dv and [B][H][N] for lse.
 *    q, k, v, o, dout hold bfloat16 values (raw 16-bit __nv_bfloat16 bits);
 *    lse, dq, dk, dv hold float32.  Entry points with other layouts (grouped
 *    key/value heads, packed sequences, decode caches, e4m3 codes) say so.
 *  - Tensor pointers must be 16-byte aligned, small int32/fp32 index and scale
 *    arrays 4-byte aligned (FA_ERR_MISALIGNED otherwise).
 *  - The caller owns every buffer.  The library allocates no device memory per
 *    call; it keeps a small per-device cache (SM count, an 8-byte device status
 *    word that lives in the library's own device data).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and never synchronise, except fa_device_status.
 *  - Argument errors are reported by the return value BEFORE anything is
 *    launched.  A launch failure returns FA_ERR_CUDA (from cudaGetLastError).
 *  - Every wait inside the kernels is bounded (about two seconds).  A wait that
 *    runs out records FA_ERR_TIMEOUT in the device status word and the kernel
 *    returns without hanging; fa_device_status reports it.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad scale, ... */
    FA_ERR_UNSUPPORTED = 2, /* head dimension not built */
    FA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
    FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    FA_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait ran out (device status) */
    FA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required */
    FA_ERR_BAD_INDEX = 7    /* device status: a block-table entry, sequence length or
                               cu_seqlens offset out of range (paged decode, packed
                               sequences); the affected work wrote nothing */
} fa_status;

/*
 * Forward pass.
 *   q, k, v : bf16 [B][H][N][d] inputs.
 *   o       : bf16 [B][H][N][d] output, O = (sum_j P_ij V_j), rounded to nearest even.
 *   lse     : fp32 [B][H][N] output, the natural-log L of each query row.
 *   B, H, N : batch, heads, sequence length (queries = keys = N); each >= 1,
 *             B*H*N < 2^31.  N need not be a multiple of any tile size.
 *   d       : head dimension, one of 64, 96, 128, 256 (96: rows padded to 128 columns
 *             in shared memory by the copies, products run over the 96 columns).
 *   causal  : nonzero for the causal mask (top-left aligned, j <= i).
 *   scale   : multiplies Q K^T before the softmax; finite and > 0 (1/sqrt(d) is
 *             the usual value).
 * Returns FA_OK or an fa_status code; nothing is launched on an error.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int N, int d, int causal, float scale, void *stream);

/*
 * Bytes of caller-provided device workspace fa_bwd needs for these sizes (the
 * per-row D_i = dO_i . O_i and the base-2 copy of L, padded per head, and a
 * 16-byte counter the kernels use to hand out their work).
 * Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass: the gradients of the forward above with respect to q, k and v,
 * given dout = dL/dO, rebuilding S and P from q, k and the saved lse.
 *   q, k, v, o, dout : bf16 [B][H][N][d] (o and lse exactly as fa_fwd wrote them).
 *   lse              : fp32 [B][H][N].
 *   dq, dk, dv       : fp32 [B][H][N][d] outputs, overwritten (fa_bwd zeroes dq
 *                      itself before accumulating into it).
 *   d                : 64, 96 or 128 (256 returns FA_ERR_UNSUPPORTED).
 *   workspace        : device buffer of at least fa_bwd_workspace_bytes(B,H,N,d)
 *                      bytes, 16-byte aligned, owned by the caller; its contents
 *                      on entry do not matter and are overwritten.
 * Other arguments as in fa_fwd.  Calls that share a workspace must not overlap.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, float *dq, float *dk, float *dv, int B, int H, int N, int d,
           int causal, float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Grouped-query attention (GQA; multi-query attention when Hkv = 1): the H query
 * heads of a batch share Hkv key/value heads, query head h reading key/value head
 * h / (H / Hkv) ("FlashAttention: Move Less, Not Compute Less", section "What It
 * Changes - and What It Does Not": GQA reduces the number of key/value heads, and
 * the official implementation has GQA/MQA paths).  The definition is the one above with
 * K and V of head h taken from that shared head; fa_fwd and fa_bwd are the case
 * Hkv = H.
 *   k, v        : bf16 [B][Hkv][N][d]; q, o, dout [B][H][N][d]; lse [B][H][N].
 *   dk, dv      : fp32 [B][Hkv][N][d], each the sum over the H / Hkv query heads that
 *                 read that key/value head (accumulated on chip, no atomics).
 *   Hkv         : >= 1 and divides H (FA_ERR_INVALID_ARG otherwise).
 * Workspace: fa_bwd_workspace_bytes(B, H, N, d) (per query row).  Other arguments,
 * results and errors as in fa_fwd / fa_bwd.
 */
int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int Hkv, int N, int d, int causal, float scale, void *stream);
int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, float *dq, float *dk, float *dv, int B, int H, int Hkv, int N,
               int d, int causal, float scale, void *workspace, size_t workspace_bytes,
               void *stream);

/*
 * Forward pass with the key range of each query row block cut over several CTAs
 * ("FlashAttention-2: ...", section "FA2 change #2: Parallelize over sequence
 * length": a batch-1 call with few heads must still fill the GPU).  Each chunk
 * yields a normalised partial O_s and its L_s = m_s + ln l_s, and the chunks of a
 * row are merged as L = ln sum_s e^(L_s), O = sum_s e^(L_s - L) O_s (the combination
 * of the course page "10 FlashAttention", section "The decode variant:
 * FlashDecoding").  Same definition, layouts, results and errors as fa_fwd_gqa.
 *   kv_chunk    : 0 lets the library choose: it cuts key ranges only when one
 *                 query tile per CTA would leave SMs idle or wait on the longest
 *                 rows (few heads, long sequences), preferably by the balanced
 *                 plan fa_fwd_split_segments reports (segments of uneven length
 *                 that give every CTA about the same work), else into even
 *                 chunks; > 0 asks for even chunks of about kv_chunk keys
 *                 (rounded up to the keys of a 128-row block's diagonal: 128, or
 *                 64 at d = 256, times one).  < 0: FA_ERR_INVALID_ARG.
 *   workspace   : device buffer of at least fa_fwd_workspace_bytes(B, H, N, d,
 *                 causal, kv_chunk) bytes, 256-byte aligned (FA_ERR_MISALIGNED),
 *                 owned by the caller, contents on entry irrelevant; may be NULL
 *                 when that size is 0 (no cut: the call is fa_fwd_gqa).  Too
 *                 small or missing: FA_ERR_WORKSPACE before anything is launched.
 *                 Calls that share a workspace must not overlap.
 * The choice and the size depend on the current device's SM count.
 */
size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal, int kv_chunk);

/*
 * The balanced cut fa_fwd_ws makes with kv_chunk = 0 on a device of num_sms SMs, for
 * inspection (host only: nothing is launched and no device is needed).  Every CTA
 * gets about the same work, counting a segment's K/V tiles plus a fixed cost of six
 * tile steps (its Q load, pipeline fill and epilogue): the row blocks of 128 query
 * rows longer than that budget (all B*H heads, longest first) are laid end to end
 * and cut where a CTA is full, into at most 15 parts; the other row blocks go whole
 * to the fullest CTA that still holds them.
 * The library uses this cut when its cost model predicts it at least 5% faster than
 * no cut and faster than even chunks, and otherwise cuts evenly or not at all.
 *   out : int[cap][7] host buffer, filled with the first cap segments in CTA order:
 *         head (b * H + h), row block, first K/V tile, K/V tiles, part s within the
 *         row block (in key order), parts of the row block, CTA.  May be NULL when
 *         cap = 0.
 * Returns the number of segments (0: the library does not cut this shape this way),
 * or FA_ERR_INVALID_ARG for invalid sizes, num_sms < 1, cap < 0 or a NULL out with
 * cap > 0.
 */
int fa_fwd_split_segments(int B, int H, int N, int d, int causal, int num_sms, int *out, int cap);
int fa_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
              int Hkv, int N, int d, int causal, float scale, int kv_chunk, void *workspace,
              size_t workspace_bytes, void *stream);

/*
 * Backward pass that allocates nothing, for callers that cannot allocate device
 * memory or pass a workspace: a host that reserves all device memory up front in
 * its own pool and forbids side allocations, or a latency-critical loop where a
 * cudaMalloc, which may synchronise the device, is not acceptable.  (The pages
 * have no counterpart to this entry point; it is a deployment convenience.)
 *
 * Same arguments, results and errors as fa_bwd, minus the workspace.  Instead of
 * a workspace it uses a scratch array of FA_NOALLOC_SCRATCH_BYTES compiled into
 * the library; every GPU that loads the library holds that array until exit.
 *   - Sizes whose fa_bwd_workspace_bytes(B, H, N, d) exceeds
 *     FA_NOALLOC_SCRATCH_BYTES, i.e. B*H*roundup(N, 128) > 1,048,576 rows, return
 *     FA_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) while that device is current; make that first call
 *     before any stream capture.  The address is cached per device ordinal for the
 *     life of the process: do not reset the device (cudaDeviceReset) or otherwise
 *     tear down its primary context between calls, which would leave the cached
 *     address pointing at memory that no longer exists.
 *   - Every call shares the one array; its contents on entry do not matter (each
 *     call rewrites what it reads).  Calls that overlap on the GPU (different
 *     streams, no ordering between them) race on it and give wrong results.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 */
/* 8 MiB for 1,048,576 rows of the two fp32 vectors, plus room for the work counter */
#define FA_NOALLOC_SCRATCH_BYTES (((size_t)8 << 20) + 256)
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dout, float *dq, float *dk, float *dv, int B,
                   int H, int N, int d, int causal, float scale, void *stream);

/*
 * e4m3 block quantisation for the low-precision forward ("FlashAttention: Move
 * Less, Not Compute Less", section "FA1 to FA3: Optimization Moves Closer to the
 * Hardware": FP8 with block quantisation and incoherent processing).  The pages
 * name the technique only; this library's reading:
 *   x           : bf16 [BH][N][d], d in {64, 128, 256}.
 *   block_rows  : rows per scale block, 0 (one block per head) or a multiple of 128.
 *   signs       : NULL, or fp32 [d] of +-1 (16-byte aligned, device memory): each
 *                 row is first multiplied by diag(signs) H / sqrt(d), H the
 *                 Sylvester-Hadamard matrix ("incoherent processing"; an orthogonal
 *                 map, so Q K^T is unchanged when Q and K take the same signs).
 *   codes       : uint8 e4m3 [BH][N][d], or with transpose != 0 [BH][d][Np] with
 *                 Np = N rounded up to 16 and columns N..Np-1 zero (the value layout
 *                 fa_fwd_fp8 reads).
 *   descale     : fp32 [BH][n_blocks] out (n_blocks = ceil(N / block_rows), or 1).
 * Per block, in IEEE fp32: amax = max |x|, inv = 448 / amax, code = e4m3(x * inv)
 * rounded to nearest even with finite overflow saturated to +-448, descale =
 * amax / 448 (an all-zero block: inv = descale = 1).  The dequantised value of a
 * code is value(code) * descale.
 *   workspace   : fa_quantize_fp8_workspace_bytes(BH, N, d) bytes, 16-byte aligned.
 * Returns FA_OK or an fa_status code; nothing is launched on an error.
 */
size_t fa_quantize_fp8_workspace_bytes(int BH, int N, int d);
int fa_quantize_fp8(const void *x, void *codes, float *descale, int BH, int N, int d,
                    int block_rows, const float *signs, int transpose, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * Low-precision forward: attention on e4m3 inputs with fp32 accumulation.  Both
 * products run on the tensor cores with 8-bit operands: S = Q K^T from the codes,
 * scaled by scale * q_descale * k_descale of the two row blocks, and O += P V with P
 * rounded to e4m3 (P <= 2^8 relative to the running reference maximum); the row
 * sum l is taken from P before rounding, so L is that of the dequantised inputs.
 *   q8        : e4m3 [B][H][N][d];  k8 : e4m3 [B][Hkv][N][d]  (d = 128).
 *   vt8       : e4m3 [B][Hkv][d][Np], V transposed per head, Np = N rounded up to 16
 *               (fa_quantize_fp8 with transpose = 1 writes it).
 *   q_descale : fp32 [B*H][ceil(N/128)];  k_descale : fp32 [B*Hkv][ceil(N/128)]
 *               (block_rows = 128);  v_descale : fp32 [B*Hkv] (block_rows = 0).
 *   o, lse    : bf16 [B][H][N][d] and fp32 [B][H][N] out, as in fa_fwd.
 * The result equals fa_fwd's definition applied to the dequantised q, k, v up to
 * the rounding of P to e4m3 (relative 2^-4 per element, absolute 2^-10 below 2^-6).
 * Other arguments as in fa_fwd_gqa.
 */
int fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *q_descale,
               const float *k_descale, const float *v_descale, void *o, float *lse, int B, int H,
               int Hkv, int N, int d, int causal, float scale, void *stream);

/*
 * Forward pass over packed sequences of different lengths (variable-length
 * batches: course page "10 FlashAttention", section "8-9. Production and
 * mistakes", counts padding sequences instead of packing them among the mistakes).  Sequence
 * b holds tokens [cu_seqlens[b], cu_seqlens[b+1]) of the packed tensors and
 * attends only within itself; the causal mask is taken per sequence (its token i
 * sees its tokens 0..i).  Layout is token-major:
 *   q, o        : bf16 [total_tokens][H][d];  k, v : bf16 [total_tokens][Hkv][d].
 *   lse         : fp32 [H][total_tokens].
 *   cu_seqlens  : int32 [B+1], device memory, 0 <= cu[b] <= cu[b+1] <= total_tokens,
 *                 each length at most max_seqlen.  Checked on the device: a sequence
 *                 that breaks these is skipped (its rows are not written) and
 *                 FA_ERR_BAD_INDEX is recorded for fa_device_status.
 *   max_seqlen  : >= 1, an upper bound on the lengths (sizes the launch).
 *   Hkv         : divides H (grouped-query attention as in fa_fwd_gqa).
 * Other arguments as in fa_fwd.
 */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *cu_seqlens, int B, int H, int Hkv, int total_tokens, int max_seqlen,
                  int d, int causal, float scale, void *stream);

/*
 * Backward pass of fa_fwd_varlen: gradients for packed sequences.
 *   q, k, v, o, dout : token-major as in fa_fwd_varlen (o, lse as it wrote them).
 *   dq               : fp32 [total_tokens][H][d]; dk, dv fp32 [total_tokens][Hkv][d].
 *                      Rows of the tokens of every sequence are overwritten; rows of
 *                      tokens that belong to no sequence are left untouched.
 *   d                : 64, 96 or 128.
 *   workspace        : fa_bwd_workspace_bytes(B, H, max_seqlen, d) bytes.
 * cu_seqlens is checked on the device as in fa_fwd_varlen (FA_ERR_BAD_INDEX).  Other
 * arguments as in fa_bwd / fa_bwd_gqa.
 */
int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dout, float *dq, float *dk, float *dv, const int *cu_seqlens, int B,
                  int H, int Hkv, int total_tokens, int max_seqlen, int d, int causal, float scale,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode attention with a split key range (course page "10 FlashAttention",
 * section "The decode variant: FlashDecoding"): Nq query rows per (b, h), usually
 * one, attend to all Nk cached keys of their head, with no mask:
 *
 *     O[i] = softmax(q_i K^T * scale) V,   L[i] = m_i + ln(l_i)   (natural log).
 *
 * The key range of each head is cut into S contiguous ranges handled by separate
 * CTAs; each produces a partial (O_s, L_s) of its range, and a second kernel
 * merges them: L = ln sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.  The result is
 * the same as with one range up to rounding.  With grouped queries (Hkv < H, see
 * fa_fwd_gqa) the H / Hkv query heads of a key/value head are handled by the same
 * CTAs, so the cache is read once for all of them.  With R = (H / Hkv) * Nq >= 2
 * query rows per key/value head and d <= 128 the products run on the tensor cores
 * (tcgen05, the CTA's rows as M = 128 against tiles of 64 or 128 keys); otherwise
 * on CUDA cores (see fa_decode_uses_tensor_cores).
 *   q      : bf16 [B][H][Nq][d] (the new tokens' queries).
 *   k, v   : bf16 [B][Hkv][Nk][d] (the key/value cache, contiguous per head).
 *   o      : bf16 [B][H][Nq][d] output, rounded to nearest even.
 *   lse    : fp32 [B][H][Nq] output.
 *   B, H   : >= 1; Hkv >= 1 divides H.  Nq in [1, 65535], (H/Hkv)*Nq <= 65535,
 *            Nk >= 1, B*H*Nq and B*Hkv*Nk < 2^31.
 *   d      : 64, 96, 128 or 256.
 *   scale  : finite and > 0.
 *   num_splits : 0 chooses S automatically (about eight CTAs per SM in total,
 *            at least four pipeline stages of keys per range); a positive value
 *            asks for that many ranges, reduced so that none is empty.
 *   workspace : device buffer of at least fa_decode_workspace_bytes(...) bytes,
 *            16-byte aligned, owned by the caller, contents on entry irrelevant;
 *            may be NULL when that size is 0 (S = 1).  Calls that share a
 *            workspace must not overlap.
 * Returns FA_OK or an fa_status code; nothing is launched on an error.
 */
int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
              int Hkv, int Nq, int Nk, int d, float scale, int num_splits, void *workspace,
              size_t workspace_bytes, void *stream);

/*
 * The number of key ranges S that fa_decode would use for these arguments on the
 * current device (>= 1), or minus an fa_status code for invalid sizes or a CUDA
 * error.  Needs the device's SM count when num_splits is 0.
 */
int fa_decode_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits);

/*
 * 1 if fa_decode (paged = 0) or fa_decode_paged (paged = 1) runs these sizes on
 * the tensor-core kernel, 0 if on the CUDA-core kernel, minus an fa_status code
 * for invalid sizes.  (Paged caches always use the CUDA-core kernel.)
 */
int fa_decode_uses_tensor_cores(int H, int Hkv, int Nq, int d, int paged);

/*
 * Workspace bytes fa_decode needs: 0 when S = 1, else room for the S partial
 * outputs (fp32, S * B*H*Nq rows of d) and their L values (fp32, S * B*H*Nq).
 * Returns 0 for invalid sizes as well.
 */
size_t fa_decode_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits);

/*
 * Decode against a paged key/value cache (course page "10 FlashAttention",
 * section "Paged FlashAttention": the K/V blocks of a sequence are gathered
 * through a block table instead of being read contiguously).  Same operation,
 * split and merge as fa_decode, except that sequence b has its own length
 * seq_lens[b] and its key j lives in physical page block_table[b][j / page_size]
 * at row j % page_size:
 *   k_cache, v_cache : bf16 [num_pages][Hkv][page_size][d]; one page holds
 *                      page_size consecutive tokens of every head, each head's
 *                      rows contiguous (one bulk copy per page and head).
 *   block_table      : int32 [B][max_pages_per_seq], device memory; entries in
 *                      [0, num_pages) for the pages a sequence uses (the rest are
 *                      never read).
 *   seq_lens         : int32 [B], device memory; 1 <= seq_lens[b] <=
 *                      page_size * max_pages_per_seq.
 *   q, o, lse        : as in fa_decode, [B][H][Nq][d] and [B][H][Nq].
 *   page_size, max_pages_per_seq, num_pages >= 1; page_size * max_pages_per_seq
 *   < 2^31.  Pages of any size work; each page costs one copy per stage.
 * The table and the lengths live on the device, so they are checked there: an
 * out-of-range entry or length makes the affected CTA write nothing and records
 * FA_ERR_BAD_INDEX in the device status word (fa_device_status); nothing outside
 * the cache is read.  The key ranges are cut from the longest possible sequence;
 * ranges past a shorter sequence's end contribute nothing to its merge.
 * Workspace as in fa_decode, sized by fa_decode_paged_workspace_bytes.
 */
int fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                    const int *block_table, const int *seq_lens, void *o, float *lse, int B, int H,
                    int Hkv, int Nq, int d, int page_size, int max_pages_per_seq, int num_pages,
                    float scale, int num_splits, void *workspace, size_t workspace_bytes,
                    void *stream);

/* Key ranges (>= 1) fa_decode_paged would use, or minus an fa_status code. */
int fa_decode_paged_num_splits(int B, int H, int Hkv, int Nq, int d, int page_size,
                               int max_pages_per_seq, int num_splits);

/* Workspace bytes fa_decode_paged needs (0 when one range suffices or sizes are invalid). */
size_t fa_decode_paged_workspace_bytes(int B, int H, int Hkv, int Nq, int d, int page_size,
                                       int max_pages_per_seq, int num_splits);

/*
 * Diagnostic: launches one warp that waits, through the same bounded wait the
 * attention kernels use, on a barrier that nothing ever arrives on.  The wait
 * gives up after `limit_ns` nanoseconds (1e3 <= limit_ns <= 5e9, else
 * FA_ERR_INVALID_ARG), records FA_ERR_TIMEOUT in the device status word and the
 * kernel returns; fa_device_status then reports FA_ERR_TIMEOUT once.  Shows that
 * a wait that runs out leaves the context usable.  Asynchronous on `stream`.
 */
int fa_selftest_wait_timeout(unsigned long long limit_ns, void *stream);

/*
 * Measurement utility (not on the attention path): the per-SM rates of the units
 * the kernels are bound by, measured on the current device with one CTA per SM and
 * clock64 stamps, `iters` iterations per probe (16 <= iters <= 2^20, else
 * FA_ERR_INVALID_ARG; 2048 takes about a millisecond per probe).  On return
 * (host array of 3 doubles, the median over SMs):
 *   rates[0]  dense bf16 tcgen05.mma kind::f16, M = 128, N = 256, K = 16, fp32
 *             accumulate: FLOPs per SM clock (the tensor core's peak shape);
 *   rates[1]  the same at N = 64 (the shape of the backward's S^T, dP^T and dQ^T
 *             products at d = 128);
 *   rates[2]  MUFU ex2.approx.f32 results per SM clock (the softmax exponential).
 * Times SM count times SM clock, rates[0] is the clock-derived tensor peak and
 * rates[2] the exponential ceiling of the forward (one ex2 per score element).
 * Synchronises `stream`.  Returns FA_ERR_TIMEOUT if an MMA completion wait gave up
 * (the record is cleared), FA_ERR_UNSUPPORTED above 1024 SMs, FA_ERR_CUDA on a
 * CUDA error.
 */
int fa_probe_unit_rates(double *rates, int iters, void *stream);

/*
 * Measurement utility (not on the attention path): the HBM read rate, the ceiling
 * of a kernel whose traffic is reads (the decode kernels read the cache once and
 * write almost nothing, which a copy rate, half reads and half writes, does not
 * describe).  Reads the `bytes` at device pointer `buf` (16-byte aligned, a multiple
 * of 16 bytes, at least 1 MiB; choose far more than the L2) with 16-byte loads that
 * do not allocate in L1, once untimed and then `iters` times (1..1000) between CUDA
 * events on `stream`, and writes the rate in GB/s (10^9 bytes per second) to *gbs.
 * Synchronises `stream`.  FA_ERR_INVALID_ARG on a bad argument, FA_ERR_CUDA on a
 * CUDA error.  The buffer's contents do not matter and are not changed.
 */
int fa_probe_read_bandwidth(const void *buf, size_t bytes, int iters, void *stream, double *gbs);

/* Static, human-readable name of a status code (never NULL). */
const char *fa_status_string(int status);

/*
 * Synchronises `stream`, then returns FA_OK if no kernel of this library has
 * recorded an error on the current device since the last call, or the recorded
 * code (FA_ERR_TIMEOUT) otherwise, and clears the record.  A CUDA error during
 * the synchronisation or the read returns FA_ERR_CUDA.
 */
int fa_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
